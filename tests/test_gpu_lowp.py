"""GPU parity of the low-precision compressed cache (FP4 E2M1 latent with a 32-dim shared scale,
FP8 E4M3 RoPE tail; [LAB41] "Lab tổng hợp DeepSeek-V4.1-Flash", section "3 Giải pháp") against the
fp64 oracle:
  * the compressor's entries, decoded by the oracle's own unpacker, are the format's rounding of the
    oracle's fp64 entries (up to fp32 computing error at rounding boundaries);
  * the decode step (the one-launch indexer and the fused attention reading the format directly, or
    the bf16 copies for the paths that do not), prefill and the S > 1 calls, stage-chained: the oracle
    scores and attends over the GPU's cache as decoded by the oracle, with the bf16 tolerances (the
    kernels expand the codes exactly)."""
import numpy as np
import pytest
import torch

import synth
from oracle import csa_oracle as O
from tests import _harness as Hn

pytestmark = pytest.mark.gpu

DECODE = {
    "csa_fp4": (synth.small_workload(1, wid=301, B=3, N=4099, t=4098, storage="fp4"), [4098, 4095, 2050]),
    "csa_fp4_B32": (synth.small_workload(1, wid=302, B=32, N=4099, t=4098, storage="fp4"),
                    [4098 - 37 * b for b in range(32)]),
    "csa_fp4_k1024": (synth.small_workload(1, wid=303, B=4, N=8195, t=8194, top_k=1024, storage="fp4"),
                      [8194, 8191, 5000, 4095]),
    "csa_fp4_early": (synth.small_workload(1, wid=304, B=5, N=520, t=519, storage="fp4"), [3, 7, 2, 0, 519]),
    "hca_fp4": (synth.small_workload(3, wid=305, B=2, N=8256, t=8255, storage="fp4"), [8255, 5000]),
    # more entries than the one-launch indexer holds per request: the index cache goes through its bf16
    # copy, the attention still reads the low-precision KV cache itself
    "csa_fp4_long": (synth.small_workload(1, wid=306, B=1, N=140003, t=140002, storage="fp4"), [140002]),
}


def _batch(name):
    wl, pos = DECODE[name]
    return Hn.DeviceBatch(wl), np.array(pos, np.int64)


def _oracle_entries(bt, o, which, entries):
    """fp64 oracle entries of every request (the single-entry form, from the raw rows)."""
    m = o.ratio
    out = []
    for r in bt.reqs:
        raw, gate, bias = ((r["kv"], r["gate"], bt.shared["bias"]) if which == 0 else
                           (r["idx_k"], r["idx_gate"], bt.shared["idx_bias"]))
        rows = []
        for e in entries:
            lo = max(0, (e - 1) * m)
            rows.append(O.compress_entry(raw[lo:(e + 1) * m], gate[lo:(e + 1) * m], bias, e, m))
        out.append(np.stack(rows))
    return out


@pytest.mark.parametrize("name", ["csa_fp4", "hca_fp4", "csa_fp4_early"])
def test_lowp_compress_matches_oracle(name):
    bt, _ = _batch(name)
    c, o = Hn.configs(bt.wl)
    L = Hn.lib()
    n = bt.wl.n_entries
    half = n // 2 + 1
    L.csa_compress(c, bt.cache(), 0, half)
    L.csa_compress(c, bt.cache(), half, n - half)
    torch.cuda.synchronize()
    for b, r in enumerate(bt.reqs):
        ref = O.compress(r["kv"], r["gate"], bt.shared["bias"], o.ratio, n)
        Hn.check_entries_lowp(bt.entries(0)[b], ref, f"{name} ckv[{b}]")
        if not o.hca:
            ref = O.compress(r["idx_k"], r["idx_gate"], bt.shared["idx_bias"], o.ratio, n)
            Hn.check_entries_lowp(bt.entries(1)[b], ref, f"{name} cidx[{b}]")


def test_lowp_compress_writes_only_its_range():
    bt, _ = _batch("csa_fp4")
    c, o = Hn.configs(bt.wl)
    Hn.lib().csa_compress(c, bt.cache(), 5, 9)
    torch.cuda.synchronize()
    ck = bt.entries(0)
    assert np.isnan(ck[:, :5]).all(axis=2).all() and np.isnan(ck[:, 14:]).all(axis=2).all()
    assert not np.isnan(ck[:, 5:14]).any()


@pytest.mark.parametrize("name", list(DECODE))
def test_lowp_decode_step_matches_oracle(name):
    """csa_decode over FP4 / FP8 caches: entries not yet visible are poisoned (NaN codes) and must
    never be read; the closing entry is written by the step in the format."""
    bt, pos = _batch(name)
    c, o = Hn.configs(bt.wl)
    L = Hn.lib()
    L.csa_compress(c, bt.cache(), 0, bt.wl.n_entries)
    torch.cuda.synchronize()
    for b, t in enumerate(pos):
        bt.poison_from(b, t // c.ratio if (t + 1) % c.ratio == 0 else O.visible(t, c.ratio))
    B = bt.B
    out = torch.full((B, c.H, c.d), float("nan"), dtype=c.dtype, device="cuda")
    topk = None if o.hca else torch.full((B, c.top_k), -7, dtype=torch.int32, device="cuda")
    L.csa_decode(c, torch.from_numpy(pos).cuda(), bt.cache(), bt.q[:, 0], None if o.hca else bt.q_idx[:, 0],
                 None if o.hca else bt.w[:, 0], bt.sink, out, topk)
    torch.cuda.synchronize()
    assert L.csa_get_device_status() == 0
    ckv, cidx = bt.entries(0), None if o.hca else bt.entries(1)
    for b, t in enumerate(pos):
        t = int(t)
        V = O.visible(t, c.ratio)
        if (t + 1) % c.ratio == 0:                  # the closing entry was written by this step
            e = t // c.ratio
            Hn.check_entries_lowp(ckv[b, e], _oracle_entries(bt, o, 0, [e])[b], f"{name} closing ckv b{b}")
            if cidx is not None:
                Hn.check_entries_lowp(cidx[b, e], _oracle_entries(bt, o, 1, [e])[b], f"{name} closing cidx b{b}")
        assert not np.isnan(ckv[b, :V]).any()
        sel = None
        if not o.hca:
            sel = topk[b].cpu().numpy()
            ref_s = O.index_scores(bt.reqs[b]["q_idx"][0], bt.reqs[b]["w"][0], cidx[b], t, c.ratio)
            Hn.check_topk_vs_oracle(sel, ref_s, c.top_k, f"{name} decode b{b}")
        ref = O.sparse_attn(bt.reqs[b]["q"][0], bt.reqs[b]["kv"], ckv[b], sel, bt.shared["sink"], t, o)
        Hn.check_attn(Hn.host64(out[b]), ref, "fp4", f"{name} decode b{b}")


@pytest.mark.parametrize("name", ["csa_fp4", "csa_fp4_B32", "csa_fp4_long"])
def test_lowp_index_topk_and_sparse_attn(name):
    """The stage calls over FP4 / FP8 caches: csa_index_topk with its score output at one query per
    request (the one-launch indexer where it applies) and at two (the bf16 copy), csa_sparse_attn at
    one query (the fused attention) and at two (the bf16 copy)."""
    bt, pos = _batch(name)
    c, o = Hn.configs(bt.wl)
    L = Hn.lib()
    L.csa_compress(c, bt.cache(), 0, bt.wl.n_entries)
    cidx, ckv = bt.entries(1), bt.entries(0)
    B, n = bt.B, bt.n_cap
    for S in (1, 2):
        P = np.stack([pos, np.maximum(pos // 3, 0)], axis=1)[:, :S]
        Pd = torch.from_numpy(np.ascontiguousarray(P)).cuda()
        q_idx = torch.stack([bt.q_idx[:, 0], torch.flip(bt.q_idx[:, 0], dims=[-1])], dim=1)[:, :S].contiguous()
        w = torch.stack([bt.w[:, 0], -bt.w[:, 0]], dim=1)[:, :S].contiguous()
        q = torch.stack([bt.q[:, 0], torch.flip(bt.q[:, 0], dims=[-1])], dim=1)[:, :S].contiguous()
        topk = torch.full((B, S, c.top_k), -7, dtype=torch.int32, device="cuda")
        scores = torch.full((B, S, n), float("nan"), device="cuda")
        L.csa_index_topk(c, Pd, q_idx, w, bt.cidx, topk, scores, n_cap=n)
        out = torch.full((B, S, c.H, c.d), float("nan"), dtype=c.dtype, device="cuda")
        L.csa_sparse_attn(c, Pd, q, bt.kv, bt.ckv, topk, bt.sink, out, n_cap=n)
        torch.cuda.synchronize()
        assert L.csa_get_device_status() == 0
        for b in range(B):
            for s in range(S):
                t = int(P[b, s])
                V = O.visible(t, c.ratio)
                ref = O.index_scores(Hn.host64(q_idx[b, s]), Hn.host64(w[b, s]), cidx[b], t, c.ratio)
                got = scores[b, s, :V].double().cpu().numpy()
                Hn.check_scores(got, ref, "fp4", f"{name} S{S} scores b{b} s{s}")
                tk = topk[b, s].cpu().numpy()
                Hn.check_topk_exact(tk, got, c.top_k, f"{name} S{S} b{b} s{s}")
                refo = O.sparse_attn(Hn.host64(q[b, s]), bt.reqs[b]["kv"], ckv[b], tk, bt.shared["sink"], t, o)
                Hn.check_attn(Hn.host64(out[b, s]), refo, "fp4", f"{name} S{S} attention b{b} s{s}")


PREFILL = {
    "csa_fp4": synth.small_workload(2, wid=311, B=2, N=1030, S=1030, top_k=64, storage="fp4"),
    "hca_fp4": synth.small_workload(2, wid=312, B=1, N=700, S=700, ratio=32, top_k=0, storage="fp4"),
}


@pytest.mark.parametrize("name", list(PREFILL))
def test_lowp_prefill_matches_oracle(name):
    wl = PREFILL[name]
    bt = Hn.DeviceBatch(wl)
    c, o = Hn.configs(wl)
    L = Hn.lib()
    B, S = bt.B, wl.S
    out = torch.full((B, S, c.H, c.d), float("nan"), dtype=c.dtype, device="cuda")
    topk = None if o.hca else torch.empty(B, S, c.top_k, dtype=torch.int32, device="cuda")
    L.csa_prefill(c, bt.cache(), bt.q, bt.q_idx, bt.w, bt.sink, out, topk)
    torch.cuda.synchronize()
    assert L.csa_get_device_status() == 0
    ckv, cidx = bt.entries(0), None if o.hca else bt.entries(1)
    outh = Hn.host64(out)
    tk = None if o.hca else topk.cpu().numpy()
    n = S // c.ratio
    for b, r in enumerate(bt.reqs):
        Hn.check_entries_lowp(ckv[b, :n], O.compress(r["kv"], r["gate"], bt.shared["bias"], o.ratio, n), f"{name} ckv")
        if cidx is not None:
            Hn.check_entries_lowp(cidx[b, :n], O.compress(r["idx_k"], r["idx_gate"], bt.shared["idx_bias"], o.ratio, n),
                                  f"{name} cidx")
        for t in range(S):
            sel = None
            if not o.hca:
                sel = tk[b, t]
                ref_s = O.index_scores(r["q_idx"][t], r["w"][t], cidx[b], t, c.ratio)
                Hn.check_topk_vs_oracle(sel, ref_s, c.top_k, f"{name} prefill b{b} t{t}")
            ref = O.sparse_attn(r["q"][t], r["kv"], ckv[b], sel, bt.shared["sink"], t, o)
            Hn.check_attn(outh[b, t], ref, "fp4", f"{name} prefill b{b} t{t}")


def test_lowp_static_entry_point():
    """csa_index_topk_static reads an FP4 / FP8 index cache through the one-launch indexer (no
    scratch) and equals csa_index_topk; beyond that kernel it refuses (no bf16 copy without a
    workspace)."""
    bt, pos = _batch("csa_fp4")
    c, o = Hn.configs(bt.wl)
    L = Hn.lib()
    L.csa_compress(c, bt.cache(), 0, bt.wl.n_entries)
    Pd = torch.from_numpy(pos[:, None].copy()).cuda()
    a = torch.full((bt.B, 1, c.top_k), -7, dtype=torch.int32, device="cuda")
    b_ = torch.full((bt.B, 1, c.top_k), -9, dtype=torch.int32, device="cuda")
    L.csa_index_topk(c, Pd, bt.q_idx, bt.w, bt.cidx, a, n_cap=bt.n_cap)
    L.csa_index_topk_static(c, Pd, bt.q_idx, bt.w, bt.cidx, b_, n_cap=bt.n_cap)
    torch.cuda.synchronize()
    assert torch.equal(a, b_)
    P2 = torch.from_numpy(np.stack([pos, pos // 2], axis=1)).cuda()
    q2 = torch.cat([bt.q_idx, bt.q_idx], dim=1).contiguous()
    w2 = torch.cat([bt.w, bt.w], dim=1).contiguous()
    t2 = torch.empty((bt.B, 2, c.top_k), dtype=torch.int32, device="cuda")
    with pytest.raises(L.CsaError) as ei:
        L.csa_index_topk_static(c, P2, q2, w2, bt.cidx, t2, n_cap=bt.n_cap)
    assert ei.value.status == 4
