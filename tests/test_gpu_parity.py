"""GPU parity of every stage of the path against the fp64 oracle, on seeded inputs that span several
tiles and ragged tails. Stages are chained on the GPU's own outputs (compressed caches, scores,
selections) so each stage's tolerance is checked on exactly the values it consumed."""
import numpy as np
import pytest
import torch

import synth
from oracle import csa_oracle as O
from tests import _harness as Hn

pytestmark = pytest.mark.gpu

# name -> (workload, decode positions per request)
DECODE = {
    "csa_bf16": (synth.small_workload(1, wid=101, B=3, N=4099, t=4098), [4098, 4095, 2050]),
    "csa_bf16_sharp": (synth.small_workload(1, wid=102, B=2, N=2051, t=2050, q_gain=16.0), [2050, 1023]),
    "hca_bf16": (synth.small_workload(3, wid=103, B=2, N=8256, t=8255), [8255, 5000]),
    "csa_f32": (synth.small_workload(0, wid=100, B=2), [2047, 1001]),
    "csa_f32_cfg0": (synth.WORKLOADS[0], [2047]),
    # enough rows that the tensor-core attention puts two candidate tiles in one CTA
    "csa_bf16_B32": (synth.small_workload(1, wid=104, B=32, N=4099, t=4098),
                     [4098 - 37 * b for b in range(32)]),
    "hca_bf16_B16_wide": (synth.small_workload(3, wid=105, B=16, N=19215, t=19214, ratio=16),
                          [19214, 19199] + [19214 - 977 * b for b in range(2, 16)]),
    # more tiles than two waves of CTAs: two tiles per CTA, one of them gathered twice
    "csa_bf16_B64": (synth.small_workload(1, wid=106, B=64, N=2051, t=2050),
                     [2050 - 13 * b for b in range(64)]),
    # the first groups: entry 0 closes at t = 3 (its previous group lies before position 0, weight
    # 0), entry 1 at t = 7; t = 0 and t = 2 see no compressed entry at all
    "csa_bf16_early": (synth.small_workload(1, wid=107, B=5, N=520, t=519), [3, 7, 2, 0, 519]),
    # the Pro variant's selection size: 1024 selected entries (8 tiles) + the window per query
    "csa_bf16_k1024": (synth.small_workload(1, wid=108, B=4, N=8195, t=8194, top_k=1024),
                       [8194, 8191, 5000, 4095]),
}
MODES = [False, True]          # tensor-core path where available, then the CUDA-core path


def _batch(name):
    wl, pos = DECODE[name]
    return Hn.DeviceBatch(wl), np.array(pos, np.int64)


def _oracle_caches(bt, o):
    out = []
    for r in bt.reqs:
        n = bt.wl.n_entries
        ckv = O.compress(r["kv"], r["gate"], bt.shared["bias"], o.ratio, n, rms_eps=o.rms_eps)
        cidx = None if o.hca else O.compress(r["idx_k"], r["idx_gate"], bt.shared["idx_bias"], o.ratio, n,
                                             rms_eps=o.rms_eps)
        out.append((ckv, cidx))
    return out


@pytest.mark.parametrize("name", list(DECODE))
def test_compress_matches_oracle(name):
    bt, _ = _batch(name)
    c, o = Hn.configs(bt.wl)
    L = Hn.lib()
    n = bt.wl.n_entries
    half = n // 2 + 1                               # second call starts mid-cache (previous group read)
    L.csa_compress(c, bt.cache(), 0, half)
    L.csa_compress(c, bt.cache(), half, n - half)
    torch.cuda.synchronize()
    for b, (ckv, cidx) in enumerate(_oracle_caches(bt, o)):
        Hn.check_entries(Hn.host64(bt.ckv[b]), ckv, bt.wl.storage, f"{name} ckv[{b}]")
        if cidx is not None:
            Hn.check_entries(Hn.host64(bt.cidx[b]), cidx, bt.wl.storage, f"{name} cidx[{b}]")


def test_compress_writes_only_its_range():
    bt, _ = _batch("csa_bf16")
    c, o = Hn.configs(bt.wl)
    Hn.lib().csa_compress(c, bt.cache(), 5, 9)
    torch.cuda.synchronize()
    ck = bt.ckv.float()
    assert torch.isnan(ck[:, :5]).all() and torch.isnan(ck[:, 14:]).all()
    assert not torch.isnan(ck[:, 5:14]).any()
    ref = O.compress(bt.reqs[1]["kv"], bt.reqs[1]["gate"], bt.shared["bias"], o.ratio, 14)
    Hn.check_entries(Hn.host64(bt.ckv[1, 5:14]), ref[5:14], "bf16", "ckv range")


def _decode_pos_pairs(bt, pos):
    """two query positions per request for the stage tests: the decode position and an earlier one"""
    return np.stack([pos, np.maximum(pos // 3, 0)], axis=1)


@pytest.mark.parametrize("simt", MODES)
@pytest.mark.parametrize("name", [n for n in DECODE if not DECODE[n][0].hca])
def test_index_topk_matches_oracle(name, simt):
    bt, pos = _batch(name)
    c, o = Hn.configs(bt.wl, simt)
    L = Hn.lib()
    L.csa_compress(c, bt.cache(), 0, bt.wl.n_entries)
    P = _decode_pos_pairs(bt, pos)
    B, S = P.shape
    q_idx = torch.stack([bt.q_idx[:, 0]] * S, dim=1).contiguous()
    q_idx[:, 1] = torch.flip(q_idx[:, 1], dims=[-1])          # a different query for the second row
    w = torch.stack([bt.w[:, 0], -bt.w[:, 0]], dim=1).contiguous()
    topk = torch.empty(B, S, c.top_k, dtype=torch.int32, device="cuda")
    scores = torch.full((B, S, bt.wl.n_entries), float("nan"), device="cuda")
    L.csa_index_topk(c, torch.from_numpy(P).cuda(), q_idx, w, bt.cidx, topk, scores)
    torch.cuda.synchronize()
    cidx = Hn.host64(bt.cidx)
    for b in range(B):
        for s in range(S):
            t = int(P[b, s])
            V = O.visible(t, c.ratio)
            ref = O.index_scores(Hn.host64(q_idx[b, s]), Hn.host64(w[b, s]), cidx[b], t, c.ratio)
            got = scores[b, s, :V].double().cpu().numpy()
            Hn.check_scores(got, ref, bt.wl.storage, f"{name} scores b{b} s{s}")
            tk = topk[b, s].cpu().numpy()
            Hn.check_topk_exact(tk, got, c.top_k, f"{name} b{b} s{s}")
            Hn.check_topk_vs_oracle(tk, ref, c.top_k, f"{name} b{b} s{s}")


@pytest.mark.parametrize("simt", MODES)
@pytest.mark.parametrize("name", list(DECODE))
def test_sparse_attn_matches_oracle(name, simt):
    bt, pos = _batch(name)
    c, o = Hn.configs(bt.wl, simt)
    L = Hn.lib()
    L.csa_compress(c, bt.cache(), 0, bt.wl.n_entries)
    B = bt.B
    P = torch.from_numpy(pos[:, None].copy()).cuda()
    topk = None
    if not o.hca:
        topk = torch.empty(B, 1, c.top_k, dtype=torch.int32, device="cuda")
        L.csa_index_topk(c, P, bt.q_idx, bt.w, bt.cidx, topk)
    out = torch.full((B, 1, c.H, c.d), float("nan"), dtype=c.dtype, device="cuda")
    L.csa_sparse_attn(c, P, bt.q, bt.kv, bt.ckv, topk, bt.sink, out)
    torch.cuda.synchronize()
    assert Hn.lib().csa_get_device_status() == 0
    ckv = Hn.host64(bt.ckv)
    for b in range(B):
        t = int(pos[b])
        sel = None if o.hca else topk[b, 0].cpu().numpy()
        ref = O.sparse_attn(bt.reqs[b]["q"][0], bt.reqs[b]["kv"], ckv[b], sel, bt.shared["sink"], t, o)
        Hn.check_attn(Hn.host64(out[b, 0]), ref, bt.wl.storage, f"{name} b{b}")


@pytest.mark.parametrize("simt", MODES)
@pytest.mark.parametrize("name", list(DECODE))
def test_decode_step_matches_oracle(name, simt):
    """csa_decode: compress-on-close, indexer, top-k, attention; entries that are not yet visible
    are poisoned with NaN and must never be read."""
    bt, pos = _batch(name)
    c, o = Hn.configs(bt.wl, simt)
    L = Hn.lib()
    L.csa_compress(c, bt.cache(), 0, bt.wl.n_entries)
    torch.cuda.synchronize()
    ref_caches = _oracle_caches(bt, o)
    for b, t in enumerate(pos):
        first_unwritten = t // c.ratio if (t + 1) % c.ratio == 0 else O.visible(t, c.ratio)
        bt.ckv[b, first_unwritten:] = float("nan")
        if bt.cidx is not None:
            bt.cidx[b, first_unwritten:] = float("nan")
    B = bt.B
    out = torch.full((B, c.H, c.d), float("nan"), dtype=c.dtype, device="cuda")
    topk = None if o.hca else torch.full((B, c.top_k), -7, dtype=torch.int32, device="cuda")
    L.csa_decode(c, torch.from_numpy(pos).cuda(), bt.cache(), bt.q[:, 0], None if o.hca else bt.q_idx[:, 0],
                 None if o.hca else bt.w[:, 0], bt.sink, out, topk)
    torch.cuda.synchronize()
    assert L.csa_get_device_status() == 0
    ckv, cidx = Hn.host64(bt.ckv), None if o.hca else Hn.host64(bt.cidx)
    for b, t in enumerate(pos):
        t = int(t)
        V = O.visible(t, c.ratio)
        if (t + 1) % c.ratio == 0:                  # the closing entry was written by this step
            Hn.check_entries(ckv[b, t // c.ratio], ref_caches[b][0][t // c.ratio], bt.wl.storage, "closing ckv")
            if cidx is not None:
                Hn.check_entries(cidx[b, t // c.ratio], ref_caches[b][1][t // c.ratio], bt.wl.storage,
                                 "closing cidx")
        assert not np.isnan(ckv[b, :V]).any()
        sel = None
        if not o.hca:
            sel = topk[b].cpu().numpy()
            ref_s = O.index_scores(bt.reqs[b]["q_idx"][0], bt.reqs[b]["w"][0], cidx[b], t, c.ratio)
            Hn.check_topk_vs_oracle(sel, ref_s, c.top_k, f"{name} decode b{b}")
        ref = O.sparse_attn(bt.reqs[b]["q"][0], bt.reqs[b]["kv"], ckv[b], sel, bt.shared["sink"], t, o)
        Hn.check_attn(Hn.host64(out[b]), ref, bt.wl.storage, f"{name} decode b{b}")


PREFILL = {
    "csa_bf16": synth.small_workload(2, wid=202, B=2, N=1030, S=1030, top_k=64),
    "hca_bf16": synth.small_workload(2, wid=203, B=1, N=700, S=700, ratio=32, top_k=0),
    "csa_f32": synth.small_workload(2, wid=204, B=1, N=600, S=600, H=8, H_idx=8, top_k=32, storage="f32"),
}


@pytest.mark.parametrize("simt", MODES)
@pytest.mark.parametrize("name", list(PREFILL))
def test_prefill_matches_oracle(name, simt):
    wl = PREFILL[name]
    bt = Hn.DeviceBatch(wl)
    c, o = Hn.configs(wl, simt)
    L = Hn.lib()
    B, S = bt.B, wl.S
    out = torch.full((B, S, c.H, c.d), float("nan"), dtype=c.dtype, device="cuda")
    topk = None if o.hca else torch.empty(B, S, c.top_k, dtype=torch.int32, device="cuda")
    L.csa_prefill(c, bt.cache(), bt.q, bt.q_idx, bt.w, bt.sink, out, topk)
    torch.cuda.synchronize()
    assert L.csa_get_device_status() == 0
    ref_caches = _oracle_caches(bt, o)
    ckv, cidx = Hn.host64(bt.ckv), None if o.hca else Hn.host64(bt.cidx)
    outh = Hn.host64(out)
    tk = None if o.hca else topk.cpu().numpy()
    for b in range(B):
        n = S // c.ratio
        Hn.check_entries(ckv[b, :n], ref_caches[b][0][:n], wl.storage, f"{name} ckv")
        if cidx is not None:
            Hn.check_entries(cidx[b, :n], ref_caches[b][1][:n], wl.storage, f"{name} cidx")
        for t in range(S):
            sel = None
            if not o.hca:
                sel = tk[b, t]
                ref_s = O.index_scores(bt.reqs[b]["q_idx"][t], bt.reqs[b]["w"][t], cidx[b], t, c.ratio)
                Hn.check_topk_vs_oracle(sel, ref_s, c.top_k, f"{name} prefill b{b} t{t}")
            ref = O.sparse_attn(bt.reqs[b]["q"][t], bt.reqs[b]["kv"], ckv[b], sel, bt.shared["sink"], t, o)
            Hn.check_attn(outh[b, t], ref, wl.storage, f"{name} prefill b{b} t{t}")


CHUNKED = {
    "csa_bf16": synth.small_workload(2, wid=206, B=2, N=1300, S=1300, top_k=64),
    "hca_bf16": synth.small_workload(2, wid=207, B=2, N=1300, S=1300, ratio=16, top_k=0),
    "csa_f32": synth.small_workload(2, wid=208, B=2, N=1300, S=1300, H=8, H_idx=8, top_k=32, storage="f32"),
}


@pytest.mark.parametrize("simt", MODES)
@pytest.mark.parametrize("name", list(CHUNKED))
def test_chunked_prefill_matches_oracle(name, simt):
    """A prefill chunk over an existing cache ([FLASH] "压缩条目必须等整组完成后才可见": every query keeps
    its own visibility): the entries of tokens 0..1023 exist, the chunk's tokens 1024..1299 close
    further groups (csa_compress on the new entry range), then S queries of the chunk at
    non-consecutive positions (each request its own order) go through csa_index_topk and
    csa_sparse_attn with S > 1. Compared with the oracle on the GPU's caches."""
    wl = CHUNKED[name]
    bt = Hn.DeviceBatch(wl)
    c, o = Hn.configs(wl, simt)
    L = Hn.lib()
    m = c.ratio
    n0, n1 = 1024 // m, wl.N // m
    L.csa_compress(c, bt.cache(), 0, n0)
    L.csa_compress(c, bt.cache(), n0, n1 - n0)
    rng = np.random.default_rng(len(name) + simt)
    S = 12
    P = np.stack([rng.permutation(np.arange(1024, wl.N))[:S] for _ in range(bt.B)]).astype(np.int64)
    P[0, :3] = [wl.N - 1, 1024, 1027]                    # the chunk's last token and its first group
    Pd = torch.from_numpy(P).cuda()
    pick = lambda T: torch.stack([T[b, Pd[b]] for b in range(bt.B)]).contiguous()
    q = pick(bt.q)
    topk = None
    if not o.hca:
        topk = torch.full((bt.B, S, c.top_k), -7, dtype=torch.int32, device="cuda")
        L.csa_index_topk(c, Pd, pick(bt.q_idx), pick(bt.w), bt.cidx, topk)
    out = torch.full((bt.B, S, c.H, c.d), float("nan"), dtype=c.dtype, device="cuda")
    L.csa_sparse_attn(c, Pd, q, bt.kv, bt.ckv, topk, bt.sink, out)
    torch.cuda.synchronize()
    assert L.csa_get_device_status() == 0
    ref_caches = _oracle_caches(bt, o)
    ckv, cidx = Hn.host64(bt.ckv), None if o.hca else Hn.host64(bt.cidx)
    for b in range(bt.B):
        Hn.check_entries(ckv[b, :n1], ref_caches[b][0][:n1], wl.storage, f"{name} chunk ckv[{b}]")
        if cidx is not None:
            Hn.check_entries(cidx[b, :n1], ref_caches[b][1][:n1], wl.storage, f"{name} chunk cidx[{b}]")
        for s in range(S):
            t = int(P[b, s])
            sel = None
            if not o.hca:
                sel = topk[b, s].cpu().numpy()
                ref_s = O.index_scores(bt.reqs[b]["q_idx"][t], bt.reqs[b]["w"][t], cidx[b], t, c.ratio)
                Hn.check_topk_vs_oracle(sel, ref_s, c.top_k, f"{name} chunk b{b} t{t}")
            ref = O.sparse_attn(bt.reqs[b]["q"][t], bt.reqs[b]["kv"], ckv[b], sel, bt.shared["sink"], t, o)
            Hn.check_attn(Hn.host64(out[b, s]), ref, wl.storage, f"{name} chunk b{b} t{t}")


@pytest.mark.parametrize("name", ["csa_bf16", "csa_f32"])
def test_prefill_equals_decode_on_gpu(name):
    """The GPU's prefill rows equal its own decode steps at the same positions (prefill ==
    streaming), within the attention tolerance."""
    wl = PREFILL[name]
    bt = Hn.DeviceBatch(wl)
    c, o = Hn.configs(wl)
    L = Hn.lib()
    B, S = bt.B, wl.S
    out = torch.empty((B, S, c.H, c.d), dtype=c.dtype, device="cuda")
    L.csa_prefill(c, bt.cache(), bt.q, bt.q_idx, bt.w, bt.sink, out)
    for t in (0, 2, 3, 4, 7, 200, S - 1):
        pos = torch.full((B,), t, dtype=torch.int64, device="cuda")
        od = torch.empty((B, c.H, c.d), dtype=c.dtype, device="cuda")
        L.csa_decode(c, pos, bt.cache(), bt.q[:, t].contiguous(), bt.q_idx[:, t].contiguous(),
                     bt.w[:, t].contiguous(), bt.sink, od)
        for b in range(B):
            Hn.check_attn(Hn.host64(od[b]), Hn.host64(out[b, t]), wl.storage, f"decode vs prefill t{t}")


def test_bad_selected_index_sets_device_error():
    bt, pos = _batch("csa_f32")
    c, o = Hn.configs(bt.wl)
    L = Hn.lib()
    L.csa_get_device_status(reset=True)
    L.csa_compress(c, bt.cache(), 0, bt.wl.n_entries)
    topk = torch.zeros(bt.B, 1, c.top_k, dtype=torch.int32, device="cuda")
    topk[0, 0, 3] = 10 ** 6                          # far beyond the visible entries
    out = torch.empty((bt.B, 1, c.H, c.d), dtype=c.dtype, device="cuda")
    L.csa_sparse_attn(c, torch.from_numpy(pos[:, None].copy()).cuda(), bt.q, bt.kv, bt.ckv, topk, bt.sink, out)
    assert L.csa_get_device_status(reset=True) == 1          # DEVERR_BAD_INDEX
    assert torch.isfinite(out.float()).all()
    assert L.csa_get_device_status() == 0


def test_bounded_wait_reports_timeout_and_recovers():
    """The device-side timeout path, made to run out on purpose: with the test hook the one-launch
    decode indexer skips its first cache-tile load and its waits (limited to 2 ms) run out; the
    kernels return, the error word holds the timeout code and csa_sync_status reports
    CSA_ERR_DEVICE_TIMEOUT. After a reset, the same step without the hook matches the oracle."""
    import dataclasses
    bt, pos = _batch("csa_bf16")
    c, o = Hn.configs(bt.wl)
    L = Hn.lib()
    L.csa_get_device_status(reset=True)
    L.csa_compress(c, bt.cache(), 0, bt.wl.n_entries)
    B = bt.B
    P = torch.from_numpy(pos).cuda()
    out = torch.zeros((B, c.H, c.d), dtype=c.dtype, device="cuda")
    topk = torch.full((B, c.top_k), -7, dtype=torch.int32, device="cuda")
    L.csa_decode(dataclasses.replace(c, test_stall=True), P, bt.cache(), bt.q[:, 0], bt.q_idx[:, 0], bt.w[:, 0],
                 bt.sink, out, topk)
    assert L.csa_sync_status() == L.CSA_ERR_DEVICE_TIMEOUT
    assert L.csa_sync_status() == L.CSA_ERR_DEVICE_TIMEOUT      # the word is kept until reset
    assert L.csa_get_device_status(reset=True) == 2
    assert L.csa_sync_status() == 0
    L.csa_decode(c, P, bt.cache(), bt.q[:, 0], bt.q_idx[:, 0], bt.w[:, 0], bt.sink, out, topk)
    assert L.csa_sync_status() == 0
    ckv, cidx = Hn.host64(bt.ckv), Hn.host64(bt.cidx)
    for b, t in enumerate(pos):
        t = int(t)
        sel = topk[b].cpu().numpy()
        ref_s = O.index_scores(bt.reqs[b]["q_idx"][0], bt.reqs[b]["w"][0], cidx[b], t, c.ratio)
        Hn.check_topk_vs_oracle(sel, ref_s, c.top_k, f"after the timeout b{b}")
        ref = O.sparse_attn(bt.reqs[b]["q"][0], bt.reqs[b]["kv"], ckv[b], sel, bt.shared["sink"], t, o)
        Hn.check_attn(Hn.host64(out[b]), ref, bt.wl.storage, f"after the timeout b{b}")


def test_argument_errors_launch_nothing():
    bt, pos = _batch("csa_f32")
    c, o = Hn.configs(bt.wl)
    L = Hn.lib()
    with pytest.raises(L.CsaError) as e:
        L.csa_compress(c, bt.cache(), 0, bt.wl.n_entries + 1)
    assert e.value.status == 2
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    out = torch.zeros((bt.B, c.H, c.d), dtype=c.dtype, device="cuda")
    with pytest.raises(L.CsaError) as e:
        L.csa_decode(c, torch.from_numpy(pos).cuda(), bt.cache(), bt.q[:, 0], bt.q_idx[:, 0], bt.w[:, 0],
                     bt.sink, out, ws=ws)
    assert e.value.status == 4
    assert torch.all(out == 0)


@pytest.mark.parametrize("n_cap,k,B,dup", [
    (20000, 512, 2, False),      # two chunks, then a candidate level
    (262144, 512, 1, False),     # the 1M-token workload's row length: sixteen chunks
    (70000, 2048, 1, True),      # k = 2048 with exact ties (repeated cache rows): three levels
    (5000, 2048, 1, False),      # fewer visible entries than k: everything, sorted, -1 tail
])
def test_topk_long_rows_exact(n_cap, k, B, dup):
    """Indexer + selection on rows longer than one CTA holds: the GPU's selection equals the exact
    (-score, index) selection of its own scores; the scores match the oracle."""
    rng = np.random.default_rng(n_cap + k)
    import synth as S
    L = Hn.lib()
    H_idx = 64
    cidx = S.round_bf16(rng.standard_normal((B, n_cap, 128), dtype=np.float32) / np.float32(np.sqrt(128)))
    if dup:
        cidx[:, 3000:] = cidx[:, np.arange(3000, n_cap) % 3000]
    q_idx = S.round_bf16(rng.standard_normal((B, 1, H_idx, 128), dtype=np.float32) / np.float32(np.sqrt(128)))
    w = (rng.standard_normal((B, 1, H_idx)) / np.sqrt(128 * H_idx)).astype(np.float32)
    c = L.Config(top_k=k, ratio=4)
    pos = np.array([[4 * n_cap - 1]] * B, np.int64)
    if B > 1:
        pos[1, 0] = 4 * (n_cap - 777) - 2          # fewer visible entries in the second row
    d_cidx, d_q = Hn.dev(cidx, "bf16"), Hn.dev(q_idx, "bf16")
    topk = torch.empty(B, 1, k, dtype=torch.int32, device="cuda")
    scores = torch.full((B, 1, n_cap), float("nan"), device="cuda")
    L.csa_index_topk(c, torch.from_numpy(pos).cuda(), d_q, torch.from_numpy(w).cuda(), d_cidx, topk, scores)
    torch.cuda.synchronize()
    for b in range(B):
        t = int(pos[b, 0])
        V = O.visible(t, 4)
        got = scores[b, 0, :V].double().cpu().numpy()
        tk = topk[b, 0].cpu().numpy()
        Hn.check_topk_exact(tk, got, k, f"long row b{b}")
        ref = O.index_scores(q_idx[b, 0], w[b, 0], cidx[b], t, 4)
        Hn.check_scores(got, ref, "bf16", f"long row scores b{b}")


@pytest.mark.parametrize("n_cap", [16384, 6000])
@pytest.mark.parametrize("mode", ["equal", "narrow", "few"])
def test_topk_one_cluster_paths(n_cap, mode):
    """Rows of 2049..16384 entries are selected by one cluster of CTAs. Score distributions that
    force each of its paths: every score equal (all digits exchanged, then the first k by
    position), scores packed into a narrow range (the threshold bin holds more than the in-bin list
    takes, so a further digit is exchanged before the bin is split locally), and few distinct
    values (large groups of exact ties). The selection must equal the exact (-score, index)
    selection of the GPU's own scores."""
    rng = np.random.default_rng(n_cap + len(mode))
    import synth as S
    L = Hn.lib()
    B, H_idx, k = 2, 64, 512
    base = rng.standard_normal((1, 1, 128), dtype=np.float32) / np.float32(np.sqrt(128))
    if mode == "equal":
        cidx = np.repeat(np.repeat(base, n_cap, axis=1), B, axis=0)
    elif mode == "narrow":
        cidx = base + np.float32(2e-3) * rng.standard_normal((B, n_cap, 128), dtype=np.float32)
    else:
        rows = rng.standard_normal((B, 37, 128), dtype=np.float32) / np.float32(np.sqrt(128))
        cidx = rows[:, rng.integers(0, 37, n_cap)]
    cidx = S.round_bf16(np.ascontiguousarray(cidx, dtype=np.float32))
    q_idx = S.round_bf16(rng.standard_normal((B, 1, H_idx, 128), dtype=np.float32) / np.float32(np.sqrt(128)))
    w = (np.abs(rng.standard_normal((B, 1, H_idx))) / np.sqrt(128 * H_idx)).astype(np.float32)
    c = L.Config(top_k=k, ratio=4)
    pos = np.array([[4 * n_cap - 1], [4 * (n_cap - 1000) - 3]], np.int64)
    topk = torch.empty(B, 1, k, dtype=torch.int32, device="cuda")
    scores = torch.full((B, 1, n_cap), float("nan"), device="cuda")
    L.csa_index_topk(c, torch.from_numpy(pos).cuda(), Hn.dev(q_idx, "bf16"), torch.from_numpy(w).cuda(),
                     Hn.dev(cidx, "bf16"), topk, scores)
    torch.cuda.synchronize()
    for b in range(B):
        V = O.visible(int(pos[b, 0]), 4)
        got = scores[b, 0, :V].double().cpu().numpy()
        Hn.check_topk_exact(topk[b, 0].cpu().numpy(), got, k, f"{mode} b{b}")
    assert L.csa_get_device_status() == 0
