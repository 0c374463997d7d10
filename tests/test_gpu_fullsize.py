"""Parity at the workloads' full sizes, in the launch configuration the benchmark times.

The decode workloads (B=32 at N=65,536; HCA B=16 at N=262,144 with m=128; B=4 at N=1,048,579
with a trailing incomplete group) and the S=8192 causal prefill run through the public calls on
the seeded synthetic inputs. The oracle checks, one by one:
  * compressed entries (the first, the last, random ones and the entry the decode step closes,
    which is poisoned with NaN beforehand so that only the decode step can have written it),
    against the oracle's single-entry form on the same raw rows;
  * the selection of every decode request and of 256 or more prefill queries (group boundaries
    around sampled points included), against the oracle's exact selection of its own fp64 scores
    of the GPU's index cache (stage-chained), with the tie band of the tolerances;
  * the attention output of those requests / queries, against the oracle on the GPU's selection
    and compressed entries;
  * one request of the B=32 decode end to end from its raw inputs (the oracle's own caches).
The raw rows the oracle reads are copied back from the device: they are the synthetic inputs
(bf16 values drawn by the seeded generator), not results of the CUDA path. Host arrays the oracle
indexes by position are zero-initialised (left unbacked by the OS) and filled only where read.
"""
import importlib.util
import os

import numpy as np
import pytest
import torch

import synth
from oracle import csa_oracle as O
from tests import _harness as Hn

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_inputs", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _rows(t: torch.Tensor, lo: int, hi: int) -> np.ndarray:
    return Hn.host64(t[lo:hi])


def _check_entries_sampled(wl, T, cache, b, entries, what):
    m = wl.ratio
    jobs = [("ckv", T["kv"], T["gate"], T["bias"], cache.ckv)]
    if not wl.hca:
        jobs.append(("cidx", T["idx_k"], T["idx_gate"], T["idx_bias"], cache.cidx))
    for name, raw, gate, bias, dst in jobs:
        bias64 = Hn.host64(bias)
        for e in entries:
            lo = max(0, (e - 1) * m)
            ref = O.compress_entry(_rows(raw[b], lo, (e + 1) * m), _rows(gate[b], lo, (e + 1) * m), bias64, e, m,
                                   d_rope=wl.d_rope)
            Hn.check_entries(Hn.host64(dst[b, e]), ref, wl.storage, f"{what} {name}[{b}, {e}]")


def _check_query(wl, o, T, cache, b, s, t, sel_gpu, out_gpu, what):
    """Selection and attention of the query at position t (row s of request b)."""
    V = O.visible(t, wl.ratio)
    sel = None
    if not wl.hca:
        cidx = Hn.host64(cache.cidx[b, :V])
        ref_s = O.index_scores(Hn.host64(T["q_idx"][b, s]), Hn.host64(T["w"][b, s]), cidx, t, wl.ratio)
        sel = sel_gpu
        Hn.check_topk_vs_oracle(sel, ref_s, wl.top_k, f"{what} top-k b{b} t{t}")
        comp = sel[sel >= 0]
    else:
        comp = np.arange(V)
    # raw rows: only the window is read; compressed rows: only the selected (all visible for HCA)
    kv = np.zeros((t + 1, wl.d))
    lo = max(0, t - wl.window + 1)
    kv[lo:t + 1] = _rows(T["kv"][b], lo, t + 1)
    ckv = np.zeros((max(V, 1), wl.d))
    if len(comp):
        idx = torch.from_numpy(np.asarray(comp, np.int64)).to(cache.ckv.device)
        ckv[np.asarray(comp)] = Hn.host64(cache.ckv[b].index_select(0, idx))
    ref = O.sparse_attn(Hn.host64(T["q"][b, s]), kv, ckv, sel, Hn.host64(T["sink"]), t, o)
    Hn.check_attn(out_gpu, ref, wl.storage, f"{what} attention b{b} t{t}")


@pytest.mark.parametrize("cid", [1, 3, 4])
def test_full_size_decode_sampled(cid):
    L = Hn.lib()
    bench = _bench()
    wl = synth.WORKLOADS[cid]
    c, o = Hn.configs(wl)
    B, t, m = wl.B, wl.t, wl.ratio
    T = bench.device_inputs(wl, list(range(B)), "cuda")
    try:
        cache = bench.make_cache(T, wl, "cuda")
        L.csa_compress(c, cache, 0, wl.n_entries)
        closes = (t + 1) % m == 0
        e_close = t // m
        if closes:                                  # only the decode step may write this entry
            cache.ckv[:, e_close] = float("nan")
            if not wl.hca:
                cache.cidx[:, e_close] = float("nan")
        pos = torch.full((B,), t, dtype=torch.int64, device="cuda")
        out = torch.full((B, c.H, c.d), float("nan"), dtype=c.dtype, device="cuda")
        topk = None if wl.hca else torch.full((B, c.top_k), -7, dtype=torch.int32, device="cuda")
        L.csa_decode(c, pos, cache, T["q"][:, 0], None if wl.hca else T["q_idx"][:, 0],
                     None if wl.hca else T["w"][:, 0], T["sink"], out, topk)
        torch.cuda.synchronize()
        assert L.csa_get_device_status() == 0
        assert not torch.isnan(out).any()
        rng = np.random.default_rng(cid)
        n = wl.n_entries
        for b in (0, B - 1):
            entries = sorted({0, 1, n - 1, *rng.integers(0, n, 6).tolist()} | ({e_close} if closes else set()))
            _check_entries_sampled(wl, T, cache, b, entries, wl.name)
        for b in range(B):                              # the selection and output of every request
            sel = None if wl.hca else topk[b].cpu().numpy()
            _check_query(wl, o, T, cache, b, 0, t, sel, Hn.host64(out[b]), wl.name)
    finally:
        del T
        torch.cuda.empty_cache()


def test_full_size_prefill_sampled():
    L = Hn.lib()
    bench = _bench()
    wl = synth.WORKLOADS[2]
    c, o = Hn.configs(wl)
    T = bench.device_inputs(wl, [0], "cuda")
    try:
        cache = bench.make_cache(T, wl, "cuda")
        out = torch.full((1, wl.S, c.H, c.d), float("nan"), dtype=c.dtype, device="cuda")
        topk = torch.full((1, wl.S, c.top_k), -7, dtype=torch.int32, device="cuda")
        L.csa_prefill(c, cache, T["q"], T["q_idx"], T["w"], T["sink"], out, topk)
        torch.cuda.synchronize()
        assert L.csa_get_device_status() == 0
        assert not torch.isnan(out).any()
        rng = np.random.default_rng(2)
        n = wl.n_entries
        _check_entries_sampled(wl, T, cache, 0, sorted({0, 1, n - 1, *rng.integers(0, n, 6).tolist()}), wl.name)
        # group boundaries (3 -> 4 tokens makes entry 0 visible), the window edge, the last query,
        # and around 24 sampled points every query from two groups before to two groups after
        # (each crosses group boundaries): 256 queries or more
        ts = {0, 1, 2, 3, 4, 5, 7, 8, 126, 127, 128, 129, 2047, 2048, 4095, 4096, wl.S - 1}
        for p0 in rng.integers(8, wl.S - 8, 24).tolist():
            ts |= set(range(p0 - 2 * wl.ratio, p0 + 2 * wl.ratio + 1))
        ts = sorted(t for t in ts if 0 <= t < wl.S)
        assert len(ts) >= 256
        outh = Hn.host64(out[0, ts])
        tk = topk[0, ts].cpu().numpy()
        for i, t in enumerate(ts):
            _check_query(wl, o, T, cache, 0, t, t, tk[i], outh[i], wl.name)
    finally:
        del T
        torch.cuda.empty_cache()


def test_full_size_decode_end_to_end():
    """One request of the B = 32, N = 65,536 decode through the oracle from its raw inputs, not
    stage-chained: the oracle compresses all 65,536 tokens itself (fp64), and
      * every compressed entry of the GPU's caches is within one bf16 rounding of the oracle's;
      * the GPU's selection equals the oracle's selection on the oracle's own caches, except swaps
        among entries whose oracle scores lie within the bf16 cache-rounding band of the k-th
        score (the selection is made on caches that differ by one rounding, so near-ties can swap);
      * the GPU's output equals the oracle's attention over the oracle's caches for that selection.
    The raw rows are the synthetic inputs copied back from the device."""
    L = Hn.lib()
    bench = _bench()
    wl = synth.WORKLOADS[1]
    c, o = Hn.configs(wl)
    B, t, m = wl.B, wl.t, wl.ratio
    T = bench.device_inputs(wl, list(range(B)), "cuda")
    try:
        cache = bench.make_cache(T, wl, "cuda")
        L.csa_compress(c, cache, 0, wl.n_entries)
        e_close = t // m
        cache.ckv[:, e_close] = float("nan")
        cache.cidx[:, e_close] = float("nan")
        pos = torch.full((B,), t, dtype=torch.int64, device="cuda")
        out = torch.full((B, c.H, c.d), float("nan"), dtype=c.dtype, device="cuda")
        topk = torch.full((B, c.top_k), -7, dtype=torch.int32, device="cuda")
        L.csa_decode(c, pos, cache, T["q"][:, 0], T["q_idx"][:, 0], T["w"][:, 0], T["sink"], out, topk)
        torch.cuda.synchronize()
        assert L.csa_get_device_status() == 0
        b = 0
        bias, ibias = Hn.host64(T["bias"]), Hn.host64(T["idx_bias"])
        kv = Hn.host64(T["kv"][b])
        ckv_o = O.compress(kv, Hn.host64(T["gate"][b]), bias, m, wl.n_entries)
        cidx_o = O.compress(Hn.host64(T["idx_k"][b]), Hn.host64(T["idx_gate"][b]), ibias, m, wl.n_entries)
        Hn.check_entries(Hn.host64(cache.ckv[b]), ckv_o, "bf16", "end-to-end ckv")
        Hn.check_entries(Hn.host64(cache.cidx[b]), cidx_o, "bf16", "end-to-end cidx")
        q, q_idx, w = (Hn.host64(T[k][b, 0]) for k in ("q", "q_idx", "w"))
        sink = Hn.host64(T["sink"])
        ref_s = O.index_scores(q_idx, w, cidx_o, t, m)
        want = O.topk_select(ref_s, c.top_k)
        got = topk[b].cpu().numpy()
        sk = ref_s[want[-1]]
        band = 2.0 ** -7 * max(abs(sk), float(np.sqrt(np.mean(ref_s * ref_s))))
        diff = set(int(i) for i in got) ^ set(int(i) for i in want)
        assert len(diff) <= 16, f"{len(diff)} entries differ from the oracle's own selection"
        for i in diff:
            assert abs(ref_s[i] - sk) <= band, f"entry {i}: score {ref_s[i]:.6g} outside the band around {sk:.6g}"
        ref = O.sparse_attn(q, kv, ckv_o, got, sink, t, o)
        Hn.check_attn(Hn.host64(out[b]), ref, "bf16", "end-to-end attention")
    finally:
        del T
        torch.cuda.empty_cache()
