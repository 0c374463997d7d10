"""Shared test plumbing: seeded inputs on the device, the oracle on the same values, and the
tolerance checks. Test infrastructure only (imports the oracle)."""
from __future__ import annotations

import math

import numpy as np
import torch

import synth
from oracle import cache_lowp as Q
from oracle import csa_oracle as O

# Tolerances (see the design notes): indexer |ds| <= 1e-3 * max(|s_ref|, rms_row(s_ref)); attention
# max|do| / max|o_ref| per (request, query, head) <= 1e-2 for bf16 storage and 1e-5 for float32;
# compressed entries are one bf16 rounding (2^-8 relative, i.e. one ulp) or 1e-5 for float32.
ATTN_TOL = {"bf16": 1e-2, "f32": 1e-5, "fp4": 1e-2}
SCORE_TOL = {"bf16": 1e-3, "f32": 1e-5, "fp4": 1e-3}
TIE_TOL = 1e-4


def lib():
    import long_context_sparse_19_b300 as L
    return L


def configs(wl: synth.Workload, simt: bool = False):
    L = lib()
    c = L.Config(H=wl.H, d=wl.d, d_rope=wl.d_rope, H_idx=wl.H_idx, d_idx=wl.d_idx, ratio=wl.ratio,
                 top_k=wl.top_k, window=wl.window, storage=wl.storage, simt=simt)
    o = O.OracleConfig(H=wl.H, d=wl.d, d_rope=wl.d_rope, H_idx=wl.H_idx, d_idx=wl.d_idx, ratio=wl.ratio,
                       top_k=wl.top_k, window=wl.window)
    return c, o


def dev(a: np.ndarray, storage: str, device="cuda") -> torch.Tensor:
    """float32 host values (already representable in the storage type) -> device tensor."""
    if storage != "f32":
        bits = synth.bf16_bits(a).view(np.int16)
        return torch.from_numpy(bits).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(device)


def host64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


class DeviceBatch:
    """Every tensor of a workload's B requests on the GPU, plus the host copies the oracle reads."""

    def __init__(self, wl: synth.Workload, requests=None, device="cuda"):
        self.wl = wl
        self.reqs = synth.gen_requests(wl, requests)
        self.shared = synth.gen_shared(wl)
        st = wl.storage
        stack = lambda k: np.stack([r[k] for r in self.reqs])
        self.kv = dev(stack("kv"), st)
        self.gate = dev(stack("gate"), st)
        self.bias = torch.from_numpy(self.shared["bias"]).to(device)
        self.sink = torch.from_numpy(self.shared["sink"]).to(device)
        self.q = dev(stack("q"), st)
        B = len(self.reqs)
        n_cap = self.n_cap = wl.n_entries
        self.lowp = st == "fp4"
        dt = torch.float32 if st == "f32" else torch.bfloat16
        # caches start poisoned: NaN, or with fp4 storage 0xFF bytes (NaN scale and NaN tail codes)
        new_cache = (lambda C: torch.full((B, Q.cache_layout(C, n_cap)["stride"]), 255, dtype=torch.uint8,
                                          device=device)) if self.lowp else \
            (lambda C: torch.full((B, n_cap, C), float("nan"), dtype=dt, device=device))
        self.ckv = new_cache(wl.d)
        if wl.hca:
            self.idx_k = self.idx_gate = self.idx_bias = self.cidx = self.q_idx = self.w = None
        else:
            self.idx_k = dev(stack("idx_k"), st)
            self.idx_gate = dev(stack("idx_gate"), st)
            self.idx_bias = torch.from_numpy(self.shared["idx_bias"]).to(device)
            self.cidx = new_cache(wl.d_idx)
            self.q_idx = dev(stack("q_idx"), st)
            self.w = torch.from_numpy(stack("w")).to(device)

    @property
    def B(self):
        return len(self.reqs)

    def cache(self):
        L = lib()
        return L.Cache(kv=self.kv, gate=self.gate, gate_bias=self.bias, ckv=self.ckv, idx_k=self.idx_k,
                       idx_gate=self.idx_gate, idx_bias=self.idx_bias, cidx=self.cidx, n_cap=self.n_cap)

    def entries(self, which: int) -> np.ndarray:
        """fp64 [B, n_cap, C] values of a compressed cache as the GPU holds it (fp4 caches decoded by
        the oracle's unpacker)."""
        t = self.cidx if which else self.ckv
        if not self.lowp:
            return host64(t)
        C = self.wl.d_idx if which else self.wl.d
        raw = t.cpu().numpy()
        return np.stack([Q.unpack_cache(raw[b], C, self.n_cap) for b in range(self.B)])

    def poison_from(self, b: int, e0: int) -> None:
        """Entries >= e0 of request b become NaN (every plane of an fp4 cache: 0xFF bytes)."""
        for which, t in ((0, self.ckv), (1, self.cidx)):
            if t is None:
                continue
            if not self.lowp:
                t[b, e0:] = float("nan")
                continue
            C = self.wl.d_idx if which else self.wl.d
            lay = Q.cache_layout(C, self.n_cap)
            L, R, sb = lay["L"] // 2, C - lay["L"], lay["sb"]
            t[b, e0 * L:self.n_cap * L] = 255
            t[b, lay["fp8"] + e0 * R:lay["fp8"] + self.n_cap * R] = 255
            t[b, lay["scale"] + e0 * sb:lay["scale"] + self.n_cap * sb] = 255


# ------------------------------------------------------------------------------------ checks
def check_entries(got: np.ndarray, ref: np.ndarray, storage: str, what: str):
    if storage == "fp4":
        return check_entries_lowp(got, ref, what)
    if storage == "bf16":
        bad = np.abs(got - ref) > 2.0 ** -8 * np.abs(ref) + 1e-6
    else:
        bad = np.abs(got - ref) > 1e-5 * np.maximum(1.0, np.abs(ref))
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} elements off; max err " \
                          f"{np.abs(got - ref).max():.3g}"


def check_entries_lowp(got: np.ndarray, ref: np.ndarray, what: str, d_rope: int = 64):
    """GPU entries held in the FP4 / FP8 cache (decoded, fp64 [n, C] or [C]) against the oracle's fp64
    entries ref: every element must be the format's rounding of a value within the fp32 computing
    error delta of ref (the GPU computes the entry in fp32 and rounds that), under a block scale that
    is the oracle's or, where the block max lies within delta of a power of two, its neighbour; and
    nearly all elements must equal the rounding of ref itself."""
    got, ref = np.atleast_2d(got), np.atleast_2d(ref)
    n, C = ref.shape
    L = C - d_rope
    delta = 1e-5 * np.maximum(np.abs(ref), 1.0)
    lat, glat = ref[:, :L].reshape(n, L // 32, 32), got[:, :L].reshape(n, L // 32, 32)
    amax = np.abs(lat).max(axis=2)
    e_lo, e_hi = Q.mx_exponent(amax * (1 - 1e-5)), Q.mx_exponent(amax * (1 + 1e-5))
    # the GPU's scale of each block: the power of two that makes its largest code's block consistent
    ok = np.zeros(glat.shape, dtype=bool)
    dl = delta[:, :L].reshape(glat.shape)
    for E in np.unique(np.concatenate([e_lo.ravel(), e_hi.ravel()])):
        X = 2.0 ** E
        lo = Q.e2m1_decode(Q.e2m1_encode((lat - dl) / X)) * X
        hi = Q.e2m1_decode(Q.e2m1_encode((lat + dl) / X)) * X
        allowed = ((E >= e_lo) & (E <= e_hi))[:, :, None]
        ok |= allowed & (glat >= lo) & (glat <= hi)
    assert ok.all(), f"{what}: {(~ok).sum()} of {ok.size} latent elements are no rounding of the oracle's"
    tl, gt = ref[:, L:], got[:, L:]
    lo = Q.e4m3_decode(Q.e4m3_encode(tl - delta[:, L:]))
    hi = Q.e4m3_decode(Q.e4m3_encode(tl + delta[:, L:]))
    bad = ~((gt >= lo) & (gt <= hi))
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} tail elements are no rounding of the oracle's"
    same = np.mean(got == Q.lowp_round(ref, d_rope))
    assert same >= 0.99, f"{what}: only {same:.4f} of the elements equal the rounding of the oracle's entry"


def check_scores(got: np.ndarray, ref: np.ndarray, storage: str, what: str):
    assert got.shape == ref.shape, f"{what}: {got.shape} scores, oracle {ref.shape}"
    if got.size == 0:                               # nothing visible yet
        return
    scale = max(np.sqrt(np.mean(ref * ref)), 1e-30)
    err = np.abs(got - ref) / np.maximum(np.abs(ref), scale)
    assert err.max() <= SCORE_TOL[storage], f"{what}: max relative score error {err.max():.3g}"


def check_topk_exact(got: np.ndarray, scores: np.ndarray, k: int, what: str):
    """The GPU selection equals the exact (-score, index) selection on the same float32 scores,
    listed in ascending entry index with -1 in the unused slots."""
    want = O.topk_select(scores, k)
    n = int((want >= 0).sum())
    exp = np.concatenate([np.sort(want[:n]), np.full(k - n, -1, dtype=want.dtype)])
    assert np.array_equal(got, exp), f"{what}: top-k differs from the exact selection on its scores"


def check_topk_vs_oracle(got: np.ndarray, ref_scores: np.ndarray, k: int, what: str):
    """Set equality with the oracle's selection, except swaps among entries whose oracle scores lie
    within TIE_TOL * |s_k| of the k-th score."""
    want = O.topk_select(ref_scores, k)
    g = set(int(i) for i in got if i >= 0)
    w = set(int(i) for i in want if i >= 0)
    assert len(g) == len(w), f"{what}: {len(g)} selected, oracle {len(w)}"
    if g == w:
        return
    sk = ref_scores[want[min(k, len(w)) - 1]]
    band = TIE_TOL * max(abs(sk), 1e-30)
    for i in g ^ w:
        assert abs(ref_scores[i] - sk) <= band, \
            f"{what}: entry {i} (score {ref_scores[i]:.6g}) differs from the oracle selection beyond " \
            f"the tie band around s_k = {sk:.6g}"


def check_attn(got: np.ndarray, ref: np.ndarray, storage: str, what: str):
    """got/ref: [H, d] for one query."""
    num = np.abs(got - ref).max(axis=1)
    den = np.maximum(np.abs(ref).max(axis=1), 1e-30)
    rel = num / den
    assert rel.max() <= ATTN_TOL[storage], f"{what}: max relative attention error {rel.max():.3g} " \
                                           f"(head {int(rel.argmax())})"
