"""A NumPy model of the selection that the fused decode indexer runs across the CTAs of one cluster,
checked against the exact selection on many score distributions (no GPU).

A request's visible entries are split into C contiguous runs of 128-entry tiles, one per CTA. The
cluster finds the k-th largest key by radix select over 8-bit digits (most significant first):
in each pass every CTA histograms the keys of the current class into 256 bins and every CTA
receives all C histograms. From those tables alone each CTA reads the threshold bin, the number of
winners above it held by lower-ranked CTAs, and (at the end) the number of final-class keys held by
lower-ranked CTAs, which places its winners in the ascending-index output without another exchange.
The model follows those steps and must give exactly the (-score, index) top-k of the oracle,
listed in ascending entry index with -1 padding.
"""
import numpy as np
import pytest

from oracle import csa_oracle as O

TILE, BINS = 128, 256


def order_keys(scores):
    """fp32 -> 32-bit keys that order like the floats (-0 == +0; 0 is kept for 'no entry')."""
    u = np.asarray(scores, np.float32).view(np.uint32).astype(np.uint64)
    u = np.where(u == 0x80000000, 0, u)
    return np.where(u & 0x80000000, (~u) & 0xFFFFFFFF, u | 0x80000000)


def cluster_select_model(scores, k, C):
    V = len(scores)
    T = -(-V // TILE)
    keys = order_keys(scores)
    parts, starts = [], []
    for r in range(C):
        t0, t1 = r * T // C, (r + 1) * T // C
        lo, hi = t0 * TILE, min(V, t1 * TILE)
        starts.append(lo)
        parts.append(keys[lo:hi] if hi > lo else keys[:0])
    prefix = pmask = 0
    need = n_valid = 0
    gt_lower = [0] * C
    eq_lower = [0] * C
    take_all = False
    for p in range(4):
        shift = 24 - 8 * p
        table = np.zeros((C, BINS), np.int64)            # row r: CTA r's histogram of this pass
        for r, part in enumerate(parts):
            live = part[(part != 0) & ((part & pmask) == prefix)]
            table[r] = np.bincount(((live >> shift) & 255).astype(np.int64), minlength=BINS)
        tot = table.sum(axis=0)
        if p == 0:
            n_valid = int(tot.sum())
            need = min(k, n_valid)
            if need == n_valid:
                take_all = True
                for r in range(C):
                    gt_lower[r] = int(table[:r].sum())
                break
        above = 0
        for b in range(BINS - 1, -1, -1):                  # scan from the top bin
            if above < need <= above + tot[b]:
                bstar = b
                break
            above += int(tot[b])
        cls = int(tot[bstar])
        for r in range(C):
            gt_lower[r] += int(table[:r, bstar + 1:].sum())
            eq_lower[r] = int(table[:r, bstar].sum())
        need -= above
        prefix |= bstar << shift
        pmask |= 255 << shift
        if cls == need:
            break
    out = np.full(k, -1, np.int64)
    for r, part in enumerate(parts):
        m = part & pmask
        valid = part != 0
        above_m = valid & (take_all | (m > prefix))
        in_cls = valid & ~np.bool_(take_all) & (m == prefix)
        slot = gt_lower[r] + min(eq_lower[r], need)
        cpos = eq_lower[r]
        for i in range(len(part)):
            win = bool(above_m[i])
            if in_cls[i]:
                win = cpos < need
                cpos += 1
            if win:
                assert slot < k
                out[slot] = starts[r] + i
                slot += 1
    return out


def _expected(scores, k):
    want = O.topk_select(np.asarray(scores, np.float64), k)
    n = int((want >= 0).sum())
    return np.concatenate([np.sort(want[:n]), np.full(k - n, -1)])


@pytest.mark.parametrize("C", [1, 2, 4, 8])
@pytest.mark.parametrize("mode", ["normal", "equal", "few", "narrow", "signed", "zeros"])
@pytest.mark.parametrize("V,k", [(16384, 512), (5000, 512), (300, 512), (4097, 1024), (129, 64), (1, 1)])
def test_radix8_cluster_select_is_exact(C, mode, V, k):
    rng = np.random.default_rng(V * 7 + k + C + len(mode))
    if mode == "normal":
        s = rng.standard_normal(V).astype(np.float32) * np.float32(0.03)
    elif mode == "equal":
        s = np.full(V, 0.25, np.float32)
    elif mode == "few":
        s = rng.choice(np.float32([-0.5, 0.125, 0.1251, 2.0]), size=V)
    elif mode == "narrow":
        s = (1.0 + rng.standard_normal(V) * 1e-6).astype(np.float32)
    elif mode == "signed":
        s = -np.abs(rng.standard_normal(V)).astype(np.float32)
    else:
        s = np.where(rng.random(V) < 0.5, np.float32(0.0), np.float32(-0.0)).astype(np.float32)
    if -(-V // TILE) / C > 32:
        pytest.skip("more than 32 tiles per CTA")
    got = cluster_select_model(s, k, C)
    assert np.array_equal(got, _expected(s, k))
