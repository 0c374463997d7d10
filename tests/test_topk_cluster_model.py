"""A NumPy model of the exchange that the one-cluster top-k performs, checked against the exact
selection on many score distributions (no GPU).

The CUDA kernel splits a row of up to 8 x 2048 scores over the CTAs of a cluster. Two shortcuts
make it fast, and each rests on an argument that this model checks numerically:
  * a CTA adds to the cluster histogram only the bins at or above the bin of its own k-th largest
    key: the row's k-th largest key is at least as large as any part's k-th largest key, so the
    threshold bin and every bin above it are still counted exactly;
  * the output offsets of a CTA (items above the threshold bin, and in it, held by lower-ranked
    CTAs) are read from a second histogram that only lower-ranked CTAs add to, instead of a separate
    exchange of counts;
then the in-bin keys are gathered in row order into one short list, whose remaining digits are
resolved locally, and ties go to the lower index. The model follows those steps with the same
digit widths (11, 11, 10 bits) and list capacity, and must select exactly the (-score, index)
top-k of the oracle.
"""
import numpy as np
import pytest

from oracle import csa_oracle as O

BINS, CHUNK, LIST_CAP = 2048, 2048, 1024
DIGITS = ((21, 2047), (10, 2047), (0, 1023))       # (shift, mask) of the three digit passes


def order_keys(scores):
    """fp32 -> 32-bit keys that order like the floats (0 is kept for 'no entry')."""
    u = np.asarray(scores, np.float32).view(np.uint32).astype(np.uint64)
    return np.where(u & 0x80000000, (~u) & 0xFFFFFFFF, u | 0x80000000)


def find_bin(hist, need):
    """Bin of the need-th largest item, items still needed from it, its count (scan from the top)."""
    run = 0
    for b in range(len(hist) - 1, -1, -1):
        if run < need <= run + hist[b]:
            return b, need - run, int(hist[b])
        run += int(hist[b])
    raise AssertionError("need exceeds the histogram")


def cluster_model(keys, k):
    n = len(keys)
    C = (n + CHUNK - 1) // CHUNK
    parts = [keys[r * CHUNK:(r + 1) * CHUNK] for r in range(C)]
    full = [np.zeros(BINS, np.int64) for _ in DIGITS]
    before = [np.zeros(BINS, np.int64) for _ in range(C)]          # first digit, lower ranks only
    n_valid = int((keys != 0).sum())
    need, take_all = min(k, n_valid), k >= n_valid
    prefix = pmask = 0
    cls, last = 0, 0
    for p, (sh, dm) in enumerate(DIGITS):
        last = p
        for r, part in enumerate(parts):
            live = part[(part != 0) & ((part & pmask) == prefix)]
            h = np.bincount(((live >> sh) & dm).astype(np.int64), minlength=BINS)
            if p == 0:
                nl = int((part != 0).sum())
                if nl > k:                                           # bins below its own k-th are not sent
                    h[:find_bin(h, k)[0]] = 0
                for r2 in range(r + 1, C):
                    before[r2] += h
            full[p] += h
        if p == 0 and take_all:
            break
        b, need, cls = find_bin(full[p], need)
        prefix |= b << sh
        pmask |= dm << sh
        if cls == need or cls <= LIST_CAP:
            break
    split = not take_all and cls > need and pmask != 0xFFFFFFFF
    # per-CTA counts, and offsets: from `before` when the first digit decided, else exchanged counts
    gt = [int(((part != 0) & (take_all | ((part & pmask) > prefix))).sum()) for part in parts]
    eq = [0 if take_all else int(((part != 0) & ((part & pmask) == prefix)).sum()) for part in parts]
    for r in range(C):
        if last == 0:
            bstar = prefix >> 21
            gt_off = int(before[r].sum() if take_all else before[r][bstar + 1:].sum())
            eq_off = 0 if take_all else int(before[r][bstar])
            assert (gt_off, eq_off) == (sum(gt[:r]), sum(eq[:r])), "offsets from the second histogram"
    in_bin = [kv for part in parts for kv in part if kv != 0 and not take_all and (kv & pmask) == prefix]
    taken = None
    if split:
        assert len(in_bin) <= LIST_CAP
        lp, lm, ln = prefix, pmask, need
        arr = np.array(in_bin, np.uint64)
        for sh, dm in DIGITS[last + 1:]:
            live = arr[(arr & lm) == lp]
            b, ln, c = find_bin(np.bincount(((live >> sh) & dm).astype(np.int64), minlength=BINS), ln)
            lp |= b << sh
            lm |= dm << sh
            if c == ln:
                break
        taken, seen = [], 0
        for kv in in_bin:
            m = kv & lm
            taken.append(m > lp or (m == lp and seen < ln))
            seen += m == lp
    out, pos = [], 0
    for r, part in enumerate(parts):
        for i, kv in enumerate(part):
            if kv == 0:
                continue
            m = kv & pmask
            if take_all or m > prefix:
                out.append(r * CHUNK + i)
            elif m == prefix:
                if cls <= need or (taken[pos] if split else pos < need):
                    out.append(r * CHUNK + i)
                pos += 1
    return np.array(out, np.int64)


@pytest.mark.parametrize("n", [2049, 6000, 16384])
@pytest.mark.parametrize("k", [1, 512, 2048, 5000])
@pytest.mark.parametrize("dist", ["normal", "narrow", "few", "equal", "invalid_tail", "one_part_heavy"])
def test_cluster_exchange_model_selects_exactly(n, k, dist):
    rng = np.random.default_rng(n * 7 + k + len(dist))
    x = rng.standard_normal(n).astype(np.float32)
    if dist == "narrow":
        x = (1 + 1e-4 * rng.standard_normal(n)).astype(np.float32)
    elif dist == "few":
        x = rng.integers(0, 37, n).astype(np.float32)
    elif dist == "equal":
        x = np.full(n, 0.5, np.float32)
    elif dist == "one_part_heavy":                     # every large score in the last part
        x[-CHUNK:] += 10.0
    keys = order_keys(x)
    if dist == "invalid_tail":
        keys[n // 3:] = 0
    got = cluster_model(keys, k)
    valid = np.nonzero(keys)[0]
    want = np.sort(O.topk_select(x[valid].astype(np.float64), k))
    want = valid[want[want >= 0]]
    assert np.array_equal(got, np.sort(want))
