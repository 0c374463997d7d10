"""The tolerant check of FP4 / FP8 cache entries (tests/_harness.py) accepts the oracle's own
rounding and values rounded from within fp32 error of the entry, and rejects a wrong rounding, a
wrong block scale and a wrong tail code (CPU only)."""
import numpy as np
import pytest

from oracle import cache_lowp as Q
from tests import _harness as Hn


def _entries():
    rng = np.random.default_rng(12)
    x = rng.standard_normal((6, 512))
    return x / np.sqrt(np.mean(x * x, axis=1, keepdims=True))


def test_accepts_the_rounding_and_near_boundary_roundings():
    x = _entries()
    Hn.check_entries_lowp(Q.lowp_round(x), x, "exact")
    Hn.check_entries_lowp(Q.lowp_round(x * (1 + 3e-6)), x, "within fp32 error")


def test_rejects_wrong_codes_and_scales():
    x = _entries()
    y = Q.lowp_round(x)
    z = y.copy()
    z[0, 3] += 0.5 * np.sign(z[0, 3] + 1e-9) * 2.0 ** Q.quantize_entries(x)[1][0, 0]   # one code step
    with pytest.raises(AssertionError):
        Hn.check_entries_lowp(z, x, "code")
    c4, E, c8 = Q.quantize_entries(x)
    E2 = E.copy()
    E2[1, 2] += 1                                       # a doubled block scale
    with pytest.raises(AssertionError):
        Hn.check_entries_lowp(Q.dequantize(c4, E2, c8), x, "scale")
    c8b = c8.copy()
    c8b[2, 5] ^= 1                                      # the next E4M3 code of one tail dim
    with pytest.raises(AssertionError):
        Hn.check_entries_lowp(Q.dequantize(c4, E, c8b), x, "tail")
