"""Pins of the low-precision cache oracle (FP4 E2M1 latent with a shared power-of-two scale per
32 dims, FP8 E4M3 RoPE tail) against the element formats' definitions, hand-worked values and
brute force."""
import json
import math
import os

import numpy as np
import pytest

from oracle import cache_lowp as Q
from oracle import csa_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _g():
    return json.load(open(os.path.join(GOLDEN, "lowp_formats.json")))


def test_decode_tables_match_hand_values():
    g = _g()
    np.testing.assert_array_equal(Q.E2M1_VALUES, g["e2m1_magnitudes_by_code"])
    np.testing.assert_array_equal(Q.e2m1_decode(np.arange(8, 16)), -np.array(g["e2m1_magnitudes_by_code"]))
    for code, v in g["e4m3_codes"].items():
        assert Q.e4m3_decode(int(code)) == v, code
    assert math.isnan(Q.e4m3_decode(0x7F)) and math.isnan(Q.e4m3_decode(0xFF))
    # every finite E4M3 value is the sign times 2^(e-7) (1 + m/8), or m 2^-9 below 2^-6
    vals = Q.e4m3_decode(np.arange(256))
    fin = ~np.isnan(vals)
    assert fin.sum() == 254 and np.nanmax(vals) == 448.0 and np.nanmin(vals) == -448.0


def _nearest_even(a, grid):
    """Brute force: the grid index nearest to a, ties to the even index."""
    d = np.abs(grid[None, :] - a[:, None])
    best = d.min(axis=1, keepdims=True)
    cand = d == best
    idx = np.argmax(cand, axis=1)
    two = cand.sum(axis=1) == 2
    idx2 = len(grid) - 1 - np.argmax(cand[:, ::-1], axis=1)
    return np.where(two & (idx % 2 == 1), idx2, idx)


def test_e2m1_encode_is_nearest_ties_to_even_and_saturates():
    g = _g()
    for y, v in g["e2m1_round_half_even"].items():
        assert Q.e2m1_decode(Q.e2m1_encode(float(y))) == v, y
        assert Q.e2m1_decode(Q.e2m1_encode(-float(y))) == -v, y
    rng = np.random.default_rng(5)
    mids = (Q.E2M1_VALUES[1:] + Q.E2M1_VALUES[:-1]) / 2
    a = np.concatenate([rng.uniform(0, 6, 4000), mids, Q.E2M1_VALUES])
    np.testing.assert_array_equal(Q.e2m1_encode(a), _nearest_even(a, Q.E2M1_VALUES))
    np.testing.assert_array_equal(Q.e2m1_encode(-a) & 7, _nearest_even(a, Q.E2M1_VALUES))
    assert Q.e2m1_decode(Q.e2m1_encode(1e30)) == 6.0 and Q.e2m1_decode(Q.e2m1_encode(-7.0)) == -6.0


def test_e4m3_encode_is_nearest_ties_to_even_and_saturates():
    rng = np.random.default_rng(6)
    pos = Q.e4m3_decode(np.arange(127))
    mids = (pos[1:] + pos[:-1]) / 2
    a = np.concatenate([np.exp(rng.uniform(-12, 6.2, 6000)), mids, pos])
    a = np.minimum(a, 448.0)
    np.testing.assert_array_equal(Q.e4m3_encode(a), _nearest_even(a, pos))
    assert Q.e4m3_decode(Q.e4m3_encode(1e9)) == 448.0 and Q.e4m3_decode(Q.e4m3_encode(-500.0)) == -448.0
    # every finite code survives decode -> encode
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)])
    np.testing.assert_array_equal(Q.e4m3_encode(Q.e4m3_decode(codes)), codes)


def test_mx_exponent_hand_values_and_range():
    for amax, e in _g()["mx_shared_exponent"].items():
        assert Q.mx_exponent(float(amax)) == e, amax
    assert Q.mx_exponent(2.0 ** 200) == 127 and Q.mx_exponent(2.0 ** -200) == -127
    rng = np.random.default_rng(7)
    a = np.exp(rng.uniform(-30, 30, 5000))
    E = Q.mx_exponent(a)
    r = a / np.exp2(E)
    assert np.all((r >= 4.0) & (r < 8.0))          # scaled block max in [4, 8): top binade of E2M1


def test_block_error_bound_and_idempotence():
    rng = np.random.default_rng(8)
    x = rng.standard_normal((64, 512)) * np.exp(rng.uniform(-6, 6, (64, 1)))
    c4, E, c8 = Q.quantize_entries(x)
    y = Q.dequantize(c4, E, c8)
    X = np.repeat(np.exp2(E), 32, axis=1)
    amax = np.repeat(np.abs(x[:, :448]).reshape(64, 14, 32).max(axis=2), 32, axis=1)
    err = np.abs(y[:, :448] - x[:, :448])
    # spacing of E2M1 is at most 2 (between 4 and 6): error <= X, or the saturation excess
    assert np.all(err <= np.maximum(X, amax - 6 * X) * (1 + 1e-15))
    tail = x[:, 448:]
    rel = np.abs(y[:, 448:] - tail)
    # E4M3: half a spacing (2^-4 relative in the normal range, 2^-10 absolute below 2^-6), or the
    # saturation excess beyond 448
    bound = np.maximum(np.maximum(np.abs(tail) * 2.0 ** -4, 2.0 ** -10), np.abs(tail) - 448.0)
    assert np.all(rel <= bound * (1 + 1e-15))
    np.testing.assert_array_equal(Q.lowp_round(y), y)


def test_pack_hand_bytes_and_round_trip():
    x = np.zeros((3, 512))
    x[1, 0], x[1, 1] = 4.0, -1.0                  # block 0 of entry 1: amax 4 -> E = 0
    x[1, 448] = 1.0
    buf = Q.pack_cache(x, n_cap=5)
    lay = Q.cache_layout(512, 5)
    assert lay["stride"] == 5 * 288 + 80 and lay["sb"] == 16
    assert buf[lay["fp4"] + 224] == 0xA6          # dim 0 -> 4.0 = code 6 (low), dim 1 -> -1.0 = 0xA
    assert buf[lay["scale"] + 16] == 127          # E8M0 of E = 0
    assert buf[lay["scale"]] == 0                 # an all-zero block: E = -127
    assert buf[lay["fp8"] + 64] == 0x38           # tail dim 0 of entry 1: 1.0
    rng = np.random.default_rng(9)
    for d in (512, 128):
        z = rng.standard_normal((7, d))
        b = Q.pack_cache(z, n_cap=9)
        assert b.size == Q.cache_layout(d, 9)["stride"] and b.size % 16 == 0
        np.testing.assert_array_equal(Q.unpack_cache(b, d, 9, 7), Q.lowp_round(z))
        np.testing.assert_array_equal(Q.unpack_cache(b, d, 9, entries=[6, 2]), Q.lowp_round(z)[[6, 2]])
    # E8M0 255 is NaN: a block whose scale byte is 255 decodes to NaN, the other blocks do not
    b = Q.pack_cache(rng.standard_normal((2, 512)), n_cap=2)
    b[Q.cache_layout(512, 2)["scale"] + 16 + 3] = 255
    y = Q.unpack_cache(b, 512, 2)
    assert np.isnan(y[1, 96:128]).all() and not np.isnan(np.delete(y[1], np.s_[96:128])).any()


def test_compress_lowp_is_the_rounded_compressor():
    rng = np.random.default_rng(10)
    m, N = 4, 32
    kv, g = rng.standard_normal((N, 512)) / 22.6, rng.standard_normal((N, 512))
    bias = rng.standard_normal((2 * m, 512)) * 0.1
    full = O.compress(kv, g, bias, m)
    lp = Q.compress_lowp(kv, g, bias, m)
    np.testing.assert_array_equal(lp, Q.lowp_round(full))
    e = 5
    one = Q.compress_entry_lowp(kv[(e - 1) * m:(e + 1) * m], g[(e - 1) * m:(e + 1) * m], bias, e, m)
    # the single-entry form rounds the same fp64 entry (up to its own summation order): the codes
    # agree except where an element sits on a rounding boundary
    assert np.mean(one == lp[e]) > 0.99
    # entries after RMSNorm hold unit mean square: the latent's block scales sit near 2^-2 .. 2^0
    E = Q.quantize_entries(full)[1]
    assert E.min() >= -6 and E.max() <= 1
