"""fp64 oracle of the low-precision compressed-cache format: FP4 E2M1 latent + FP8 E4M3 RoPE tail.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s cpu_baseline /
reference arm may import this module; the CUDA library never does, and this module imports nothing
from it.

Source: [LAB41] "Lab tổng hợp DeepSeek-V4.1-Flash — chạy toàn trình 1A → 6B bằng NumPy", section
"3 Giải pháp" (and the diagram tab "3. MLA & FP4 KV (890B)"): the KV budget per token is priced with
FP4 E2M1 for the latent part of a cache entry and FP8 E4M3 for its RoPE tail. The page names the two
element formats and nothing else. Readings where it is silent (listed with the design notes):

* latent = the first d - d_rope dims of a compressed entry, RoPE tail = the last d_rope dims; the
  rule applies to both compressed caches (KV entries of width 512 and index entries of width 128);
  raw rows, queries and outputs keep their bf16 storage.
* E2M1 is used the way its published definition (OCP Microscaling Formats, MXFP4) uses it: blocks
  of 32 consecutive latent dims share one power-of-two scale X = 2**E stored as an E8M0 byte
  (E + 127), with E = floor(log2(max |x| over the block)) - 2 (2 = the largest E2M1 exponent),
  clamped to [-127, 127] (an all-zero block takes E = -127); each element is x / X rounded to the
  nearest E2M1 value, ties to the even code, magnitudes beyond 6 saturating to 6.
* E4M3 is the OCP FP8 format (exponent bias 7, 3 mantissa bits, no infinities, S.1111.111 = NaN,
  largest finite 448), rounded to nearest, ties to the even code, saturating to +-448; no scale.
* byte layout of one request's cache of n_cap entries (planes, entry-major inside each plane):
    plane 0: n_cap x (L / 2) bytes, byte j of an entry = latent dims 2j (low nibble), 2j+1 (high);
    plane 1: n_cap x d_rope bytes, byte j = tail dim j (E4M3 code);
    plane 2: n_cap x sb bytes, byte k < L / 32 = E8M0 scale of latent dims 32k .. 32k + 31, the
             rest zero; sb = the next power of two >= L / 32 (16 for L = 448, 2 for L = 64);
  with L = d - d_rope (scale byte 255 is E8M0's NaN). Requests follow one another at a stride of
  n_cap (L/2 + d_rope) + n_cap sb rounded up to 16 bytes.
"""
from __future__ import annotations

import math

import numpy as np

from .csa_oracle import compress, compress_entry

__all__ = [
    "E2M1_VALUES", "e2m1_decode", "e2m1_encode", "e4m3_decode", "e4m3_encode", "mx_exponent",
    "quantize_entries", "dequantize", "cache_layout", "pack_cache", "unpack_cache", "compress_lowp",
    "compress_entry_lowp", "lowp_round",
]

# E2M1: 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit; exponent 0 is subnormal (m * 0.5).
# Magnitudes by code 0..7, built from that definition.
E2M1_VALUES = np.array([(m * 0.5) if e == 0 else 2.0 ** (e - 1) * (1.0 + m / 2.0)
                        for e in range(4) for m in range(2)])


def e2m1_decode(code) -> np.ndarray:
    """Value of 4-bit E2M1 codes (bit 3 = sign)."""
    c = np.asarray(code, dtype=np.int64)
    v = E2M1_VALUES[c & 7]
    return np.where(c & 8, -v, v)


def _round_to_grid(a, grid):
    """Index of the grid value nearest to each a >= 0 (grid ascending, a within its range), ties to
    the even index."""
    hi = np.searchsorted(grid, a, side="left").clip(0, len(grid) - 1)
    lo = (hi - 1).clip(0)
    dlo, dhi = a - grid[lo], grid[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0))
    return np.where(pick_hi, hi, lo)


def e2m1_encode(y) -> np.ndarray:
    """4-bit E2M1 code of y: nearest value, ties to the even code, |y| > 6 saturates to 6."""
    y = np.asarray(y, dtype=np.float64)
    a = np.minimum(np.abs(y), 6.0)
    c = _round_to_grid(a, E2M1_VALUES)
    return (c | np.where(np.signbit(y), 8, 0)).astype(np.int64)


def _e4m3_table() -> np.ndarray:
    vals = np.empty(256)
    for c in range(256):
        s, e, m = c >> 7, (c >> 3) & 15, c & 7
        if e == 15 and m == 7:
            v = math.nan
        elif e == 0:
            v = m * 2.0 ** -9                       # subnormal: m/8 * 2^(1-7)
        else:
            v = 2.0 ** (e - 7) * (1.0 + m / 8.0)
        vals[c] = -v if s else v
    return vals


_E4M3 = _e4m3_table()
_E4M3_POS = _E4M3[:127]                             # codes 0..126: ascending, 0 .. 448


def e4m3_decode(code) -> np.ndarray:
    """Value of 8-bit E4M3 codes."""
    return _E4M3[np.asarray(code, dtype=np.int64) & 255]


def e4m3_encode(y) -> np.ndarray:
    """8-bit E4M3 code of y: nearest finite value, ties to the even code, |y| > 448 saturates."""
    y = np.asarray(y, dtype=np.float64)
    a = np.minimum(np.abs(y), 448.0)
    c = _round_to_grid(a, _E4M3_POS)
    return (c | np.where(np.signbit(y), 128, 0)).astype(np.int64)


def mx_exponent(block_amax) -> np.ndarray:
    """Shared exponent E of MX blocks with the given max |x|: floor(log2 amax) - 2, clamped to
    [-127, 127]; amax == 0 gives -127."""
    a = np.asarray(block_amax, dtype=np.float64)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0))) - 2
    # log2 of an exact power of two is exact in IEEE arithmetic; guard the float floor anyway
    e = np.where(2.0 ** (e + 2) > a, e - 1, e)
    e = np.where(2.0 ** (e + 3) <= a, e + 1, e)
    return np.where(a > 0, np.clip(e, -127, 127), -127).astype(np.int64)


def quantize_entries(x, d_rope: int = 64):
    """Codes of entries x [n, d]: (fp4 codes [n, L], E [n, L/32], fp8 codes [n, d_rope])."""
    x = np.asarray(x, dtype=np.float64)
    n, d = x.shape
    L = d - d_rope
    assert L % 32 == 0
    lat = x[:, :L].reshape(n, L // 32, 32)
    E = mx_exponent(np.abs(lat).max(axis=2))
    c4 = e2m1_encode(lat / np.exp2(E)[:, :, None]).reshape(n, L)
    c8 = e4m3_encode(x[:, L:])
    return c4, E, c8


def dequantize(c4, E, c8) -> np.ndarray:
    """Entries [n, d] from their codes (exact in fp64)."""
    n, L = c4.shape
    lat = (e2m1_decode(c4).reshape(n, L // 32, 32) * np.exp2(E)[:, :, None]).reshape(n, L)
    return np.concatenate([lat, e4m3_decode(c8)], axis=1)


def lowp_round(x, d_rope: int = 64) -> np.ndarray:
    """x as the low-precision cache holds it: quantise, then dequantise."""
    return dequantize(*quantize_entries(np.atleast_2d(x), d_rope)).reshape(np.shape(x))


def cache_layout(d: int, n_cap: int, d_rope: int = 64) -> dict:
    """Byte offsets of the three planes inside one request and the request stride."""
    L = d - d_rope
    nb = L // 32
    sb = 1 << max(0, (nb - 1).bit_length())
    p0 = 0
    p1 = n_cap * (L // 2)
    p2 = p1 + n_cap * d_rope
    stride = p2 + (n_cap * sb + 15) // 16 * 16
    return {"L": L, "nb": nb, "sb": sb, "fp4": p0, "fp8": p1, "scale": p2, "stride": stride}


def pack_cache(x, n_cap: int, d_rope: int = 64) -> np.ndarray:
    """Bytes of one request's cache holding entries x [n <= n_cap, d] (entries >= n are zero)."""
    x = np.asarray(x, dtype=np.float64)
    n, d = x.shape
    lay = cache_layout(d, n_cap, d_rope)
    L, nb, sb = lay["L"], lay["nb"], lay["sb"]
    c4, E, c8 = quantize_entries(x, d_rope)
    buf = np.zeros(lay["stride"], dtype=np.uint8)
    nib = (c4[:, 0::2] | (c4[:, 1::2] << 4)).astype(np.uint8)          # [n, L/2]
    buf[lay["fp4"]:lay["fp4"] + n * (L // 2)] = nib.reshape(-1)
    buf[lay["fp8"]:lay["fp8"] + n * d_rope] = c8.astype(np.uint8).reshape(-1)
    sc = np.zeros((n, sb), dtype=np.uint8)
    sc[:, :nb] = (E + 127).astype(np.uint8)
    buf[lay["scale"]:lay["scale"] + n * sb] = sc.reshape(-1)
    return buf


def unpack_cache(buf, d: int, n_cap: int, n: int | None = None, d_rope: int = 64,
                 entries=None) -> np.ndarray:
    """fp64 entries of one request's cache bytes (all n first entries, or the listed ones)."""
    buf = np.asarray(buf, dtype=np.uint8).reshape(-1)
    lay = cache_layout(d, n_cap, d_rope)
    L, nb, sb = lay["L"], lay["nb"], lay["sb"]
    idx = np.arange(n_cap if n is None else n) if entries is None else np.asarray(entries, np.int64)
    nib = buf[lay["fp4"]:lay["fp4"] + n_cap * (L // 2)].reshape(n_cap, L // 2)[idx].astype(np.int64)
    c4 = np.empty((len(idx), L), dtype=np.int64)
    c4[:, 0::2] = nib & 15
    c4[:, 1::2] = nib >> 4
    c8 = buf[lay["fp8"]:lay["fp8"] + n_cap * d_rope].reshape(n_cap, d_rope)[idx]
    sbyte = buf[lay["scale"]:lay["scale"] + n_cap * sb].reshape(n_cap, sb)[idx, :nb].astype(np.int64)
    out = dequantize(c4, sbyte - 127, c8)
    # E8M0 byte 255 is NaN (never written by a quantiser: E <= 127)
    nan_blk = np.repeat(sbyte == 255, 32, axis=1)
    out[:, :L][nan_blk] = np.nan
    return out


def compress_lowp(kv, gate, bias, ratio: int, n_entries: int | None = None, **kw) -> np.ndarray:
    """The compressor's entries (``compress``) as the low-precision cache holds them."""
    d_rope = kw.get("d_rope", 64)
    return lowp_round(compress(kv, gate, bias, ratio, n_entries, **kw), d_rope)


def compress_entry_lowp(kv_rows, gate_rows, bias, e: int, ratio: int, **kw) -> np.ndarray:
    """One entry (``compress_entry``) as the low-precision cache holds it."""
    d_rope = kw.get("d_rope", 64)
    return lowp_round(compress_entry(kv_rows, gate_rows, bias, e, ratio, **kw), d_rope)
