"""Seeded synthetic inputs for the compressed-sparse-attention path.

This module holds no arithmetic of the method: it only draws random numbers, rounds them to the
storage type and describes the workload shapes. Both the test oracle and the CUDA path consume
exactly what it returns.

Recipe: every request b of workload id c draws from
``Generator(PCG64(SeedSequence([seed, c, b])))`` in the order kv, gate, idx_k, idx_gate, q,
q_idx, w; the tensors shared by all requests (gate bias, index-gate bias, sink) draw from
``SeedSequence([seed, c, 1 << 20])``. Values are drawn in float32 as ``sigma * N(0, 1)`` and,
for bf16 storage, rounded to the nearest bf16 (ties to even). N(0, v) below means variance v.

=========  ==================  ===========================================================
tensor     shape               distribution
=========  ==================  ===========================================================
kv         [N, d]              N(0, 1/d)            raw shared KV head (K = V)
gate       [N, d]              N(0, 1)              compressor gate logits
bias       [2m, d]             N(0, 0.1)            compressor positional gate bias
idx_k      [N, d_I]            N(0, 1/d_I)          raw index keys
idx_gate   [N, d_I]            N(0, 1)              index-key gate logits
idx_bias   [2m, d_I]           N(0, 0.1)
q          [S, H, d]           N(0, 1/d) * q_gain   query heads (before RoPE)
q_idx      [S, H_I, d_I]       N(0, 1/d_I)          indexer query heads (before RoPE)
w          [S, H_I]            N(0, 1)/sqrt(d_I)/sqrt(H_I)   signed indexer head weights
sink       [H]                 N(0, 1)              per-head sink logits
=========  ==================  ===========================================================
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, replace

import numpy as np

__all__ = ["Workload", "WORKLOADS", "round_bf16", "bf16_bits", "bits_to_f32",
           "gen_shared", "gen_request", "gen_requests", "small_workload"]


@dataclass(frozen=True)
class Workload:
    name: str
    wid: int                 # workload id used in the seed
    B: int                   # requests
    N: int                   # raw tokens held per request
    S: int                   # queries per request (1 = decode at t, N = causal prefill)
    t: int | None            # decode position (None for prefill)
    H: int = 64
    d: int = 512
    d_rope: int = 64
    H_idx: int = 64
    d_idx: int = 128
    ratio: int = 4
    top_k: int = 512         # 0 = HCA
    window: int = 128
    storage: str = "bf16"    # "f32" | "bf16" | "fp4" (bf16 raw rows, FP4 / FP8 compressed caches)
    q_gain: float = 1.0      # > 1 sharpens the attention softmax (test variants)
    seed: int = 0

    @property
    def hca(self) -> bool:
        return self.top_k == 0

    @property
    def decode(self) -> bool:
        return self.t is not None

    @property
    def n_entries(self) -> int:
        """compressed-cache capacity in entries"""
        return self.N // self.ratio

    def positions(self) -> np.ndarray:
        return np.array([self.t], np.int64) if self.decode else np.arange(self.S, dtype=np.int64)


WORKLOADS = {
    0: Workload("csa_decode_tiny_f32_B1_N2048_H8_k64", 0, B=1, N=2048, S=1, t=2047, H=8, H_idx=8,
                top_k=64, storage="f32"),
    1: Workload("csa_decode_bf16_B32_N65536_H64_k512", 1, B=32, N=65536, S=1, t=65535),
    2: Workload("csa_prefill_bf16_B1_S8192_H64_k512", 2, B=1, N=8192, S=8192, t=None),
    3: Workload("hca_decode_bf16_B16_N262144_m128_H64", 3, B=16, N=262144, S=1, t=262143,
                ratio=128, top_k=0),
    4: Workload("csa_decode_bf16_B4_N1048576+3_H64_k512", 4, B=4, N=1048579, S=1, t=1048578),
}


def small_workload(base: int, **kw) -> Workload:
    """A reduced copy of workload ``base`` (tests); keyword arguments override fields."""
    return replace(WORKLOADS[base], **kw)


# ---------------------------------------------------------------- storage rounding (no method math)
def round_bf16(x: np.ndarray) -> np.ndarray:
    """float32 -> float32 holding the nearest bf16 value (round to nearest, ties to even)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return u.astype(np.uint32).view(np.float32)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) of float32 values that are already bf16-representable."""
    return (np.ascontiguousarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def bits_to_f32(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float32 values."""
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


def _draw(rng: np.random.Generator, shape, sigma: float, storage: str) -> np.ndarray:
    a = rng.standard_normal(shape, dtype=np.float32)
    if sigma != 1.0:
        a *= np.float32(sigma)
    return a if storage == "f32" else round_bf16(a)      # "bf16", and "fp4" (bf16 raw rows)


def gen_shared(wl: Workload) -> dict:
    """Tensors shared by every request: bias [2m, d], idx_bias [2m, d_I], sink [H]. The gate
    biases and sink stay float32 (they are parameters, not cache contents)."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([wl.seed, wl.wid, 1 << 20])))
    m = wl.ratio
    out = {"bias": _draw(rng, (2 * m, wl.d), math.sqrt(0.1), "f32")}
    out["idx_bias"] = None if wl.hca else _draw(rng, (2 * m, wl.d_idx), math.sqrt(0.1), "f32")
    out["sink"] = _draw(rng, (wl.H,), 1.0, "f32")
    return out


def gen_request(wl: Workload, b: int) -> dict:
    """All per-request tensors of request b (float32, already rounded to the storage type)."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([wl.seed, wl.wid, b])))
    N = wl.N
    st = wl.storage
    r = {"kv": _draw(rng, (N, wl.d), 1.0 / math.sqrt(wl.d), st),
         "gate": _draw(rng, (N, wl.d), 1.0, st)}
    if wl.hca:
        r["idx_k"] = r["idx_gate"] = None
    else:
        r["idx_k"] = _draw(rng, (N, wl.d_idx), 1.0 / math.sqrt(wl.d_idx), st)
        r["idx_gate"] = _draw(rng, (N, wl.d_idx), 1.0, st)
    r["q"] = _draw(rng, (wl.S, wl.H, wl.d), wl.q_gain / math.sqrt(wl.d), st)
    if wl.hca:
        r["q_idx"] = r["w"] = None
    else:
        r["q_idx"] = _draw(rng, (wl.S, wl.H_idx, wl.d_idx), 1.0 / math.sqrt(wl.d_idx), st)
        r["w"] = _draw(rng, (wl.S, wl.H_idx), 1.0 / math.sqrt(wl.d_idx * wl.H_idx), "f32")
    return r


def gen_requests(wl: Workload, requests=None, threads: int | None = None, fn=None):
    """Draw several requests in parallel threads (NumPy releases the GIL while drawing).
    ``fn(b, req)`` may consume each request as it is drawn (e.g. upload and drop it) so the host
    never holds every request at once; without ``fn`` the list of requests is returned."""
    reqs = list(range(wl.B)) if requests is None else list(requests)
    threads = threads or max(1, min(len(reqs), os.cpu_count() or 1, 16))

    def one(b):
        r = gen_request(wl, b)
        return fn(b, r) if fn is not None else r

    with ThreadPoolExecutor(threads) as ex:
        return list(ex.map(one, reqs))
