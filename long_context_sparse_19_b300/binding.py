"""Thin ctypes binding of ``libcsa.so`` (the C ABI declared in ``include/csa.h``).

Each function has the C name, takes torch tensors that already live on the GPU, checks that their
shapes / dtypes / contiguity match the call, and passes raw device pointers plus the current CUDA
stream. Every step of the computation runs in the library's CUDA kernels; if the library cannot be
loaded, importing this module raises instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char_p, c_float, c_int, c_int32, c_int64, c_size_t, c_uint32, c_void_p
from dataclasses import dataclass

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libcsa.so")

CSA_F32, CSA_BF16, CSA_FP4 = 0, 1, 2
_STORAGE = {"f32": CSA_F32, "bf16": CSA_BF16, "fp4": CSA_FP4}
CSA_FLAG_SIMT = 1
CSA_FLAG_TEST_STALL = 1 << 30          # timeout test hook (include/csa.h)
CSA_ERR_DEVICE, CSA_ERR_DEVICE_TIMEOUT = 6, 8

# the public entry points declared in include/csa.h
EXPORTS = ("csa_status_string", "csa_last_error", "csa_get_device_status", "csa_sync_status", "csa_workspace_bytes",
           "csa_cache_bytes",
           "csa_compress", "csa_index_topk", "csa_index_topk_static", "csa_sparse_attn", "csa_decode",
           "csa_prefill",
           "csa_index_topk_shard", "csa_topk_merge", "csa_sparse_attn_shard", "csa_attn_merge",
           "csa_launch_count", "csa_profile_begin", "csa_profile_end")
STAGES = ("compress", "index", "topk", "attn", "merge")


class CsaConfig(ctypes.Structure):
    _fields_ = [("H", c_int32), ("d", c_int32), ("d_rope", c_int32), ("H_idx", c_int32),
                ("d_idx", c_int32), ("ratio", c_int32), ("top_k", c_int32), ("window", c_int32),
                ("rope_base", c_float), ("softmax_scale", c_float), ("rms_eps", c_float),
                ("storage", c_int32), ("flags", c_uint32)]


class CsaCache(ctypes.Structure):
    _fields_ = [("kv", c_void_p), ("gate", c_void_p), ("gate_bias", c_void_p), ("idx_k", c_void_p),
                ("idx_gate", c_void_p), ("idx_bias", c_void_p), ("N", c_int64), ("ckv", c_void_p),
                ("cidx", c_void_p), ("n_cap", c_int64)]


class CsaError(RuntimeError):
    def __init__(self, status: int, where: str, msg: str):
        super().__init__(f"{where}: status {status} ({msg})")
        self.status = status


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libcsa.so once and declares the prototypes of every exported call."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with `python long_context_sparse_19_b300/build.py`")
    L = ctypes.CDLL(path)
    cp, vp = POINTER(CsaConfig), c_void_p
    L.csa_status_string.argtypes, L.csa_status_string.restype = [c_int], c_char_p
    L.csa_last_error.argtypes, L.csa_last_error.restype = [], c_char_p
    L.csa_get_device_status.argtypes, L.csa_get_device_status.restype = [vp, c_int, POINTER(c_int32)], c_int
    L.csa_sync_status.argtypes, L.csa_sync_status.restype = [vp], c_int
    L.csa_workspace_bytes.argtypes, L.csa_workspace_bytes.restype = [cp, c_int32, c_int32, c_int64], c_size_t
    L.csa_cache_bytes.argtypes, L.csa_cache_bytes.restype = [cp, c_int32, c_int64], c_size_t
    L.csa_compress.argtypes, L.csa_compress.restype = [cp, c_int32, POINTER(CsaCache), c_int64, c_int64, vp], c_int
    L.csa_index_topk.argtypes = [cp, c_int32, c_int32, vp, vp, vp, vp, c_int64, vp, vp, vp, c_size_t, vp]
    L.csa_index_topk.restype = c_int
    L.csa_index_topk_static.argtypes = [cp, c_int32, c_int32, vp, vp, vp, vp, c_int64, vp, vp, vp]
    L.csa_index_topk_static.restype = c_int
    L.csa_sparse_attn.argtypes = [cp, c_int32, c_int32, vp, vp, vp, c_int64, vp, c_int64, vp, vp, vp, vp,
                                  c_size_t, vp]
    L.csa_sparse_attn.restype = c_int
    L.csa_decode.argtypes = [cp, c_int32, vp, POINTER(CsaCache), vp, vp, vp, vp, vp, vp, vp, c_size_t, vp]
    L.csa_decode.restype = c_int
    L.csa_prefill.argtypes = [cp, c_int32, c_int32, POINTER(CsaCache), vp, vp, vp, vp, vp, vp, vp, c_size_t, vp]
    L.csa_prefill.restype = c_int
    L.csa_index_topk_shard.argtypes = [cp, c_int32, vp, vp, vp, vp, c_int64, c_int64, vp, vp, vp, c_size_t, vp]
    L.csa_index_topk_shard.restype = c_int
    L.csa_topk_merge.argtypes = [cp, c_int32, c_int32, vp, vp, POINTER(c_int64), POINTER(c_int64), vp, vp, vp]
    L.csa_topk_merge.restype = c_int
    L.csa_sparse_attn_shard.argtypes = [cp, c_int32, vp, vp, vp, c_int64, vp, c_int64, c_int64, vp, c_int32, vp, vp,
                                        vp]
    L.csa_sparse_attn_shard.restype = c_int
    L.csa_attn_merge.argtypes = [cp, c_int32, c_int32, vp, vp, vp, vp, vp, vp]
    L.csa_attn_merge.restype = c_int
    L.csa_launch_count.argtypes, L.csa_launch_count.restype = [], c_int64
    L.csa_profile_begin.argtypes, L.csa_profile_begin.restype = [c_int32], c_int
    L.csa_profile_end.argtypes, L.csa_profile_end.restype = [POINTER(c_float), POINTER(c_int32), c_int32], c_int
    _lib = L
    return L


def _check(status: int, where: str) -> None:
    if status != 0:
        L = load()
        raise CsaError(status, where, (L.csa_last_error() or b"").decode() or
                       L.csa_status_string(status).decode())


# ------------------------------------------------------------------------------------ config
@dataclass
class Config:
    """Python mirror of csa_config (see include/csa.h)."""
    H: int = 64
    d: int = 512
    d_rope: int = 64
    H_idx: int = 64
    d_idx: int = 128
    ratio: int = 4
    top_k: int = 512
    window: int = 128
    rope_base: float = 10000.0
    softmax_scale: float = 0.0
    rms_eps: float = 1e-6
    storage: str = "bf16"              # "bf16", "f32", or "fp4" (FP4 E2M1 + FP8 E4M3 caches, bf16 rows)
    simt: bool = False
    test_stall: bool = False           # the timeout test hook; never set in production

    @property
    def dtype(self) -> torch.dtype:
        """dtype of raw rows, queries and outputs (and of the caches, except with "fp4")."""
        return torch.float32 if self.storage == "f32" else torch.bfloat16

    @property
    def lowp(self) -> bool:
        return self.storage == "fp4"

    def c(self) -> CsaConfig:
        return CsaConfig(self.H, self.d, self.d_rope, self.H_idx, self.d_idx, self.ratio, self.top_k,
                         self.window, self.rope_base, self.softmax_scale, self.rms_eps,
                         _STORAGE[self.storage],
                         (CSA_FLAG_SIMT if self.simt else 0) | (CSA_FLAG_TEST_STALL if self.test_stall else 0))


def _ptr(t, shape=None, dtype=None, name="tensor"):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return t.data_ptr()


def csa_cache_bytes(cfg: Config, which: int, n_cap: int) -> int:
    """Bytes of one request's compressed cache (which = 0: ckv, 1: cidx)."""
    return int(load().csa_cache_bytes(ctypes.byref(cfg.c()), which, n_cap))


def cache_tensor(cfg: Config, B: int, n_cap: int, which: int, device="cuda") -> torch.Tensor:
    """An uninitialised compressed cache: [B, n_cap, C] of cfg.dtype, or with "fp4" storage
    [B, csa_cache_bytes] bytes."""
    if cfg.lowp:
        return torch.empty((B, csa_cache_bytes(cfg, which, n_cap)), dtype=torch.uint8, device=device)
    return torch.empty((B, n_cap, cfg.d_idx if which else cfg.d), dtype=cfg.dtype, device=device)


def _n_cap(cfg: Config, t, n_cap):
    if n_cap is not None:
        return int(n_cap)
    if cfg.lowp:
        raise ValueError("n_cap must be given with fp4 caches")
    return t.shape[1]


def _cache_ptr(cfg: Config, t, which: int, B: int, n_cap: int, name: str):
    if cfg.lowp:
        return _ptr(t, (B, csa_cache_bytes(cfg, which, n_cap)), torch.uint8, name)
    return _ptr(t, (B, n_cap, cfg.d_idx if which else cfg.d), cfg.dtype, name)


def _stream(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


@dataclass
class Cache:
    """Device tensors of the raw per-token inputs and compressed caches of B requests."""
    kv: torch.Tensor                # [B, N, d]
    gate: torch.Tensor              # [B, N, d]
    gate_bias: torch.Tensor         # [2m, d] float32
    ckv: torch.Tensor               # [B, n_cap, d]
    idx_k: torch.Tensor | None = None      # [B, N, d_idx]
    idx_gate: torch.Tensor | None = None
    idx_bias: torch.Tensor | None = None   # [2m, d_idx] float32
    cidx: torch.Tensor | None = None       # [B, n_cap, d_idx]
    n_cap: int | None = None               # required with fp4 caches ([B, csa_cache_bytes] bytes)

    def capacity(self, cfg: Config) -> int:
        return _n_cap(cfg, self.ckv, self.n_cap)

    def c(self, cfg: Config) -> CsaCache:
        B, N, _ = self.kv.shape
        n_cap = self.capacity(cfg)
        dt = cfg.dtype
        m = cfg.ratio
        k = CsaCache()
        k.kv = _ptr(self.kv, (B, N, cfg.d), dt, "kv")
        k.gate = _ptr(self.gate, (B, N, cfg.d), dt, "gate")
        k.gate_bias = _ptr(self.gate_bias, (2 * m, cfg.d), torch.float32, "gate_bias")
        k.ckv = _cache_ptr(cfg, self.ckv, 0, B, n_cap, "ckv")
        if self.idx_k is not None:
            k.idx_k = _ptr(self.idx_k, (B, N, cfg.d_idx), dt, "idx_k")
            k.idx_gate = _ptr(self.idx_gate, (B, N, cfg.d_idx), dt, "idx_gate")
            k.idx_bias = _ptr(self.idx_bias, (2 * m, cfg.d_idx), torch.float32, "idx_bias")
            k.cidx = _cache_ptr(cfg, self.cidx, 1, B, n_cap, "cidx")
        k.N, k.n_cap = N, n_cap
        return k


# ------------------------------------------------------------------------------------ entry points
def csa_status_string(status: int) -> str:
    return load().csa_status_string(status).decode()


def csa_get_device_status(reset: bool = True, stream=None) -> int:
    """Synchronises the stream and returns the device error word (0 = no error)."""
    code = c_int32(0)
    load().csa_get_device_status(_stream(stream), int(reset), ctypes.byref(code))
    return code.value


def csa_sync_status(stream=None) -> int:
    """Synchronises the stream and returns the device status (0 = CSA_OK, CSA_ERR_DEVICE_TIMEOUT,
    CSA_ERR_DEVICE); the device error word is left as it is."""
    return int(load().csa_sync_status(_stream(stream)))


def csa_workspace_bytes(cfg: Config, B: int, S: int, n_cap: int) -> int:
    return int(load().csa_workspace_bytes(ctypes.byref(cfg.c()), B, S, n_cap))


def workspace(cfg: Config, B: int, S: int, n_cap: int, device="cuda") -> torch.Tensor:
    return torch.empty(max(16, csa_workspace_bytes(cfg, B, S, n_cap)), dtype=torch.uint8, device=device)


def csa_compress(cfg: Config, cache: Cache, first_entry: int, n_entries: int, stream=None) -> None:
    B = cache.kv.shape[0]
    _check(load().csa_compress(ctypes.byref(cfg.c()), B, ctypes.byref(cache.c(cfg)), first_entry, n_entries,
                               _stream(stream)), "csa_compress")


def csa_index_topk(cfg: Config, pos, q_idx, w, cidx, topk, scores=None, ws=None, stream=None, n_cap=None) -> None:
    B, S = pos.shape
    n_cap = _n_cap(cfg, cidx, n_cap)
    ws = workspace(cfg, B, S, n_cap) if ws is None else ws
    _check(load().csa_index_topk(
        ctypes.byref(cfg.c()), B, S, _ptr(pos, (B, S), torch.int64, "pos"),
        _ptr(q_idx, (B, S, cfg.H_idx, cfg.d_idx), cfg.dtype, "q_idx"), _ptr(w, (B, S, cfg.H_idx), torch.float32, "w"),
        _cache_ptr(cfg, cidx, 1, B, n_cap, "cidx"), n_cap,
        _ptr(topk, (B, S, cfg.top_k), torch.int32, "topk"), _ptr(scores, (B, S, n_cap), torch.float32, "scores"),
        _ptr(ws, None, torch.uint8, "ws"), ws.numel(), _stream(stream)), "csa_index_topk")


def csa_index_topk_static(cfg: Config, pos, q_idx, w, cidx, topk, scores=None, stream=None, n_cap=None) -> None:
    """csa_index_topk without a workspace: the library's fixed device scratch array is used instead
    (nothing is allocated; see include/csa.h for the size limit and the sharing rules)."""
    B, S = pos.shape
    n_cap = _n_cap(cfg, cidx, n_cap)
    _check(load().csa_index_topk_static(
        ctypes.byref(cfg.c()), B, S, _ptr(pos, (B, S), torch.int64, "pos"),
        _ptr(q_idx, (B, S, cfg.H_idx, cfg.d_idx), cfg.dtype, "q_idx"), _ptr(w, (B, S, cfg.H_idx), torch.float32, "w"),
        _cache_ptr(cfg, cidx, 1, B, n_cap, "cidx"), n_cap,
        _ptr(topk, (B, S, cfg.top_k), torch.int32, "topk"), _ptr(scores, (B, S, n_cap), torch.float32, "scores"),
        _stream(stream)), "csa_index_topk_static")


def csa_sparse_attn(cfg: Config, pos, q, kv, ckv, topk, sink, out, ws=None, stream=None, n_cap=None) -> None:
    B, S = pos.shape
    N, n_cap = kv.shape[1], _n_cap(cfg, ckv, n_cap)
    ws = workspace(cfg, B, S, n_cap) if ws is None else ws
    _check(load().csa_sparse_attn(
        ctypes.byref(cfg.c()), B, S, _ptr(pos, (B, S), torch.int64, "pos"),
        _ptr(q, (B, S, cfg.H, cfg.d), cfg.dtype, "q"), _ptr(kv, (B, N, cfg.d), cfg.dtype, "kv"), N,
        _cache_ptr(cfg, ckv, 0, B, n_cap, "ckv"), n_cap,
        _ptr(topk, (B, S, cfg.top_k), torch.int32, "topk") if cfg.top_k else None,
        _ptr(sink, (cfg.H,), torch.float32, "sink"), _ptr(out, (B, S, cfg.H, cfg.d), cfg.dtype, "out"),
        _ptr(ws, None, torch.uint8, "ws"), ws.numel(), _stream(stream)), "csa_sparse_attn")


def csa_decode(cfg: Config, pos, cache: Cache, q, q_idx, w, sink, out, topk_out=None, ws=None,
               stream=None) -> None:
    B = pos.shape[0]
    n_cap = cache.capacity(cfg)
    ws = workspace(cfg, B, 1, n_cap) if ws is None else ws
    hca = cfg.top_k == 0
    _check(load().csa_decode(
        ctypes.byref(cfg.c()), B, _ptr(pos, (B,), torch.int64, "pos"), ctypes.byref(cache.c(cfg)),
        _ptr(q, (B, cfg.H, cfg.d), cfg.dtype, "q"),
        None if hca else _ptr(q_idx, (B, cfg.H_idx, cfg.d_idx), cfg.dtype, "q_idx"),
        None if hca else _ptr(w, (B, cfg.H_idx), torch.float32, "w"),
        _ptr(sink, (cfg.H,), torch.float32, "sink"), _ptr(out, (B, cfg.H, cfg.d), cfg.dtype, "out"),
        _ptr(topk_out, (B, cfg.top_k), torch.int32, "topk_out"),
        _ptr(ws, None, torch.uint8, "ws"), ws.numel(), _stream(stream)), "csa_decode")


def csa_prefill(cfg: Config, cache: Cache, q, q_idx, w, sink, out, topk_out=None, ws=None,
                stream=None) -> None:
    B, S = q.shape[0], q.shape[1]
    n_cap = cache.capacity(cfg)
    ws = workspace(cfg, B, S, n_cap) if ws is None else ws
    hca = cfg.top_k == 0
    _check(load().csa_prefill(
        ctypes.byref(cfg.c()), B, S, ctypes.byref(cache.c(cfg)),
        _ptr(q, (B, S, cfg.H, cfg.d), cfg.dtype, "q"),
        None if hca else _ptr(q_idx, (B, S, cfg.H_idx, cfg.d_idx), cfg.dtype, "q_idx"),
        None if hca else _ptr(w, (B, S, cfg.H_idx), torch.float32, "w"),
        _ptr(sink, (cfg.H,), torch.float32, "sink"), _ptr(out, (B, S, cfg.H, cfg.d), cfg.dtype, "out"),
        _ptr(topk_out, (B, S, cfg.top_k), torch.int32, "topk_out"),
        _ptr(ws, None, torch.uint8, "ws"), ws.numel(), _stream(stream)), "csa_prefill")


# ------------------------------------------------------------------------------------ entry-range shards
def csa_index_topk_shard(cfg: Config, pos, q_idx, w, cidx_shard, entry_base: int, cand_idx, cand_score, ws=None,
                         stream=None) -> None:
    """A shard's candidates (local indices and their scores) for one query per request."""
    B = pos.shape[0]
    n = cidx_shard.shape[1]
    ws = workspace(cfg, B, 1, n) if ws is None else ws
    _check(load().csa_index_topk_shard(
        ctypes.byref(cfg.c()), B, _ptr(pos, (B,), torch.int64, "pos"),
        _ptr(q_idx, (B, cfg.H_idx, cfg.d_idx), cfg.dtype, "q_idx"), _ptr(w, (B, cfg.H_idx), torch.float32, "w"),
        _ptr(cidx_shard, (B, n, cfg.d_idx), cfg.dtype, "cidx_shard"), n, entry_base,
        _ptr(cand_idx, (B, cfg.top_k), torch.int32, "cand_idx"), _ptr(cand_score, (B, cfg.top_k), torch.float32,
                                                                       "cand_score"),
        _ptr(ws, None, torch.uint8, "ws"), ws.numel(), _stream(stream)), "csa_index_topk_shard")


def csa_topk_merge(cfg: Config, cand_score, cand_idx, entry_base, n_shard, topk, shard_sel=None, stream=None) -> None:
    """The global selection from the G shards' candidates [B, G, k] (entry_base, n_shard: G ints)."""
    B, G, k = cand_idx.shape
    eb = (c_int64 * G)(*[int(x) for x in entry_base])
    ns = (c_int64 * G)(*[int(x) for x in n_shard])
    _check(load().csa_topk_merge(
        ctypes.byref(cfg.c()), B, G, _ptr(cand_score, (B, G, k), torch.float32, "cand_score"),
        _ptr(cand_idx, (B, G, k), torch.int32, "cand_idx"), eb, ns, _ptr(topk, (B, k), torch.int32, "topk"),
        _ptr(shard_sel, (B, G, k), torch.int32, "shard_sel"), _stream(stream)), "csa_topk_merge")


def csa_sparse_attn_shard(cfg: Config, pos, q, kv, ckv_shard, entry_base: int, sel, with_window: bool, part_o, part_ml,
                          stream=None) -> None:
    """A shard's attention partials (unnormalised o, and (max logit, sum)) for one query per request."""
    B = pos.shape[0]
    N, n = kv.shape[1], ckv_shard.shape[1]
    _check(load().csa_sparse_attn_shard(
        ctypes.byref(cfg.c()), B, _ptr(pos, (B,), torch.int64, "pos"), _ptr(q, (B, cfg.H, cfg.d), cfg.dtype, "q"),
        _ptr(kv, (B, N, cfg.d), cfg.dtype, "kv"), N, _ptr(ckv_shard, (B, n, cfg.d), cfg.dtype, "ckv_shard"), n,
        entry_base, _ptr(sel, (B, cfg.top_k), torch.int32, "sel") if cfg.top_k else None, int(with_window),
        _ptr(part_o, (B, cfg.H, cfg.d), torch.float32, "part_o"), _ptr(part_ml, (B, cfg.H, 2), torch.float32, "part_ml"),
        _stream(stream)), "csa_sparse_attn_shard")


def csa_attn_merge(cfg: Config, pos, part_o, part_ml, sink, out, stream=None) -> None:
    """out [B, H, d] from G shards' partials [B, G, H, d] and [B, G, H, 2]."""
    B, G = part_o.shape[0], part_o.shape[1]
    _check(load().csa_attn_merge(
        ctypes.byref(cfg.c()), B, G, _ptr(pos, (B,), torch.int64, "pos"),
        _ptr(part_o, (B, G, cfg.H, cfg.d), torch.float32, "part_o"),
        _ptr(part_ml, (B, G, cfg.H, 2), torch.float32, "part_ml"), _ptr(sink, (cfg.H,), torch.float32, "sink"),
        _ptr(out, (B, cfg.H, cfg.d), cfg.dtype, "out"), _stream(stream)), "csa_attn_merge")


def csa_launch_count() -> int:
    return int(load().csa_launch_count())


def csa_profile_begin(max_launches: int) -> None:
    _check(load().csa_profile_begin(max_launches), "csa_profile_begin")


def csa_profile_end() -> dict:
    """{stage: (total device ms, launches)} of the launches recorded since csa_profile_begin."""
    n = len(STAGES)
    ms = (c_float * n)()
    cnt = (c_int32 * n)()
    _check(load().csa_profile_end(ms, cnt, n), "csa_profile_end")
    return {STAGES[i]: (float(ms[i]), int(cnt[i])) for i in range(n)}


def bind_decode(cfg: Config, pos, cache: Cache, q, q_idx, w, sink, out, topk_out=None, ws=None):
    """csa_decode with every argument marshalled once; the returned callable enqueues one decode
    step on the current stream (so it can be replayed or captured into a CUDA graph cheaply)."""
    B = pos.shape[0]
    n_cap = cache.capacity(cfg)
    ws = workspace(cfg, B, 1, n_cap) if ws is None else ws
    hca = cfg.top_k == 0
    c = cfg.c()
    k = cache.c(cfg)
    args = (ctypes.byref(c), B, _ptr(pos, (B,), torch.int64, "pos"), ctypes.byref(k),
            _ptr(q, (B, cfg.H, cfg.d), cfg.dtype, "q"),
            None if hca else _ptr(q_idx, (B, cfg.H_idx, cfg.d_idx), cfg.dtype, "q_idx"),
            None if hca else _ptr(w, (B, cfg.H_idx), torch.float32, "w"),
            _ptr(sink, (cfg.H,), torch.float32, "sink"), _ptr(out, (B, cfg.H, cfg.d), cfg.dtype, "out"),
            _ptr(topk_out, (B, cfg.top_k), torch.int32, "topk_out"),
            _ptr(ws, None, torch.uint8, "ws"), ws.numel())
    fn = load().csa_decode
    # the call holds raw device pointers: keep every tensor they point into alive with it
    keep = (c, k, ws, pos, cache, q, q_idx, w, sink, out, topk_out)

    def call(stream=None):
        _ = keep
        _check(fn(*args, _stream(stream)), "csa_decode")
    return call
