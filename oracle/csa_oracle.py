"""Plain fp64 CPU oracle for the compressed-sparse-attention (CSA / HCA) path.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
cpu_baseline / reference arm may import this module. The product path (the CUDA library
and its Python binding) never imports, links or executes anything under ``oracle/``, and
this module imports nothing from the product path.

Every function computes in float64 with NumPy and follows the method as the source pages
state it. Sources (cited by page title and section):

* [FLASH] "DeepSeek-V4-Flash 架构：一个 token 的旅程" (hs-black.github.io/posts/deepseek-v4-flash),
  sections "低秩 Q：两次矩阵乘法接起来" (q RoPE on the last 64 dims), "局部和压缩记忆，共用一次归一化"
  (joint softmax over local + selected compressed entries, per-head sink in the denominator
  only), "输出投影也分组，并且降低中间维度" (inverse RoPE on the output), "压缩是逐通道的
  learned pooling" (per-channel softmax pooling over the token axis, then RMSNorm, then RoPE on
  the last 64 dims), "一个通道，逐项算出压缩结果" (missing previous group gets gate -inf / weight
  0), "压缩条目必须等整组完成后才可见" (visible = (t+1)//ratio; an entry is written when its group
  completes), "少读 KV 之前，Indexer 仍要给历史打分" (64 heads x 128 dims against one shared
  128-dim index cache; signed weights, not a softmax; sum over heads then select).
* [LAB41] "Lab tổng hợp DeepSeek-V4.1-Flash — chạy toàn trình 1A → 6B bằng NumPy"
  (openarchlab.com), sections "3 Giải pháp" and "6 Thuật ngữ / attn_sink" (the sink adds a
  score column to each softmax row and owns no value).
* [ATLAS] "LLM Atlas — DeepSeek" (llm-atlas.k1412.top/deepseek), section "19 V4 / HETEROGENEOUS
  STATE MACHINE": CSA compresses then keeps a top-k subset chosen by the indexer; HCA compresses
  harder and keeps every compressed entry.

Readings where the pages are silent (each is listed in the repository's design notes):
* overlap: entry i pools raw tokens j in [(i-1)m, (i+1)m) with the same kv / gate rows for both
  halves and a positional bias indexed by p = j - (i-1)m in [0, 2m); rows with j < 0 get -inf.
* RMSNorm has unit weight and eps = 1e-6, over all channels of the entry, before RoPE.
* RoPE rotates interleaved pairs (2i, 2i+1) of the last 64 dims by pos * base**(-2i/64).
  q and the index query are rotated at t, raw entry j at j, compressed entry i at i*m, and the
  output is rotated back by -t.
* raw window entries are the raw kv rows (not normalised) rotated at their own positions.
* indexer score s_i = sum_h w_h * relu(rope(q_h, t) . cidx_i): no extra scale (the weights carry
  it); one shared selection per query.
* attention logit = softmax_scale * q_h . e_c (default 1/sqrt(512)); sink logits are not scaled.
* window = raw tokens [max(0, t-W+1), t], concatenated with the selected compressed entries
  without de-duplication.
* top-k orders by (-score, index); if fewer than k entries are visible all are taken and the
  rest of the k slots hold -1.
"""

from __future__ import annotations

import math
from dataclasses import dataclass
from collections import deque

import numpy as np

__all__ = [
    "OracleConfig", "rope", "rms_norm", "pool_window", "compress", "visible",
    "index_scores", "topk_select", "attn_candidates", "sparse_attn", "decode_step",
    "prefill", "decode_stream",
]


@dataclass(frozen=True)
class OracleConfig:
    """Shape and hyper-parameters of one CSA / HCA layer (tensor contract of [FLASH],
    section "每个算子先对齐四个维度": B requests, S tokens this call, H heads, widths d)."""
    H: int = 64              # query heads
    d: int = 512             # shared KV head width (K = V)
    d_rope: int = 64         # rotary tail width
    H_idx: int = 64          # indexer heads
    d_idx: int = 128         # indexer width
    ratio: int = 4           # compression ratio m
    top_k: int = 512         # 0 selects HCA (every visible entry)
    window: int = 128        # raw sliding window W
    rope_base: float = 10000.0
    softmax_scale: float | None = None   # None -> 1/sqrt(d)
    rms_eps: float = 1e-6

    @property
    def hca(self) -> bool:
        return self.top_k == 0

    @property
    def scale(self) -> float:
        return (1.0 / math.sqrt(self.d)) if self.softmax_scale is None else float(self.softmax_scale)


def _f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


# --------------------------------------------------------------------------------------------
# RoPE and RMSNorm
# --------------------------------------------------------------------------------------------
def rope(x, pos, d_rope: int = 64, base: float = 10000.0, inverse: bool = False) -> np.ndarray:
    """Rotate the last ``d_rope`` dims of ``x`` (interleaved pairs) by angle pos * theta_i.

    [FLASH] "低秩 Q": ``q[..., -64:] = RoPE(q[..., -64:], position)``; "压缩是逐通道的 learned
    pooling": RoPE on the last 64 dims after pooling; "输出投影也分组": ``o = inverse_RoPE(o)``.
    theta_i = base ** (-2 i / d_rope), i < d_rope/2; ``pos`` broadcasts against x.shape[:-1].
    """
    x = _f64(x)
    out = x.copy()
    half = d_rope // 2
    theta = base ** (-2.0 * np.arange(half, dtype=np.float64) / d_rope)
    ang = _f64(pos)[..., None] * theta
    if inverse:
        ang = -ang
    c, s = np.cos(ang), np.sin(ang)
    a = x[..., x.shape[-1] - d_rope::2]
    b = x[..., x.shape[-1] - d_rope + 1::2]
    tail = out[..., x.shape[-1] - d_rope:]
    tail[..., 0::2] = a * c - b * s
    tail[..., 1::2] = a * s + b * c
    return out


def rms_norm(x, eps: float = 1e-6) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) over the last axis, unit weight ([FLASH] "压缩是逐通道的 learned
    pooling": pooling is followed by RMSNorm)."""
    x = _f64(x)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)


# --------------------------------------------------------------------------------------------
# Compressor
# --------------------------------------------------------------------------------------------
def pool_window(kv_win, gate_win, bias) -> np.ndarray:
    """Per-channel learned softmax pooling of one 2m-token window, before normalisation.

    [FLASH] "压缩是逐通道的 learned pooling": the softmax runs along the token axis separately for
    every channel. "一个通道，逐项算出压缩结果": a missing previous-group row has gate -inf and
    weight 0. ``kv_win``/``gate_win``/``bias`` are [2m, C]; missing rows carry gate = -inf.
    Returns the pooled [C] vector.
    """
    kv_win, logits = _f64(kv_win), _f64(gate_win) + _f64(bias)
    C = logits.shape[1]
    out = np.empty(C)
    for c in range(C):                       # one independent softmax per channel
        col = logits[:, c]
        live = np.isfinite(col)
        mx = col[live].max()
        wts = np.where(live, np.exp(np.where(live, col, 0.0) - mx), 0.0)
        out[c] = np.dot(wts, np.where(live, kv_win[:, c], 0.0)) / wts.sum()
    return out


def compress(kv, gate, bias, ratio: int, n_entries: int | None = None, *, rms_eps: float = 1e-6,
             d_rope: int = 64, rope_base: float = 10000.0, chunk: int = 1024) -> np.ndarray:
    """All compressed entries 0..n_entries-1 of one request (the whole-sequence prefill form).

    Entry i pools tokens [(i-1)m, (i+1)m) with per-channel softmax weights over
    gate[j] + bias[j - (i-1)m] (rows j < 0: -inf), then RMSNorm, then RoPE of the last
    ``d_rope`` dims at position i*m. [FLASH] sections "压缩是逐通道的 learned pooling",
    "一个通道，逐项算出压缩结果", "压缩条目必须等整组完成后才可见" (entry i needs tokens < (i+1)m).
    kv/gate: [N, C]; bias: [2m, C]. Returns [n_entries, C] float64.
    """
    kv, gate, bias = _f64(kv), _f64(gate), _f64(bias)
    m = ratio
    N, C = kv.shape
    if n_entries is None:
        n_entries = N // m
    if n_entries * m > N:
        raise ValueError("entry needs tokens beyond N")
    assert bias.shape == (2 * m, C)
    out = np.empty((n_entries, C))
    for e0 in range(0, n_entries, chunk):
        e1 = min(n_entries, e0 + chunk)
        n = e1 - e0
        lo = (e0 - 1) * m                                   # first token of entry e0's window
        rows = lo + np.arange((n + 1) * m)                  # tokens (e0-1)m .. e1*m-1
        valid = rows >= 0
        kv_rows = np.where(valid[:, None], kv[np.maximum(rows, 0)], 0.0)
        g_rows = np.where(valid[:, None], gate[np.maximum(rows, 0)], -np.inf)
        # window of entry e0+r = rows [r*m, r*m + 2m)
        idx = (np.arange(n)[:, None] * m + np.arange(2 * m)[None, :])   # [n, 2m]
        kv_w = kv_rows[idx]                                  # [n, 2m, C]
        lg = g_rows[idx] + bias[None]                        # [n, 2m, C]
        mx = lg.max(axis=1, keepdims=True)                   # own group is always finite
        p = np.exp(lg - mx)                                  # exp(-inf) = 0 for missing rows
        x = (p * kv_w).sum(axis=1) / p.sum(axis=1)
        x = rms_norm(x, rms_eps)
        out[e0:e1] = rope(x, (e0 + np.arange(n)) * m, d_rope, rope_base)
    return out


def compress_entry(kv_rows, gate_rows, bias, e: int, ratio: int, *, rms_eps: float = 1e-6,
                   d_rope: int = 64, rope_base: float = 10000.0) -> np.ndarray:
    """Entry e alone, from the raw rows of its own window: the same rule as ``compress`` for one
    entry (pooling of tokens [(e-1)m, (e+1)m), RMSNorm, RoPE at position e*m), for spot checks of
    long caches whose every entry would be too costly to recompute.

    kv_rows/gate_rows: [2m, C] = tokens (e-1)m .. (e+1)m-1, or [m, C] = tokens 0 .. m-1 for e = 0
    (the previous group does not exist: weight 0). Returns [C] float64.
    """
    m = ratio
    kv_rows, gate_rows = _f64(kv_rows), _f64(gate_rows)
    if e == 0:
        assert kv_rows.shape[0] == m
        kv_rows = np.concatenate([np.zeros_like(kv_rows), kv_rows])
        gate_rows = np.concatenate([np.full_like(gate_rows, -np.inf), gate_rows])
    assert kv_rows.shape[0] == 2 * m
    x = rms_norm(pool_window(kv_rows, gate_rows, bias), rms_eps)
    return rope(x, e * m, d_rope, rope_base)


def visible(t: int, ratio: int) -> int:
    """Number of compressed entries a query at position t may read: (t+1)//ratio
    ([FLASH] "压缩条目必须等整组完成后才可见")."""
    return (t + 1) // ratio


# --------------------------------------------------------------------------------------------
# Indexer and selection
# --------------------------------------------------------------------------------------------
def index_scores(q_idx, w, cidx, t: int, ratio: int, *, d_rope: int = 64,
                 rope_base: float = 10000.0) -> np.ndarray:
    """Indexer scores of every visible compressed entry for the query at position t.

    [FLASH] "少读 KV 之前，Indexer 仍要给历史打分": H_I heads of 128 dims score the shared
    128-dim compressed index cache; w is signed and is not a softmax; the heads are summed
    before selection. s_i = sum_h w_h * max(0, rope(q_h, t) . cidx_i), i < (t+1)//m.
    q_idx: [H_I, d_I] (unrotated); w: [H_I]; cidx: [>=V, d_I]. Returns [V] float64.
    """
    V = visible(t, ratio)
    qr = rope(q_idx, t, d_rope, rope_base)
    dots = _f64(cidx)[:V] @ qr.T                              # [V, H_I]
    return np.maximum(dots, 0.0) @ _f64(w)


def topk_select(scores, k: int) -> np.ndarray:
    """Indices of the k largest scores, ordered by (-score, index); -1 pads when fewer than k
    entries exist ([FLASH] "少读 KV 之前": top-k fixes how many entries main attention reads)."""
    s = _f64(scores)
    order = np.lexsort((np.arange(s.shape[0]), -s))
    out = np.full(k, -1, dtype=np.int64)
    n = min(k, s.shape[0])
    out[:n] = order[:n]
    return out


# --------------------------------------------------------------------------------------------
# Sparse joint attention with sink
# --------------------------------------------------------------------------------------------
def attn_candidates(kv, ckv, sel, t: int, cfg: OracleConfig):
    """Candidate entries of the query at t: the raw window [max(0,t-W+1), t], each raw row
    rotated at its own position, followed by the selected compressed entries (already rotated
    by the compressor). HCA keeps every visible compressed entry ([ATLAS] section 19).
    Returns (E [C, d], kinds list) where kinds marks raw (0) or compressed (1)."""
    lo = max(0, t - cfg.window + 1)
    win = rope(_f64(kv)[lo:t + 1], np.arange(lo, t + 1), cfg.d_rope, cfg.rope_base)
    V = visible(t, cfg.ratio)
    if cfg.hca:
        comp = np.arange(V)
    else:
        sel = np.asarray(sel)
        comp = sel[sel >= 0]
        if np.any(comp >= V):
            raise ValueError("selected entry is not visible")
    E = np.concatenate([win, _f64(ckv)[comp].reshape(len(comp), win.shape[1])], axis=0)
    return E, np.concatenate([np.zeros(len(win), np.int64), np.ones(len(comp), np.int64)])


def sparse_attn(q, kv, ckv, sel, sink, t: int, cfg: OracleConfig, return_weights: bool = False):
    """One query position t, all heads: single joint softmax over the raw window and the
    selected compressed entries plus a per-head sink logit that enlarges the denominator and owns
    no value; K = V = the candidate entry; the output is rotated back by -t.

    [FLASH] "局部和压缩记忆，共用一次归一化" and "输出投影也分组" (o = inverse_RoPE(o));
    [LAB41] "6 Thuật ngữ / attn_sink". q: [H, d] unrotated; sink: [H]. Returns o [H, d]
    (and, on request, the weights [H, C] and the sink share [H]).
    """
    E, _ = attn_candidates(kv, ckv, sel, t, cfg)
    qr = rope(q, t, cfg.d_rope, cfg.rope_base)                # [H, d]
    logits = cfg.scale * (qr @ E.T)                           # [H, C]
    sink = _f64(sink)
    mx = np.maximum(logits.max(axis=1) if E.shape[0] else -np.inf, sink)
    p = np.exp(logits - mx[:, None])
    z = np.exp(sink - mx) + p.sum(axis=1)
    o = (p @ E) / z[:, None]
    o = rope(o, t, cfg.d_rope, cfg.rope_base, inverse=True)
    if return_weights:
        return o, p / z[:, None], np.exp(sink - mx) / z
    return o


# --------------------------------------------------------------------------------------------
# Whole path: one decode step, whole-sequence prefill, and token-by-token streaming
# --------------------------------------------------------------------------------------------
def decode_step(t, q, q_idx, w, sink, kv, ckv, cidx, cfg: OracleConfig, return_sel: bool = False):
    """The path for one request and one query at t, given compressed caches holding at least
    (t+1)//m entries: indexer scores -> top-k -> sparse attention (HCA: no indexer)."""
    if cfg.hca:
        sel, sc = None, None
    else:
        sc = index_scores(q_idx, w, cidx, t, cfg.ratio, d_rope=cfg.d_rope, rope_base=cfg.rope_base)
        sel = topk_select(sc, cfg.top_k)
    o = sparse_attn(q, kv, ckv, sel, sink, t, cfg)
    return (o, sel, sc) if return_sel else o


def prefill(kv, gate, bias, idx_k, idx_gate, idx_bias, q, q_idx, w, sink, cfg: OracleConfig,
            S: int | None = None):
    """Causal prefill of S tokens for one request: every compressed entry is built at once, then
    each query t applies its own visibility mask (i < (t+1)//m) ([FLASH] "压缩条目必须等整组
    完成后才可见": prefill computes all entries in parallel, every query keeps its causal mask).
    Returns (o [S, H, d], ckv, cidx)."""
    N = kv.shape[0] if S is None else S
    n_ent = N // cfg.ratio
    ckv = compress(kv[:N], gate[:N], bias, cfg.ratio, n_ent, rms_eps=cfg.rms_eps,
                   d_rope=cfg.d_rope, rope_base=cfg.rope_base)
    cidx = None
    if not cfg.hca:
        cidx = compress(idx_k[:N], idx_gate[:N], idx_bias, cfg.ratio, n_ent, rms_eps=cfg.rms_eps,
                        d_rope=cfg.d_rope, rope_base=cfg.rope_base)
    o = np.stack([decode_step(t, q[t], None if cfg.hca else q_idx[t], None if cfg.hca else w[t],
                              sink, kv, ckv, cidx, cfg) for t in range(N)])
    return o, ckv, cidx


class _StreamingPool:
    """Token-by-token compressor state: a ring of the last 2m raw rows. When token t closes a
    group ((t+1) % m == 0) the entry t//m is pooled from the ring ([FLASH] "压缩条目必须等整组完成
    后才可见": ``if (t+1) % ratio == 0: cache[t // ratio] = pool(completed_group)``)."""

    def __init__(self, C: int, m: int, bias, cfg: OracleConfig):
        self.m, self.bias, self.cfg = m, _f64(bias), cfg
        self.kv = deque([np.zeros(C)] * (2 * m), maxlen=2 * m)
        self.g = deque([np.full(C, -np.inf)] * (2 * m), maxlen=2 * m)
        self.entries: list[np.ndarray] = []

    def push(self, t: int, kv_row, g_row) -> None:
        self.kv.append(_f64(kv_row))
        self.g.append(_f64(g_row))
        if (t + 1) % self.m == 0:
            i = t // self.m
            x = pool_window(np.stack(self.kv), np.stack(self.g), self.bias)
            x = rms_norm(x, self.cfg.rms_eps)
            self.entries.append(rope(x, i * self.m, self.cfg.d_rope, self.cfg.rope_base))


def decode_stream(kv, gate, bias, idx_k, idx_gate, idx_bias, q, q_idx, w, sink, cfg: OracleConfig,
                  T: int | None = None):
    """Token-by-token decode of T tokens for one request, caches growing as groups close; the
    number of readable entries is simply the length of the cache. Must equal ``prefill``
    ([FLASH] "把推导变成可以检查的程序": prefill == streaming). Returns o [T, H, d]."""
    T = kv.shape[0] if T is None else T
    kvp = _StreamingPool(kv.shape[1], cfg.ratio, bias, cfg)
    ixp = None if cfg.hca else _StreamingPool(idx_k.shape[1], cfg.ratio, idx_bias, cfg)
    outs = []
    for t in range(T):
        kvp.push(t, kv[t], gate[t])
        if ixp is not None:
            ixp.push(t, idx_k[t], idx_gate[t])
        n = len(kvp.entries)
        ckv = np.stack(kvp.entries) if n else np.zeros((0, kv.shape[1]))
        lo = max(0, t - cfg.window + 1)
        win = rope(_f64(kv)[lo:t + 1], np.arange(lo, t + 1), cfg.d_rope, cfg.rope_base)
        if cfg.hca:
            comp = ckv
        else:
            cidx = np.stack(ixp.entries) if n else np.zeros((0, idx_k.shape[1]))
            qr = rope(q_idx[t], t, cfg.d_rope, cfg.rope_base)
            sc = np.maximum(cidx @ qr.T, 0.0) @ _f64(w[t])
            order = sorted(range(n), key=lambda i: (-sc[i], i))[:cfg.top_k]
            comp = ckv[order] if order else np.zeros((0, kv.shape[1]))
        E = np.concatenate([win, comp])
        qr = rope(q[t], t, cfg.d_rope, cfg.rope_base)
        lg = cfg.scale * (qr @ E.T)
        mx = np.maximum(lg.max(axis=1), sink)
        p = np.exp(lg - mx[:, None])
        o = (p @ E) / (np.exp(_f64(sink) - mx) + p.sum(axis=1))[:, None]
        outs.append(rope(o, t, cfg.d_rope, cfg.rope_base, inverse=True))
    return np.stack(outs)
