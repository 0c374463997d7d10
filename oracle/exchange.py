"""fp64 oracle of the exchange over entry-range shards: one long request's compressed caches split by
entry range over G shards (devices), each scoring and attending over its own entries.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s cpu_baseline /
reference arm may import this module; the CUDA library never does, and this module imports nothing
from it.

Source: [FLASH] "DeepSeek-V4-Flash 架构：一个 token 的旅程", section "少读 KV 之前，Indexer 仍要给历史打分"
(with tensor parallelism the scores are combined before entries are selected), and section
"局部和压缩记忆，共用一次归一化" (one softmax over the window and the selected entries, the sink once in
the denominator). Reading where the page is silent: the shards split the entry range (not the
indexer heads); each shard keeps its local top k as (score, entry) candidates, which are gathered
and merged; the attention splits into per-shard partials (max logit, sum of exponentials,
unnormalised weighted sum), merged with the sink counted once.
"""
from __future__ import annotations

import numpy as np

from .csa_oracle import OracleConfig, rope, topk_select

__all__ = ["shard_ranges", "local_candidates", "merge_candidates", "attn_partial", "merge_partials"]


def shard_ranges(n_entries: int, G: int) -> list[tuple[int, int]]:
    """G contiguous entry ranges (first entry, count) covering [0, n_entries), as equal as possible."""
    edges = [n_entries * g // G for g in range(G + 1)]
    return [(edges[g], edges[g + 1] - edges[g]) for g in range(G)]


def local_candidates(scores, base: int, n: int, k: int):
    """A shard's candidates: the top k of the visible scores of entries [base, base + n) under
    (-score, index). ``scores`` holds the scores of the visible entries 0 .. V-1 (global indices).
    Returns (global indices, scores), at most k of each."""
    s = np.asarray(scores, dtype=np.float64)
    hi = min(base + n, s.shape[0])
    if hi <= base:
        return np.zeros(0, np.int64), np.zeros(0)
    sel = topk_select(s[base:hi], k)
    sel = sel[sel >= 0]
    return sel + base, s[base:hi][sel]


def merge_candidates(cands, k: int) -> np.ndarray:
    """The global selection from the shards' candidate lists [(global indices, scores), ...]: the top
    k of their union under (-score, index), in ascending index, -1 padded to k."""
    idx = np.concatenate([np.asarray(c[0], np.int64) for c in cands])
    sc = np.concatenate([np.asarray(c[1], np.float64) for c in cands])
    order = np.lexsort((idx, -sc))[:k]
    out = np.full(k, -1, dtype=np.int64)
    out[:len(order)] = np.sort(idx[order])
    return out


def attn_partial(q, rows, t: int, cfg: OracleConfig):
    """Partials of one shard for the query at t over its candidate rows (already rotated, [n, d]):
    m_h = max logit (-inf if n = 0), l_h = sum exp(logit - m_h), o_h = sum exp(logit - m_h) e_c."""
    E = np.asarray(rows, dtype=np.float64).reshape(-1, cfg.d)
    H = np.asarray(q).shape[0]
    if E.shape[0] == 0:
        return np.full(H, -np.inf), np.zeros(H), np.zeros((H, cfg.d))
    qr = rope(q, t, cfg.d_rope, cfg.rope_base)
    lg = cfg.scale * (qr @ E.T)
    m = lg.max(axis=1)
    p = np.exp(lg - m[:, None])
    return m, p.sum(axis=1), p @ E


def merge_partials(parts, sink, t: int, cfg: OracleConfig) -> np.ndarray:
    """The attention output from the shards' partials [(m, l, o), ...] with the sink counted once:
    M = max(sink, m_g); o = sum_g e^(m_g - M) o_g / (e^(sink - M) + sum_g e^(m_g - M) l_g), then
    rotated back by -t."""
    sink = np.asarray(sink, dtype=np.float64)
    M = sink.copy()
    for m, _, _ in parts:
        M = np.maximum(M, m)
    num = np.zeros_like(np.asarray(parts[0][2], dtype=np.float64))
    den = np.exp(sink - M)
    for m, l, o in parts:
        w = np.where(np.isfinite(m), np.exp(np.where(np.isfinite(m), m, 0.0) - M), 0.0)
        num += w[:, None] * o
        den += w * l
    return rope(num / den[:, None], t, cfg.d_rope, cfg.rope_base, inverse=True)
