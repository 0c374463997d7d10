"""Pins of the exchange oracle (entry-range shards): the merged selection equals the unsharded
selection, and the merged attention partials equal the unsharded attention, on random data with
planted ties, empty shards and shards past the visible entries (CPU)."""
import numpy as np
import pytest

from oracle import csa_oracle as O
from oracle import exchange as X


@pytest.mark.parametrize("G", [1, 2, 3, 5])
def test_shard_ranges_cover_disjointly(G):
    for n in (0, 1, 7, 1000, 16384):
        r = X.shard_ranges(n, G)
        assert len(r) == G and r[0][0] == 0 and sum(c for _, c in r) == n
        assert all(r[g][0] + r[g][1] == r[g + 1][0] for g in range(G - 1))


@pytest.mark.parametrize("G,k,V,n_cap", [(2, 64, 1000, 1200), (3, 512, 400, 900), (4, 16, 5000, 5000), (5, 8, 3, 40)])
def test_merged_candidates_equal_the_global_selection(G, k, V, n_cap):
    rng = np.random.default_rng(G * 1000 + k)
    s = rng.standard_normal(V)
    s[rng.integers(0, V, V // 4)] = 0.5                      # planted ties across shards
    cands = [X.local_candidates(s, b, n, k) for b, n in X.shard_ranges(n_cap, G)]
    want = O.topk_select(s, k)
    n_sel = int((want >= 0).sum())
    exp = np.concatenate([np.sort(want[:n_sel]), np.full(k - n_sel, -1)])
    np.testing.assert_array_equal(X.merge_candidates(cands, k), exp)


@pytest.mark.parametrize("G", [1, 2, 3])
def test_merged_partials_equal_the_attention(G):
    rng = np.random.default_rng(40 + G)
    cfg = O.OracleConfig(H=4, top_k=24, window=16, ratio=4)
    t = 399
    V = O.visible(t, cfg.ratio)
    kv = rng.standard_normal((t + 1, cfg.d)) / 22.6
    ckv = rng.standard_normal((V, cfg.d))
    q = rng.standard_normal((cfg.H, cfg.d)) / 22.6
    sink = rng.standard_normal(cfg.H)
    sel = np.sort(rng.choice(V, cfg.top_k, replace=False))
    ref = O.sparse_attn(q, kv, ckv, sel, sink, t, cfg)
    lo = max(0, t - cfg.window + 1)
    win = O.rope(kv[lo:t + 1], np.arange(lo, t + 1), cfg.d_rope, cfg.rope_base)
    parts = []
    for g, (b, n) in enumerate(X.shard_ranges(V, G)):
        mine = sel[(sel >= b) & (sel < b + n)]
        rows = ckv[mine]
        if g == 0:
            rows = np.concatenate([win, rows])
        parts.append(X.attn_partial(q, rows, t, cfg))
    parts.append(X.attn_partial(q, np.zeros((0, cfg.d)), t, cfg))   # a shard that contributes nothing
    np.testing.assert_allclose(X.merge_partials(parts, sink, t, cfg), ref, rtol=1e-12, atol=1e-14)
