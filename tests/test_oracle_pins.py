"""Pins of the fp64 oracle against facts fixed outside the oracle itself: hand-worked values,
closed forms, library routines, brute force on tiny inputs, and the invariants the source pages
state (prefill == streaming, causality, the group-boundary visibility fault)."""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import csa_oracle as O
from oracle.extras import mhc_residual_update, routing_weights

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(rng, *shape, s=1.0):
    return rng.standard_normal(shape) * s


# ------------------------------------------------------------------------------------ RoPE / norm
def test_rope_identity_at_zero_and_hand_value_at_one():
    rng = np.random.default_rng(1)
    x = _rand(rng, 3, 16)
    np.testing.assert_array_equal(O.rope(x, 0, d_rope=8), x)
    y = O.rope(x, 1, d_rope=8, base=10000.0)
    # untouched head dims
    np.testing.assert_array_equal(y[:, :8], x[:, :8])
    # pair 0 (dims 8, 9) turns by exactly 1 rad; pair 1 (dims 10, 11) by 10000**(-2/8) rad
    for j, ang in ((8, 1.0), (10, 10000.0 ** (-2.0 / 8))):
        a, b = x[:, j], x[:, j + 1]
        np.testing.assert_allclose(y[:, j], a * math.cos(ang) - b * math.sin(ang), rtol=0, atol=1e-15)
        np.testing.assert_allclose(y[:, j + 1], a * math.sin(ang) + b * math.cos(ang), rtol=0, atol=1e-15)


def test_rope_is_a_rotation_and_inverse_undoes_it():
    rng = np.random.default_rng(2)
    x = _rand(rng, 5, 512)
    pos = np.array([0, 3, 77, 65535, 1048578])
    y = O.rope(x, pos)
    np.testing.assert_allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-14)
    np.testing.assert_allclose(O.rope(y, pos, inverse=True), x, rtol=0, atol=1e-13)
    # composition: rope(p1) then rope(p2) == rope(p1 + p2)
    np.testing.assert_allclose(O.rope(O.rope(x, 5), 9), O.rope(x, 14), atol=1e-13)


def test_rms_norm_closed_form():
    rng = np.random.default_rng(3)
    x = _rand(rng, 4, 512, s=7.0)
    y = O.rms_norm(x, eps=0.0)
    np.testing.assert_allclose(np.mean(y * y, axis=1), 1.0, rtol=1e-14)
    c = np.full((1, 8), 0.5)
    np.testing.assert_allclose(O.rms_norm(c, eps=1e-6), 0.5 / math.sqrt(0.25 + 1e-6), rtol=1e-15)


# ------------------------------------------------------------------------------------ compressor
def _golden_pool():
    g = json.load(open(os.path.join(GOLDEN, "pool_hand.json")))
    kv = np.array(g["kv"], float)
    gate = np.log(np.stack([g["gate_c0_exp"], g["gate_c1_exp"]], axis=1).astype(float))
    bias = np.log(np.array(g["bias_exp"], float))
    exp = {k: [float(Fraction(v["c0"])), float(Fraction(v["c1"]))] for k, v in g["expected"].items()}
    return g["ratio"], kv, gate, bias, exp


def test_pool_window_hand_example():
    m, kv, gate, bias, exp = _golden_pool()
    # entry 0: previous group missing (gate -inf), own group = tokens 0, 1
    kv_w0 = np.concatenate([np.zeros((2, 2)), kv[0:2]])
    g_w0 = np.concatenate([np.full((2, 2), -np.inf), gate[0:2]])
    np.testing.assert_allclose(O.pool_window(kv_w0, g_w0, bias), exp["entry0"], rtol=1e-14)
    np.testing.assert_allclose(O.pool_window(kv[0:4], gate[0:4], bias), exp["entry1"], rtol=1e-14)


def test_compress_hand_example_through_norm_and_rope():
    m, kv, gate, bias, exp = _golden_pool()
    got = O.compress(kv, gate, bias, m, 2, rms_eps=1e-6, d_rope=2, rope_base=10000.0)
    for i, key in enumerate(("entry0", "entry1")):
        x = np.array(exp[key])
        x = x / math.sqrt(np.mean(x * x) + 1e-6)
        ang = i * m * 1.0                      # pair 0 has theta = 1; entry i sits at i*m
        want = np.array([x[0] * math.cos(ang) - x[1] * math.sin(ang),
                         x[0] * math.sin(ang) + x[1] * math.cos(ang)])
        np.testing.assert_allclose(got[i], want, rtol=1e-13)


def test_pooling_equal_gates_is_plain_mean():
    """Equal gates and zero bias: entry 0 averages its own m tokens, later entries all 2m."""
    rng = np.random.default_rng(4)
    m, C, n = 4, 16, 6
    kv = _rand(rng, n * m, C)
    gate = np.full((n * m, C), 0.3)
    got = O.compress(kv, gate, np.zeros((2 * m, C)), m, n, rms_eps=1e-6, d_rope=8)
    for i in range(n):
        lo = max(0, (i - 1) * m)
        want = O.rope(O.rms_norm(kv[lo:(i + 1) * m].mean(axis=0)), i * m, 8)
        np.testing.assert_allclose(got[i], want, rtol=1e-12, atol=1e-14)


def test_pooling_dominant_gate_picks_token():
    rng = np.random.default_rng(5)
    m, C = 4, 8
    kv = _rand(rng, 3 * m, C)
    gate = _rand(rng, 3 * m, C)
    gate[6, :] = 1e3                 # token 6 lies in entry 1 (tokens 0..7) and entry 2 (4..11)
    x = O.pool_window(kv[0:8], gate[0:8], np.zeros((8, C)))
    np.testing.assert_allclose(x, kv[6], rtol=1e-12)
    x = O.pool_window(kv[4:12], gate[4:12], np.zeros((8, C)))
    np.testing.assert_allclose(x, kv[6], rtol=1e-12)


def test_compress_matches_per_entry_window_loop():
    rng = np.random.default_rng(6)
    m, C, N = 4, 32, 40
    kv, gate, bias = _rand(rng, N, C), _rand(rng, N, C), _rand(rng, 2 * m, C, s=0.3)
    got = O.compress(kv, gate, bias, m, chunk=3, d_rope=8)
    for i in range(N // m):
        rows = np.arange((i - 1) * m, (i + 1) * m)
        kvw = np.where((rows >= 0)[:, None], kv[np.maximum(rows, 0)], 0.0)
        gw = np.where((rows >= 0)[:, None], gate[np.maximum(rows, 0)], -np.inf)
        want = O.rope(O.rms_norm(O.pool_window(kvw, gw, bias)), i * m, 8)
        np.testing.assert_allclose(got[i], want, rtol=1e-12, atol=1e-14)


def test_compress_entry_equals_the_whole_sequence_form():
    """The single-entry form (used for spot checks of long caches) against compress(): entry 0
    (no previous group), interior entries and the last one, at large positions where RoPE
    angles are far from zero."""
    rng = np.random.default_rng(16)
    m, C, N = 4, 64, 4096
    kv, gate, bias = _rand(rng, N, C), _rand(rng, N, C), _rand(rng, 2 * m, C, s=0.3)
    whole = O.compress(kv, gate, bias, m, d_rope=16)
    for e in (0, 1, 2, 517, N // m - 1):
        lo = max(0, (e - 1) * m)
        got = O.compress_entry(kv[lo:(e + 1) * m], gate[lo:(e + 1) * m], bias, e, m, d_rope=16)
        np.testing.assert_allclose(got, whole[e], rtol=1e-12, atol=1e-14)


def test_pooling_weights_sum_to_one():
    """The pooled value of a constant column is that constant (weights sum to 1)."""
    rng = np.random.default_rng(7)
    m, C = 8, 4
    kv = np.tile(np.array([1.5, -2.0, 0.25, 7.0]), (2 * m, 1))
    x = O.pool_window(kv, _rand(rng, 2 * m, C, s=3.0), _rand(rng, 2 * m, C))
    np.testing.assert_allclose(x, kv[0], rtol=1e-14)


# ------------------------------------------------------------------------------------ visibility
def test_visibility_rule_values():
    assert [O.visible(t, 4) for t in range(10)] == [0, 0, 0, 1, 1, 1, 1, 2, 2, 2]
    assert O.visible(1048578, 4) == 262144          # three-token tail stays invisible
    assert O.visible(262143, 128) == 2048


# ------------------------------------------------------------------------------------ indexer
def test_index_scores_brute_force_and_signed_weights():
    rng = np.random.default_rng(8)
    H, dI, m, t = 3, 8, 4, 21
    V = O.visible(t, m)
    q = _rand(rng, H, dI)
    w = np.array([0.7, -1.3, 0.2])
    cidx = _rand(rng, V + 2, dI)                     # extra rows beyond V must be ignored
    got = O.index_scores(q, w, cidx, t, m, d_rope=4)
    assert got.shape == (V,)
    qr = O.rope(q, t, 4)
    for i in range(V):
        s = 0.0
        for h in range(H):
            dot = sum(qr[h, j] * cidx[i, j] for j in range(dI))
            s += w[h] * (dot if dot > 0 else 0.0)
        assert abs(got[i] - s) < 1e-12
    # a negative weight lowers the score of an entry whose dot product with that head is positive
    i = int(np.argmax(cidx[:V] @ qr[1]))
    w2 = w.copy(); w2[1] = -5.0
    assert O.index_scores(q, w2, cidx, t, m, d_rope=4)[i] < got[i]


# ------------------------------------------------------------------------------------ top-k
def test_topk_brute_force_with_ties_and_padding():
    s = np.array([0.5, 2.0, -1.0, 2.0, 0.5, 3.0, 0.5])
    brute = sorted(range(len(s)), key=lambda i: (-s[i], i))
    for k in range(1, 10):
        got = O.topk_select(s, k)
        want = (brute + [-1] * k)[:k]
        assert got.tolist() == want
    rng = np.random.default_rng(9)
    s = np.round(rng.standard_normal(300), 1)        # many exact ties
    assert O.topk_select(s, 64).tolist() == sorted(range(300), key=lambda i: (-s[i], i))[:64]


# ------------------------------------------------------------------------------------ attention
def _small_cfg(**kw):
    base = dict(H=3, d=16, d_rope=8, H_idx=2, d_idx=8, ratio=4, top_k=3, window=5)
    base.update(kw)
    return O.OracleConfig(**base)


def test_attention_without_sink_or_compressed_is_textbook_softmax_attention():
    """sink -> -inf, no compressed entry visible, window >= t+1: plain causal softmax attention,
    checked against torch's scaled_dot_product_attention in float64."""
    rng = np.random.default_rng(10)
    cfg = _small_cfg(ratio=64, window=64)
    t = 9
    kv, q = _rand(rng, 12, cfg.d), _rand(rng, cfg.H, cfg.d)
    sink = np.full(cfg.H, -np.inf)
    o = O.sparse_attn(q, kv, np.zeros((0, cfg.d)), np.full(3, -1), sink, t, cfg)
    K = torch.from_numpy(O.rope(kv[:t + 1], np.arange(t + 1), cfg.d_rope))
    Q = torch.from_numpy(O.rope(q, t, cfg.d_rope))
    ref = torch.nn.functional.scaled_dot_product_attention(Q[None], K[None], K[None], scale=cfg.scale)[0]
    np.testing.assert_allclose(O.rope(o, t, cfg.d_rope), ref.numpy(), rtol=1e-12, atol=1e-14)


def test_single_candidate_gives_sigmoid_gate():
    rng = np.random.default_rng(11)
    cfg = _small_cfg(window=1)
    kv, q, sink = _rand(rng, 1, cfg.d), _rand(rng, cfg.H, cfg.d), _rand(rng, cfg.H)
    o = O.sparse_attn(q, kv, np.zeros((0, cfg.d)), np.full(3, -1), sink, 0, cfg)
    lg = cfg.scale * (q @ kv[0])                      # t = 0: RoPE is the identity
    sig = 1.0 / (1.0 + np.exp(sink - lg))
    np.testing.assert_allclose(o, sig[:, None] * kv[0][None], rtol=1e-13)


def test_sink_share_completes_the_weights():
    rng = np.random.default_rng(12)
    cfg = _small_cfg()
    t = 30
    kv, ckv = _rand(rng, 32, cfg.d), _rand(rng, 8, cfg.d)
    q, sink = _rand(rng, cfg.H, cfg.d), _rand(rng, cfg.H)
    sel = np.array([5, 0, 2])
    o, p, share = O.sparse_attn(q, kv, ckv, sel, sink, t, cfg, return_weights=True)
    np.testing.assert_allclose(p.sum(axis=1) + share, 1.0, rtol=1e-14)
    assert np.all(share > 0) and np.all(p.sum(axis=1) < 1)
    E, _ = O.attn_candidates(kv, ckv, sel, t, cfg)
    np.testing.assert_allclose(O.rope(o, t, cfg.d_rope), p @ E, rtol=1e-12, atol=1e-14)


def test_csa_with_k_at_least_visible_equals_hca_equals_dense_loops():
    rng = np.random.default_rng(13)
    cfg = _small_cfg(top_k=16)
    t = 27
    V = O.visible(t, cfg.ratio)
    kv, ckv = _rand(rng, 32, cfg.d), _rand(rng, 10, cfg.d)
    q, sink = _rand(rng, cfg.H, cfg.d, s=3.0), _rand(rng, cfg.H)
    sel = np.concatenate([np.random.default_rng(0).permutation(V), np.full(16 - V, -1)])
    o_csa = O.sparse_attn(q, kv, ckv, sel, sink, t, cfg)
    o_hca = O.sparse_attn(q, kv, ckv, None, sink, t, _small_cfg(top_k=0))
    np.testing.assert_allclose(o_csa, o_hca, rtol=1e-12, atol=1e-14)
    # dense scalar loops over every candidate (window rows rotated at own position)
    qr = O.rope(q, t, cfg.d_rope)
    cands = [O.rope(kv[j], j, cfg.d_rope) for j in range(t - cfg.window + 1, t + 1)] + [ckv[i] for i in range(V)]
    for h in range(cfg.H):
        lg = [cfg.scale * float(np.dot(qr[h], e)) for e in cands]
        z = math.exp(sink[h]) + sum(math.exp(v) for v in lg)
        oh = sum(math.exp(v) * e for v, e in zip(lg, cands)) / z
        np.testing.assert_allclose(o_csa[h], O.rope(oh, t, cfg.d_rope, inverse=True),
                                   rtol=1e-11, atol=1e-14)


# ------------------------------------------------------------------------------------ whole path
def _seq(rng, cfg, N):
    return dict(kv=_rand(rng, N, cfg.d, s=0.3), gate=_rand(rng, N, cfg.d),
                bias=_rand(rng, 2 * cfg.ratio, cfg.d, s=0.3), idx_k=_rand(rng, N, cfg.d_idx, s=0.3),
                idx_gate=_rand(rng, N, cfg.d_idx), idx_bias=_rand(rng, 2 * cfg.ratio, cfg.d_idx, s=0.3),
                q=_rand(rng, N, cfg.H, cfg.d, s=2.0), q_idx=_rand(rng, N, cfg.H_idx, cfg.d_idx),
                w=_rand(rng, N, cfg.H_idx), sink=_rand(rng, cfg.H))


@pytest.mark.parametrize("top_k", [3, 0])
def test_prefill_equals_streaming(top_k):
    rng = np.random.default_rng(14)
    cfg = _small_cfg(top_k=top_k)
    x = _seq(rng, cfg, 26)
    o_pre, _, _ = O.prefill(**x, cfg=cfg)
    o_str = O.decode_stream(**x, cfg=cfg)
    np.testing.assert_allclose(o_pre, o_str, rtol=0, atol=1e-12)


def test_group_boundary_fault_is_caught(monkeypatch):
    """A visibility rule one token late (t // m) matches streaming for the first 3 tokens,
    breaks at the 4th and again at the 8th: the mutation must fail prefill == streaming."""
    rng = np.random.default_rng(15)
    cfg = _small_cfg(top_k=2)
    x = _seq(rng, cfg, 9)
    o_str = O.decode_stream(**x, cfg=cfg)
    monkeypatch.setattr(O, "visible", lambda t, m: t // m)
    o_bad, _, _ = O.prefill(**x, cfg=cfg)
    err = np.abs(o_bad - o_str).max(axis=(1, 2))
    assert np.all(err[:3] < 1e-12)
    assert err[3] > 1e-6 and err[7] > 1e-6
    assert np.all(err[4:7] < 1e-12)


def test_causality_future_tokens_do_not_change_past_outputs():
    rng = np.random.default_rng(16)
    cfg = _small_cfg(top_k=2)
    x = _seq(rng, cfg, 20)
    o1, _, _ = O.prefill(**x, cfg=cfg)
    t0 = 10
    y = {k: v.copy() for k, v in x.items()}
    for k in ("kv", "gate", "idx_k", "idx_gate", "q", "q_idx", "w"):
        y[k][t0 + 1:] += 5.0
    o2, _, _ = O.prefill(**y, cfg=cfg)
    assert np.array_equal(o1[:t0 + 1], o2[:t0 + 1])
    assert np.abs(o1[t0 + 1:] - o2[t0 + 1:]).max() > 1e-3


# ------------------------------------------------------------------------------------ off-path toys
def test_mhc_worked_example():
    new = mhc_residual_update(r_old=[2, 4, 6, 8], z=6.0, F=lambda z: 2 * z, B=np.eye(4),
                              post=[0.25, 0.5, 0.75, 1.0])
    np.testing.assert_allclose(new, [5, 10, 15, 20])


def test_routing_worked_example():
    # the lab prints [0.3, 1.2]: two selected experts with un-biased scores in ratio 1:4
    ids, w = routing_weights(scores=[0.2, 0.8, 0.1], bias=[0.7, 0, 0], k=2, route_scale=1.5)
    assert ids.tolist() == [0, 1]           # the bias decides the choice, not the weights
    np.testing.assert_allclose(w, [0.3, 1.2])
    assert abs(w.sum() - 1.5) < 1e-15
