"""GPU parity of the exchange over entry-range shards, with G shards laid out side by side on one
device (what a multi-device caller all-gathers is here simply stacked): each shard's candidates, the
merged selection, each shard's attention partials and their merge, against the fp64 oracle on the
GPU's compressed caches (stage-chained), and the candidate merge kernel alone against the oracle's
merge on planted ties."""
import numpy as np
import pytest
import torch

import synth
from oracle import csa_oracle as O
from oracle import exchange as X
from tests import _harness as Hn

pytestmark = pytest.mark.gpu

CASES = {
    "csa_bf16": (synth.small_workload(1, wid=330, B=3, N=4099, t=4098), [4098, 4095, 2050]),
    "csa_bf16_k256": (synth.small_workload(1, wid=331, B=2, N=8195, t=8194, top_k=256), [8194, 3001]),
    "csa_f32": (synth.small_workload(0, wid=332, B=2), [2047, 1001]),
    "hca_bf16": (synth.small_workload(3, wid=333, B=2, N=8256, t=8255), [8255, 5000]),
}


@pytest.mark.parametrize("G", [2, 3])
@pytest.mark.parametrize("name", list(CASES))
def test_exchange_matches_oracle(name, G):
    wl, pos_l = CASES[name]
    bt = Hn.DeviceBatch(wl)
    c, o = Hn.configs(wl)
    L = Hn.lib()
    L.csa_compress(c, bt.cache(), 0, wl.n_entries)
    B, k, n_cap = bt.B, c.top_k, wl.n_entries
    pos = torch.tensor(pos_l, dtype=torch.int64, device="cuda")
    ranges = X.shard_ranges(n_cap, G)
    ckv_sh = [bt.ckv[:, b:b + n].contiguous() for b, n in ranges]
    sel_sh = None
    topk = None
    if not o.hca:
        cidx_sh = [bt.cidx[:, b:b + n].contiguous() for b, n in ranges]
        cand_idx = torch.full((B, G, k), -7, dtype=torch.int32, device="cuda")
        cand_score = torch.full((B, G, k), float("nan"), device="cuda")
        for g, (b0, n) in enumerate(ranges):
            ci = torch.full((B, k), -7, dtype=torch.int32, device="cuda")
            cs = torch.full((B, k), float("nan"), device="cuda")
            L.csa_index_topk_shard(c, pos, bt.q_idx[:, 0].contiguous(), bt.w[:, 0].contiguous(), cidx_sh[g], b0, ci, cs)
            cand_idx[:, g], cand_score[:, g] = ci, cs
        topk = torch.full((B, k), -7, dtype=torch.int32, device="cuda")
        sel_sh = torch.full((B, G, k), -7, dtype=torch.int32, device="cuda")
        L.csa_topk_merge(c, cand_score, cand_idx, [b for b, _ in ranges], [n for _, n in ranges], topk, sel_sh)
    part_o = torch.full((B, G, c.H, c.d), float("nan"), device="cuda")
    part_ml = torch.full((B, G, c.H, 2), float("nan"), device="cuda")
    for g, (b0, n) in enumerate(ranges):
        po = torch.empty((B, c.H, c.d), device="cuda")
        pm = torch.empty((B, c.H, 2), device="cuda")
        L.csa_sparse_attn_shard(c, pos, bt.q[:, 0].contiguous(), bt.kv, ckv_sh[g], b0,
                                None if o.hca else sel_sh[:, g].contiguous(), g == 0, po, pm)
        part_o[:, g], part_ml[:, g] = po, pm
    out = torch.full((B, c.H, c.d), float("nan"), dtype=c.dtype, device="cuda")
    L.csa_attn_merge(c, pos, part_o, part_ml, bt.sink, out)
    torch.cuda.synchronize()
    assert L.csa_get_device_status() == 0
    ckv = Hn.host64(bt.ckv)
    cidx = None if o.hca else Hn.host64(bt.cidx)
    for b, t in enumerate(pos_l):
        sel = None
        if not o.hca:
            ref_s = O.index_scores(bt.reqs[b]["q_idx"][0], bt.reqs[b]["w"][0], cidx[b], t, c.ratio)
            cands = []
            for g, (b0, n) in enumerate(ranges):
                ci = cand_idx[b, g].cpu().numpy().astype(np.int64)
                cs = cand_score[b, g].double().cpu().numpy()
                valid = ci >= 0
                assert np.all(np.diff(ci[valid]) > 0) and np.all(ci[~valid] == -1)
                # the candidates are the shard's exact top k on its own scores, and those scores are
                # the oracle's within the indexer tolerance
                Hn.check_scores(cs[valid], ref_s[ci[valid] + b0], wl.storage,
                                f"{name} G{G} shard {g} candidate scores b{b}")
                cands.append((ci[valid] + b0, cs[valid]))
            sel = topk[b].cpu().numpy()
            np.testing.assert_array_equal(sel, X.merge_candidates(cands, k))      # the merge kernel, exactly
            Hn.check_topk_vs_oracle(sel, ref_s, k, f"{name} G{G} merged selection b{b}")
            for g, (b0, n) in enumerate(ranges):                                   # each shard's own list
                mine = sel[(sel >= b0) & (sel < b0 + n)] - b0
                got = sel_sh[b, g].cpu().numpy()
                np.testing.assert_array_equal(got[:len(mine)], mine)
                assert np.all(got[len(mine):] == -1)
        ref = O.sparse_attn(bt.reqs[b]["q"][0], bt.reqs[b]["kv"], ckv[b], sel, bt.shared["sink"], t, o)
        Hn.check_attn(Hn.host64(out[b]), ref, wl.storage, f"{name} G{G} merged attention b{b}")


@pytest.mark.parametrize("G,k", [(2, 512), (4, 64), (8, 512), (3, 1024)])
def test_candidate_merge_kernel_exact_with_ties(G, k):
    """csa_topk_merge on random candidate lists with planted equal scores (ties broken by the lower
    global index), empty slots, and unequal shards: exactly the oracle's merge."""
    L = Hn.lib()
    c = L.Config(top_k=k)
    rng = np.random.default_rng(G * 7 + k)
    B = 3
    counts = [int(x) for x in rng.integers(k // 2, 4 * k, G)]
    bases = list(np.cumsum([0] + counts[:-1]))
    cand_idx = np.full((B, G, k), -1, np.int32)
    cand_score = np.full((B, G, k), -np.inf, np.float32)
    for b in range(B):
        for g in range(G):
            m = int(rng.integers(0, min(k, counts[g]) + 1))
            cand_idx[b, g, :m] = np.sort(rng.choice(counts[g], m, replace=False))
            cand_score[b, g, :m] = np.round(rng.standard_normal(m), 1)          # many equal scores
    topk = torch.full((B, k), -7, dtype=torch.int32, device="cuda")
    sel_sh = torch.full((B, G, k), -7, dtype=torch.int32, device="cuda")
    L.csa_topk_merge(c, torch.from_numpy(cand_score).cuda(), torch.from_numpy(cand_idx).cuda(), bases, counts, topk, sel_sh)
    torch.cuda.synchronize()
    for b in range(B):
        cands = []
        for g in range(G):
            v = cand_idx[b, g] >= 0
            cands.append((cand_idx[b, g][v].astype(np.int64) + bases[g], cand_score[b, g][v].astype(np.float64)))
        np.testing.assert_array_equal(topk[b].cpu().numpy(), X.merge_candidates(cands, k))
