"""The exchange over entry-range shards as a world_size-2 gloo process group on the CPU: each rank
holds half of one request's compressed caches, scores and selects among its own entries, the ranks
all-gather their (score, entry) candidates and merge them, attend over their own selected rows (rank
0 also over the raw window), all-gather the partials and merge them with the sink once. Both ranks
must reach exactly the unsharded selection and the unsharded attention output (fp64 oracle)."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port):
    import sys
    sys.path.insert(0, ROOT)
    from oracle import csa_oracle as O
    from oracle import exchange as X
    import synth
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wl = synth.small_workload(1, wid=320, B=1, N=2051, t=2050, top_k=64, window=32, H=8, H_idx=8)
        cfg = O.OracleConfig(H=wl.H, H_idx=wl.H_idx, top_k=wl.top_k, window=wl.window, ratio=wl.ratio)
        r = synth.gen_requests(wl, [0])[0]
        sh = synth.gen_shared(wl)
        t, k = wl.t, wl.top_k
        n = wl.n_entries
        ckv = O.compress(r["kv"], r["gate"], sh["bias"], wl.ratio, n)
        cidx = O.compress(r["idx_k"], r["idx_gate"], sh["idx_bias"], wl.ratio, n)
        base, cnt = X.shard_ranges(n, world)[rank]
        # this rank's share: its entries only (scores of the global visible entries it holds)
        V = O.visible(t, wl.ratio)
        s_all = np.zeros(V)
        hi = min(base + cnt, V)
        if hi > base:
            s_all[base:hi] = _scores_of_rows(O, r, cidx[base:hi], t, wl.ratio)
        gi, gs = X.local_candidates(s_all, base, cnt, k)
        pad_i = np.full(k, -1, np.int64)
        pad_s = np.full(k, -np.inf)
        pad_i[:len(gi)], pad_s[:len(gs)] = gi, gs
        all_i = [torch.zeros(k, dtype=torch.int64) for _ in range(world)]
        all_s = [torch.zeros(k, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(all_i, torch.from_numpy(pad_i))
        dist.all_gather(all_s, torch.from_numpy(pad_s))
        cands = [(a.numpy()[a.numpy() >= 0], b.numpy()[a.numpy() >= 0]) for a, b in zip(all_i, all_s)]
        sel = X.merge_candidates(cands, k)
        ref_s = O.index_scores(r["q_idx"][0], r["w"][0], cidx, t, wl.ratio)
        want = O.topk_select(ref_s, k)
        np.testing.assert_array_equal(sel, np.sort(want[want >= 0]))
        # attention partials over this rank's selected rows (rank 0 also the raw window)
        mine = sel[(sel >= base) & (sel < base + cnt)]
        rows = ckv[mine]
        if rank == 0:
            lo = max(0, t - cfg.window + 1)
            rows = np.concatenate([O.rope(r["kv"][lo:t + 1], np.arange(lo, t + 1), cfg.d_rope, cfg.rope_base), rows])
        m, l, o = X.attn_partial(r["q"][0], rows, t, cfg)
        part = torch.from_numpy(np.concatenate([m, l, o.reshape(-1)]))
        parts = [torch.zeros_like(part) for _ in range(world)]
        dist.all_gather(parts, part)
        H, d = cfg.H, cfg.d
        got = X.merge_partials([(p[:H].numpy(), p[H:2 * H].numpy(), p[2 * H:].numpy().reshape(H, d)) for p in parts],
                               sh["sink"], t, cfg)
        ref = O.sparse_attn(r["q"][0], r["kv"], ckv, want, sh["sink"], t, cfg)
        np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-14)
    finally:
        dist.destroy_process_group()


def _scores_of_rows(O, r, rows, t, ratio):
    """The indexer score of each of these rows (the oracle's formula on a shard's own rows)."""
    qr = O.rope(r["q_idx"][0], t)
    return np.maximum(np.asarray(rows) @ qr.T, 0.0) @ np.asarray(r["w"][0], np.float64)


def test_two_ranks_exchange_equals_unsharded():
    mp.spawn(_rank_main, args=(2, _free_port()), nprocs=2, join=True)
