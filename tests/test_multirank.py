"""The multi-rank logic of the benchmark, as world_size-2 gloo process groups on the CPU.

Decode requests are independent, so N GPUs serve N disjoint sets of requests with no data-path
collective (weak scaling); the only exchanges are the timing barrier and the max over ranks of the
elapsed time, and the whole-job value counts every rank's requests. These tests run that logic in
two CPU processes, and run the reference arm as rank 0 and rank 1 of a two-rank launch.
"""
import importlib.util
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench = _bench()
        import synth
        B = 32
        mine = bench.rank_requests(rank, B)
        every = [None] * world
        dist.all_gather_object(every, mine)
        flat = [r for part in every for r in part]
        assert len(flat) == len(set(flat)) == world * B, "ranks serve overlapping requests"
        assert sorted(flat) == list(range(world * B))
        # distinct requests draw distinct data (their own seeds)
        wl = synth.small_workload(1, wid=300, B=2, N=64, t=63)
        reqs = synth.gen_requests(wl, bench.rank_requests(rank, 2))
        digest = float(np.sum(reqs[0]["q"]))
        digests = [None] * world
        dist.all_gather_object(digests, digest)
        assert len(set(digests)) == world, "two ranks drew the same request"
        # the job takes as long as its slowest rank; the value counts every rank's requests
        bench.barrier(world)
        el = bench.max_over_ranks(1.0 + 0.5 * rank, world)
        assert el == 1.0 + 0.5 * (world - 1)
        assert bench.job_value(world, B, 10, el) == pytest.approx(world * B * 10 / el)
    finally:
        dist.destroy_process_group()


def test_two_ranks_disjoint_requests_and_max_timing():
    mp.spawn(_rank_main, args=(2, _free_port()), nprocs=2, join=True)


def test_reference_arm_two_ranks():
    """Under a two-rank launch only rank 0 times the oracle and prints the line; rank 1 exits 0."""
    env = dict(os.environ, WORLD_SIZE="2", MASTER_ADDR="127.0.0.1", MASTER_PORT=str(_free_port()))
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2", "--warmup", "3"]
    r1 = subprocess.run(cmd, env=dict(env, RANK="1", LOCAL_RANK="1"), capture_output=True, text=True, timeout=600)
    assert r1.returncode == 0 and r1.stdout.strip() == "", r1.stderr[-2000:]
    r0 = subprocess.run(cmd, env=dict(env, RANK="0", LOCAL_RANK="0"), capture_output=True, text=True, timeout=600)
    assert r0.returncode == 0, r0.stderr[-2000:]
    lines = [ln for ln in r0.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["steps"] == 2
    assert line["value"] > 0 and line["e2e"]["value"] == line["value"]
    assert line["cpu_baseline"]["kind"] == "oracle"
