"""The bench's algorithmic byte and flop counts (CPU): the headline step's figures as written out by
hand from the workload's shapes, and the FP4 / FP8 cache counted with the bytes of the format
(the oracle's own description of its layout)."""
import importlib.util
import os

import pytest

import synth
from oracle import cache_lowp as Q

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_accounting", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_headline_step_bytes_and_flops():
    b = _bench()
    w = b.decode_work(synth.WORKLOADS[1], 32)
    # index cache 32 x 16,384 x 256 B, q_idx + w; KV rows 32 x (128 + 512) x 1 KB; q, sink, out;
    # the closing group: 8 raw tokens x (512 + 128) channels x (kv + gate) x 2 B + both new entries
    idx = 32 * (16384 * 256 + 64 * 128 * 2 + 64 * 4)
    kv = 32 * 640 * 1024
    q = 32 * 64 * 512 * 2 + 64 * 4
    out = 32 * 64 * 512 * 2
    close = 32 * (8 * 640 * 2 * 2 + 640 * 2)
    assert w["index_bytes"] == idx == 134750208
    assert w["bytes"] == idx + kv + q + out + close
    assert w["flops"] == 2 * 32 * 64 * 128 * 16384 + 4 * 32 * 64 * 640 * 512


@pytest.mark.parametrize("C", [512, 128])
def test_fp4_entry_bytes_follow_the_format(C):
    b = _bench()
    wl = b.FP4_DECODE_WL
    n = 4096
    lay = Q.cache_layout(C, n)
    assert b.entry_bytes(wl, C) * n == lay["stride"]          # n a multiple of 8: no padding
    assert b.entry_bytes(synth.WORKLOADS[1], C) == 2 * C


def test_fp4_headline_moves_fewer_bytes():
    b = _bench()
    bf, fp = b.decode_work(synth.WORKLOADS[1], 32), b.decode_work(b.FP4_DECODE_WL, 32)
    assert fp["index_bytes"] == 32 * (16384 * 98 + 64 * 128 * 2 + 64 * 4)
    assert fp["flops"] == bf["flops"] and fp["bytes"] < bf["bytes"] / 2.4
