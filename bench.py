#!/usr/bin/env python3
"""CSA decode benchmark on B300: query-tokens/s and HBM GB/s of one decode step of B = 32 requests
at N = 65,536 (one query each at t = N - 1: compress-on-close, indexer, top-k 512, sparse attention
over window 128 + 512 selected entries, sink, inverse RoPE), plus the 8K causal prefill (TFLOP/s).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line on rank 0. Under torchrun (N > 1) every rank runs its own 32 requests
(weak scaling, no data-path collective); the timed region is bracketed by a barrier and a device
synchronise on both sides and the max over ranks is reported. `--impl reference` times the fp64
NumPy oracle on the host cores on the same workload.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

DECODE_WL = synth.WORKLOADS[1]
PREFILL_WL = synth.WORKLOADS[2]
ROTATIONS = 3                      # input copies cycled between steps (defeats the 126 MB L2)
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
# DRAM bytes (read + write) of one launch of the fused decode indexer (scores, closing entries,
# top-k selection) at the decode workload. Captured on B=4 requests (one kernel, one launch; the
# profile is profiles/index_select_decode_B32_N65536.md) and scaled by 8 to B=32: every request
# streams its own cache, so the bytes grow with B. They hold only for the kernel source they were
# taken on: the roofline's "traffic" is null as soon as the code of any of these files differs.
INDEX_TRAFFIC = {"bytes_per_launch": 8 * (19144448 + 0),
                 "sources": ["long_context_sparse_19_b300/csrc/tc_index_select.cu",
                             "long_context_sparse_19_b300/csrc/tc_ptx.cuh",
                             "long_context_sparse_19_b300/csrc/common.cuh",
                             "long_context_sparse_19_b300/csrc/close_entry.cuh"],
                 "sha256": "4a071f5fb49a8b2d018aa72d2c55a31696ac1504f2b3cf04b5412c70f1da1b55"}
# GPU sleep queued ahead of each profiled step, so that the host has submitted the whole step before
# it starts and the per-kernel events time the GPU, not the host's launch rate (~250 us at 2 GHz)
PROFILE_SLEEP_CYCLES = 500_000


def source_digest(paths) -> str:
    """SHA-256 of the code of CUDA sources: // comments and blank lines do not count, so that a
    comment edit does not void a counter taken on the same code."""
    import hashlib
    import re
    h = hashlib.sha256()
    for rel in paths:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            for line in f:
                code = re.sub(r"//.*", "", line).rstrip()
                if code:
                    h.update(code.encode() + b"\n")
    return h.hexdigest()


def index_traffic() -> int | None:
    ok = source_digest(INDEX_TRAFFIC["sources"]) == INDEX_TRAFFIC["sha256"]
    return INDEX_TRAFFIC["bytes_per_launch"] if ok else None


def load_peaks() -> dict:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        d["source"] = "measured"
    except (OSError, ValueError):
        d = dict(FALLBACK_PEAKS)
        d["source"] = "fallback"
    return d


# ----------------------------------------------------------------------------- work accounting
def entry_bytes(wl: synth.Workload, C: int) -> int:
    """Bytes of one compressed entry of C dims in the workload's cache storage (the FP4 / FP8 format:
    (C - 64) / 2 bytes of E2M1 codes, 64 of E4M3 codes and the block scales: 304 for C = 512, 98 for
    C = 128)."""
    if wl.storage == "fp4":
        nb = (C - wl.d_rope) // 32
        return (C - wl.d_rope) // 2 + wl.d_rope + (16 if nb > 2 else 2)
    return C * (4 if wl.storage == "f32" else 2)


def decode_work(wl: synth.Workload, B: int) -> dict:
    """Algorithmic bytes / flops of one decode step of B requests (what the method must move:
    the visible index cache, the gathered candidate rows, q / q_idx / w / sink, the output, and the
    closing group of the compressor). Score round-trips and split partials are overhead, excluded."""
    es = 4 if wl.storage == "f32" else 2              # raw rows, q, out (bf16 also with fp4 caches)
    t, m = wl.t, wl.ratio
    V = (t + 1) // m
    n_win = min(wl.window, t + 1)
    n_comp = V if wl.hca else min(wl.top_k, V)
    C = n_win + n_comp
    idx_bytes = 0 if wl.hca else B * (V * entry_bytes(wl, wl.d_idx) + wl.H_idx * wl.d_idx * es + wl.H_idx * 4)
    kv_bytes = B * (n_win * wl.d * es + n_comp * entry_bytes(wl, wl.d))
    q_bytes = B * wl.H * wl.d * es + wl.H * 4
    out_bytes = B * wl.H * wl.d * es
    close = (t + 1) % m == 0
    chans = wl.d + (0 if wl.hca else wl.d_idx)
    ent = entry_bytes(wl, wl.d) + (0 if wl.hca else entry_bytes(wl, wl.d_idx))
    comp_bytes = B * (2 * m * chans * 2 * es + ent) if close else 0
    flops_idx = 0 if wl.hca else 2 * B * wl.H_idx * wl.d_idx * V
    flops_attn = 4 * B * wl.H * C * wl.d
    return {"bytes": idx_bytes + kv_bytes + q_bytes + out_bytes + comp_bytes, "index_bytes": idx_bytes,
            "flops": flops_idx + flops_attn, "flops_index": flops_idx, "flops_attn": flops_attn}


def prefill_flops(wl: synth.Workload) -> dict:
    t = np.arange(wl.S, dtype=np.int64)
    V = (t + 1) // wl.ratio
    idx = 0 if wl.hca else int(2 * wl.H_idx * wl.d_idx * V.sum())
    comp = V if wl.hca else np.minimum(wl.top_k, V)
    attn = int(4 * wl.H * wl.d * (comp + np.minimum(wl.window, t + 1)).sum())
    return {"index": wl.B * idx, "attn": wl.B * attn, "total": wl.B * (idx + attn)}


# ----------------------------------------------------------------------------- clocks during the run
class ClockSampler:
    PERIOD_MS = 20                        # several samples even inside a sub-second timed region
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.samples: list[tuple[float, list[str]]] = []
        self.err = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(ClockSampler.PERIOD_MS), "-i", gpu_id], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError as e:
            self.proc, self.err = None, str(e)
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float) -> dict:
        if self.proc is None:
            return {"unavailable": self.err}
        inside = [s for ts, s in self.samples if t0 <= ts <= t1]
        note = "in timed region"
        if not inside:                           # region shorter than the sampling period
            near = sorted(self.samples, key=lambda x: min(abs(x[0] - t0), abs(x[0] - t1)))[:2]
            inside = [s for _, s in near]
            note = f"nearest samples (timed region shorter than the {self.PERIOD_MS} ms sampling period)"
        if not inside:
            return {"unavailable": "no nvidia-smi samples"}
        sm = [float(s[1]) for s in inside if s[1].replace(".", "").isdigit()]
        mx = [float(s[2]) for s in inside if s[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for s in inside for n, v in zip(names, s[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(inside), "note": note}


# ----------------------------------------------------------------------------- distributed plumbing
def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group(dist_backend(), device_id=torch.device("cuda", local))
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def dist_backend() -> str:
    """NCCL between GPUs; gloo where there is none (the host-side tests of the multi-rank logic)."""
    import torch
    return "nccl" if torch.cuda.is_available() else "gloo"


def rank_requests(rank: int, B: int) -> list[int]:
    """The requests rank `rank` serves: its own B of them, so every rank's work is distinct (weak
    scaling: the job's requests grow with the ranks, nothing is exchanged on the data path)."""
    return list(range(rank * B, rank * B + B))


def job_value(world: int, B: int, K: int, seconds_max: float) -> float:
    """Whole-job query-tokens/s: every rank decodes B requests per step for K steps, and the job
    takes as long as its slowest rank."""
    return world * B * K / seconds_max


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- device inputs
def device_inputs(wl: synth.Workload, requests, device):
    """Draws the requests (host threads) and uploads them into [B, ...] device tensors as they
    are drawn, so the host never holds the whole batch."""
    import torch
    B = len(requests)
    dt = torch.float32 if wl.storage == "f32" else torch.bfloat16
    T = {"kv": torch.empty(B, wl.N, wl.d, dtype=dt, device=device),
         "gate": torch.empty(B, wl.N, wl.d, dtype=dt, device=device),
         "q": torch.empty(B, wl.S, wl.H, wl.d, dtype=dt, device=device)}
    if not wl.hca:
        T["idx_k"] = torch.empty(B, wl.N, wl.d_idx, dtype=dt, device=device)
        T["idx_gate"] = torch.empty(B, wl.N, wl.d_idx, dtype=dt, device=device)
        T["q_idx"] = torch.empty(B, wl.S, wl.H_idx, wl.d_idx, dtype=dt, device=device)
        T["w"] = torch.empty(B, wl.S, wl.H_idx, dtype=torch.float32, device=device)
    slot = {b: i for i, b in enumerate(requests)}

    def up(b, r):
        i = slot[b]
        for k, v in r.items():
            if v is None:
                continue
            if k == "w" or wl.storage == "f32":
                src = torch.from_numpy(np.ascontiguousarray(v, np.float32))
            else:
                src = torch.from_numpy(synth.bf16_bits(v).view(np.int16)).view(torch.bfloat16)
            T[k][i].copy_(src)
        return None

    synth.gen_requests(wl, requests, fn=up)
    sh = synth.gen_shared(wl)
    T["bias"] = torch.from_numpy(sh["bias"]).to(device)
    T["sink"] = torch.from_numpy(sh["sink"]).to(device)
    if not wl.hca:
        T["idx_bias"] = torch.from_numpy(sh["idx_bias"]).to(device)
    torch.cuda.synchronize()
    return T


def make_cfg(wl):
    import long_context_sparse_19_b300 as L
    return L.Config(H=wl.H, d=wl.d, d_rope=wl.d_rope, H_idx=wl.H_idx, d_idx=wl.d_idx, ratio=wl.ratio,
                    top_k=wl.top_k, window=wl.window, storage=wl.storage)


def make_cache(T, wl, device):
    import long_context_sparse_19_b300 as L
    B = T["kv"].shape[0]
    cfg = make_cfg(wl)
    ckv = L.cache_tensor(cfg, B, wl.n_entries, 0, device=device)
    cidx = None if wl.hca else L.cache_tensor(cfg, B, wl.n_entries, 1, device=device)
    return L.Cache(kv=T["kv"], gate=T["gate"], gate_bias=T["bias"], ckv=ckv, idx_k=T.get("idx_k"),
                   idx_gate=T.get("idx_gate"), idx_bias=T.get("idx_bias"), cidx=cidx, n_cap=wl.n_entries)


# ----------------------------------------------------------------------------- our decode leg
def run_decode(args, world, rank, device, peaks) -> dict:
    import torch
    import long_context_sparse_19_b300 as L
    wl = headline_wl(args)
    B = wl.B
    R = args.rotations
    cfg = make_cfg(wl)
    t_setup = time.time()
    T = device_inputs(wl, rank_requests(rank, B), device)
    cache = make_cache(T, wl, device)
    L.csa_compress(cfg, cache, 0, wl.n_entries)            # the caches the decode step reads
    pos = torch.full((B,), wl.t, dtype=torch.int64, device=device)
    rot = []
    for r in range(R):
        if r == 0:
            c, q, qi, w = cache, T["q"][:, 0].contiguous(), T["q_idx"][:, 0].contiguous(), T["w"][:, 0].contiguous()
        else:
            c = L.Cache(kv=cache.kv.clone(), gate=cache.gate.clone(), gate_bias=cache.gate_bias,
                        ckv=cache.ckv.clone(), idx_k=cache.idx_k.clone(), idx_gate=cache.idx_gate.clone(),
                        idx_bias=cache.idx_bias, cidx=cache.cidx.clone(), n_cap=cache.n_cap)
            q, qi, w = rot[0]["q"].clone(), rot[0]["q_idx"].clone(), rot[0]["w"].clone()
        out = torch.empty(B, wl.H, wl.d, dtype=cache.kv.dtype, device=device)
        ws = L.workspace(cfg, B, 1, wl.n_entries, device=device)
        rot.append({"cache": c, "q": q, "q_idx": qi, "w": w, "out": out, "pos": pos.clone(), "ws": ws, "cfg": cfg,
                    "sink": T["sink"]})
        rot[-1]["call"] = L.binding.bind_decode(cfg, rot[-1]["pos"], c, q, qi, w, T["sink"], out, ws=ws)
    torch.cuda.synchronize()
    setup_s = time.time() - t_setup

    # CUDA graph of one decode step per input copy (the C-ABI call captured on the capture stream)
    for r in rot:
        r["call"]()
    torch.cuda.synchronize()
    n0 = L.csa_launch_count()
    graphs = []
    for r in rot:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            r["call"]()
        graphs.append(g)
    launches_per_step = (L.csa_launch_count() - n0) // R
    assert L.csa_get_device_status() == 0

    for i in range(args.warmup):
        graphs[i % R].replay()
    K = args.steps
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(gpu_ident(device))
    time.sleep(0.25)
    barrier(world)
    torch.cuda.synchronize()
    wall0 = time.time()
    ev0.record()
    for i in range(K):
        graphs[i % R].replay()
    ev1.record()
    torch.cuda.synchronize()
    wall1 = time.time()
    barrier(world)
    clocks.stop()
    ms = ev0.elapsed_time(ev1)
    ms_max = max_over_ranks(ms, world)
    clk = clocks.summary(wall0, wall1)

    # Second pass, same steps without the graph, with a CUDA event pair around every kernel on its
    # launching stream: per-kernel average durations for the roofline. A GPU sleep ahead of each
    # step lets the host queue the whole step first, so no event waits on a host-side launch.
    L.csa_profile_begin(K * launches_per_step + 16)
    for i in range(K):
        torch.cuda._sleep(PROFILE_SLEEP_CYCLES)
        rot[i % R]["call"]()
    torch.cuda.synchronize()
    prof = L.csa_profile_end()

    # End to end: per step, the step's inputs (q, q_idx, w, the new token's raw rows) come from
    # pinned host memory and the output goes back to pinned host memory, all inside the region.
    e2e = None if args.no_e2e else run_e2e(args, wl, rot, world, device)
    assert L.csa_get_device_status() == 0

    work = decode_work(wl, B)
    idx_ms, idx_n = prof["index"]
    idx_avg_s = idx_ms / max(idx_n, 1) / 1e3
    achieved = work["index_bytes"] / idx_avg_s / 1e9 if idx_n else None
    step_s = ms_max / K / 1e3
    qtok = job_value(world, B, K, ms_max / 1e3)
    res = {
        "value": qtok, "ms_per_step": ms_max / K, "hbm_gbs": work["bytes"] / step_s / 1e9,
        "hbm_frac_of_measured": work["bytes"] / step_s / 1e9 / peaks["hbm_gbs"],
        "step_bytes": work["bytes"], "step_flops": work["flops"], "gpu_launches": launches_per_step * K,
        "clocks": clk, "setup_s": round(setup_s, 1),
        "stage_sum_ms_per_step": sum(v[0] for v in prof.values()) / K,
        "stages_ms_per_step": {k: round(v[0] / K, 5) for k, v in prof.items()},
        "stage_launches": {k: v[1] for k, v in prof.items()},
        "roofline": {"kernel": "fused indexer: scores + closing entries + top-k (csa_decode stage 1)", "bound": "hbm",
                     "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": (achieved / peaks["hbm_gbs"]) if achieved else None,
                     "traffic": index_traffic() if wl.storage == "bf16" else None,
                     "algorithmic_bytes_per_launch": work["index_bytes"],
                     "avg_launch_us": idx_avg_s * 1e6, "peak_source": peaks["source"]},
        "e2e": e2e,
    }
    return res


def gpu_ident(device) -> str:
    import torch
    try:
        u = str(torch.cuda.get_device_properties(device).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return str(torch.cuda.current_device())


def run_e2e(args, wl, rot, world, device) -> dict:
    import torch
    import long_context_sparse_19_b300 as L
    B, t = wl.B, wl.t
    dt = rot[0]["q"].dtype
    # Per input copy: the step's inputs packed in one pinned host buffer (q, q_idx, w, pos and the
    # new token's raw rows of the four raw caches), uploaded by one copy into a device staging
    # buffer; csa_decode reads q, q_idx, w and pos in place there, and the raw rows are copied into
    # the caches on the device.
    parts = [("q", (B, wl.H, wl.d), dt), ("q_idx", (B, wl.H_idx, wl.d_idx), dt), ("w", (B, wl.H_idx), torch.float32),
             ("pos", (B,), torch.int64), ("kv", (B, wl.d), dt), ("gate", (B, wl.d), dt),
             ("idx_k", (B, wl.d_idx), dt), ("idx_gate", (B, wl.d_idx), dt)]
    offs, o = {}, 0
    for name, shape, typ in parts:
        offs[name] = o
        o += -(-math.prod(shape) * torch.empty((), dtype=typ).element_size() // 256) * 256
    total = o

    def views(buf):
        out = {}
        for name, shape, typ in parts:
            n = math.prod(shape) * torch.empty((), dtype=typ).element_size()
            out[name] = buf[offs[name]:offs[name] + n].view(typ).view(shape)
        return out

    host, stage = [], []
    for r in rot:
        c = r["cache"]
        hbuf = torch.empty(total, dtype=torch.uint8).pin_memory()
        hv = views(hbuf)
        src = {"q": r["q"], "q_idx": r["q_idx"], "w": r["w"], "pos": r["pos"], "kv": c.kv[:, t], "gate": c.gate[:, t],
               "idx_k": c.idx_k[:, t], "idx_gate": c.idx_gate[:, t]}
        for name in hv:
            hv[name].copy_(src[name].cpu())
        dbuf = torch.empty(total, dtype=torch.uint8, device=device)
        dv = views(dbuf)
        stage.append({"buf": dbuf, **dv})
        host.append({"buf": hbuf, "out": torch.empty((B, wl.H, wl.d), dtype=dt).pin_memory()})
        # the decode call reads its per-step inputs straight from the staging buffer
        r["e2e_call"] = L.binding.bind_decode(r["cfg"], dv["pos"], c, dv["q"], dv["q_idx"], dv["w"], r["sink"],
                                              r["out"], ws=r["ws"])
    h2d = total
    d2h = host[0]["out"].numel() * host[0]["out"].element_size()

    R = len(rot)

    def upload(r, hb, sb):
        c = r["cache"]
        sb["buf"].copy_(hb["buf"], non_blocking=True)
        c.kv[:, t].copy_(sb["kv"])
        c.gate[:, t].copy_(sb["gate"])
        c.idx_k[:, t].copy_(sb["idx_k"])
        c.idx_gate[:, t].copy_(sb["idx_gate"])

    # How a serving loop runs the step: per input copy, one CUDA graph uploads the step's inputs
    # from pinned host memory, one runs csa_decode, one reads the output back to pinned host
    # memory, on three streams, so that step i+1's upload and step i-1's read-back overlap step i.
    s_up, s_run, s_down = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    g_up, g_run, g_down = [], [], []
    for r, hb, sb in zip(rot, host, stage):
        upload(r, hb, sb)
        r["e2e_call"]()
        hb["out"].copy_(r["out"], non_blocking=True)
        torch.cuda.synchronize()
        gu, gr, gd = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(gu, stream=s_up):
            upload(r, hb, sb)
        with torch.cuda.graph(gr, stream=s_run):
            r["e2e_call"]()
        with torch.cuda.graph(gd, stream=s_down):
            hb["out"].copy_(r["out"], non_blocking=True)
        g_up.append(gu); g_run.append(gr); g_down.append(gd)
    torch.cuda.synchronize()
    ev_up = [torch.cuda.Event() for _ in range(R)]
    ev_run = [torch.cuda.Event() for _ in range(R)]
    ev_down = [torch.cuda.Event() for _ in range(R)]

    def step(i):
        j = i % R
        if i >= R:
            s_up.wait_event(ev_run[j])        # the previous step on these buffers has read its inputs
            s_run.wait_event(ev_down[j])      # ... and its output has been read back
        with torch.cuda.stream(s_up):
            g_up[j].replay()
        ev_up[j].record(s_up)
        s_run.wait_event(ev_up[j])
        with torch.cuda.stream(s_run):
            g_run[j].replay()
        ev_run[j].record(s_run)
        s_down.wait_event(ev_run[j])
        with torch.cuda.stream(s_down):
            g_down[j].replay()
        ev_down[j].record(s_down)

    for i in range(max(args.warmup, 3)):
        step(i)
    K = args.steps
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(K):
        step(i)
    torch.cuda.synchronize()
    el = time.perf_counter() - t0
    barrier(world)
    el = max_over_ranks(el, world)
    return {"value": job_value(world, B, K, el), "unit": "query-tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": el / K * 1e3,
            "how": "per step: one packed upload from pinned host memory (+ the raw rows placed into the "
                   "caches on the device), csa_decode, read-back to pinned host memory; one CUDA graph "
                   "each on three streams, consecutive steps overlap; wall clock"}


# ----------------------------------------------------------------------------- every decode workload
# the headline decode (B=32, N=65,536) over FP4 E2M1 + FP8 E4M3 caches: the same raw inputs
FP4_DECODE_WL = dataclasses.replace(synth.WORKLOADS[1], name="csa_decode_fp4_B32_N65536_H64_k512", storage="fp4")
# the tiny fp32 decode, HCA B=16 at N=262,144, B=4 at N=1,048,576 (+3), and the FP4 / FP8 cache decode
EXTRA_WORKLOADS = {"0": synth.WORKLOADS[0], "3": synth.WORKLOADS[3], "4": synth.WORKLOADS[4], "1fp4": FP4_DECODE_WL}


def compress_bytes(wl: synth.Workload, B: int) -> int:
    """Algorithmic bytes of a full-cache build: every raw token's rows read once (kv, gate and, for
    CSA, idx_k, idx_gate) and every entry written once."""
    es = 4 if wl.storage == "f32" else 2
    chans = wl.d + (0 if wl.hca else wl.d_idx)
    n = wl.n_entries
    ent = entry_bytes(wl, wl.d) + (0 if wl.hca else entry_bytes(wl, wl.d_idx))
    return B * (n * wl.ratio * chans * 2 * es + n * ent)


def time_graph(call, K: int, W: int) -> float:
    """Milliseconds per replay of a CUDA graph of `call` (W untimed replays first)."""
    import torch
    call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    for _ in range(W):
        g.replay()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(K):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / K


def run_decode_workload(wl: synth.Workload, args, device, peaks) -> dict:
    """One decode step of workload `wl` per step (CUDA graph of csa_decode), plus the full-cache
    compressor build of the same workload and the oracle timed on the host beside it."""
    import torch
    import long_context_sparse_19_b300 as L
    B = wl.B
    cfg = make_cfg(wl)
    T = device_inputs(wl, list(range(B)), device)
    cache = make_cache(T, wl, device)
    calls, keep, graphs = [], [], []
    try:
        # compressor: whole cache, CUDA events (second of two builds)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for rep in range(2):
            torch.cuda.synchronize()
            e0.record()
            L.csa_compress(cfg, cache, 0, wl.n_entries)
            e1.record()
            torch.cuda.synchronize()
        c_ms = e0.elapsed_time(e1)
        c_bytes = compress_bytes(wl, B)
        # decode: rotate over R copies of the compressed caches (and R positions) so that no step
        # reads the previous step's compressed rows from L2 when a step's bytes fit in it
        work = decode_work(wl, B)
        R = 1 if work["bytes"] > 2 * 126e6 or wl.storage == "f32" else 4
        # bind_decode captures raw device pointers: every tensor a call reads or writes stays
        # referenced here for as long as the calls exist
        calls, keep = [], []
        for r in range(R):
            t_r = wl.t - r * 2 * wl.ratio if R > 1 else wl.t
            c = cache if r == 0 else L.Cache(kv=cache.kv, gate=cache.gate, gate_bias=cache.gate_bias,
                                             ckv=cache.ckv.clone(), idx_k=cache.idx_k, idx_gate=cache.idx_gate,
                                             idx_bias=cache.idx_bias,
                                             cidx=None if wl.hca else cache.cidx.clone(), n_cap=cache.n_cap)
            pos = torch.full((B,), t_r, dtype=torch.int64, device=device)
            out = torch.empty(B, wl.H, wl.d, dtype=cache.kv.dtype, device=device)
            ws = L.workspace(cfg, B, 1, wl.n_entries, device=device)
            q = T["q"][:, 0].contiguous()
            qi = None if wl.hca else T["q_idx"][:, 0].contiguous()
            w = None if wl.hca else T["w"][:, 0].contiguous()
            calls.append(L.binding.bind_decode(cfg, pos, c, q, qi, w, T["sink"], out, ws=ws))
            keep.append((c, pos, out, ws, q, qi, w))
        K = max(args.steps, 200)
        if R == 1:
            ms = time_graph(calls[0], K, max(args.warmup, 3))
        else:                                     # one graph per copy, replayed in turn
            graphs = []
            for cl in calls:
                cl()
                torch.cuda.synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    cl()
                graphs.append(g)
            for i in range(max(args.warmup, 3)):
                graphs[i % R].replay()
            torch.cuda.synchronize()
            e0.record()
            for i in range(K):
                graphs[i % R].replay()
            e1.record()
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / K
        assert L.csa_get_device_status() == 0
        step_s = ms / 1e3
        gbs = work["bytes"] / step_s / 1e9
        res = {"workload": wl.name, "B": B, "N": wl.N, "t": wl.t, "ratio": wl.ratio, "top_k": wl.top_k,
               "storage": wl.storage, "value": B / step_s, "unit": "query-tokens/s", "ms_per_step": ms,
               "steps": K, "step_bytes": work["bytes"], "hbm_gbs": gbs, "hbm_frac_of_measured": gbs / peaks["hbm_gbs"],
               "l2": (f"compressed caches rotated over {R} copies and {R} positions" if R > 1 else
                      ("one copy: the step's bytes exceed twice the 126 MB L2" if work["bytes"] > 2 * 126e6
                       else "one copy: the step's 0.7 MB stay in L2 (a launch-bound workload)")),
               "compress": {"ms": c_ms, "bytes": c_bytes, "gbs": c_bytes / c_ms / 1e6,
                            "frac_of_measured": c_bytes / c_ms / 1e6 / peaks["hbm_gbs"],
                            "entries": B * wl.n_entries}}
        if not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline_workload(wl, T, cache, args.cpu_budget_extra)
        return res
    finally:
        torch.cuda.synchronize()
        calls, keep, graphs, T, cache = None, None, None, None, None
        torch.cuda.empty_cache()


def cpu_baseline_workload(wl, T, cache, budget_s: float) -> dict:
    """The oracle's decode step of request 0 on the host, given its caches (copied from the device,
    untimed; the oracle reads only the window of the raw rows, so those alone are copied)."""
    from oracle import csa_oracle as O
    o = O.OracleConfig(H=wl.H, d=wl.d, d_rope=wl.d_rope, H_idx=wl.H_idx, d_idx=wl.d_idx, ratio=wl.ratio,
                       top_k=wl.top_k, window=wl.window)
    t = wl.t
    V = (t + 1) // wl.ratio
    h64 = lambda x: x.detach().float().cpu().numpy().astype(np.float64)
    kv = np.zeros((t + 1, wl.d))                  # left unbacked except the window
    lo = max(0, t - wl.window + 1)
    kv[lo:t + 1] = h64(T["kv"][0, lo:t + 1])
    if wl.storage == "fp4":                      # decoded by the oracle's unpacker (untimed)
        from oracle import cache_lowp as Q
        ckv = Q.unpack_cache(cache.ckv[0].cpu().numpy(), wl.d, wl.n_entries, V)
        cidx = None if wl.hca else Q.unpack_cache(cache.cidx[0].cpu().numpy(), wl.d_idx, wl.n_entries, V)
    else:
        ckv = h64(cache.ckv[0, :V])
        cidx = None if wl.hca else h64(cache.cidx[0, :V])
    q = h64(T["q"][0, 0])
    qi = None if wl.hca else h64(T["q_idx"][0, 0])
    w = None if wl.hca else h64(T["w"][0, 0])
    sink = h64(T["sink"])
    O.decode_step(t, q, qi, w, sink, kv, ckv, cidx, o)          # warm-up
    done, t0 = 0, time.perf_counter()
    while True:
        O.decode_step(t, q, qi, w, sink, kv, ckv, cidx, o)
        done += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    hc = host_cores()
    return {"value": done / el, "unit": "query-tokens/s", "cores": hc["blas_threads"] or hc["affinity_cores"],
            "kind": "oracle", "sample": f"{done} decode steps of request 0 (fp64 NumPy, caches from the device, "
                                        f"untimed), {el:.1f} s"}


# ----------------------------------------------------------------------------- prefill leg
def run_prefill(args, device, peaks) -> dict:
    import torch
    import long_context_sparse_19_b300 as L
    wl = PREFILL_WL
    cfg = make_cfg(wl)
    T = device_inputs(wl, list(range(wl.B)), device)
    cache = make_cache(T, wl, device)
    out = torch.empty(wl.B, wl.S, wl.H, wl.d, dtype=cache.kv.dtype, device=device)
    ws = L.workspace(cfg, wl.B, wl.S, wl.n_entries, device=device)

    def call():
        L.csa_prefill(cfg, cache, T["q"], T["q_idx"], T["w"], T["sink"], out, ws=ws)

    for _ in range(2):
        call()
    torch.cuda.synchronize()
    reps = args.prefill_reps
    L.csa_profile_begin(reps * 8 + 8)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        call()
    e1.record()
    torch.cuda.synchronize()
    prof = L.csa_profile_end()
    assert L.csa_get_device_status() == 0
    ms = e0.elapsed_time(e1) / reps
    fl = prefill_flops(wl)
    pk = peaks["bf16_tflops"]
    idx_ms = prof["index"][0] / reps
    attn_ms = prof["attn"][0] / reps
    return {"workload": wl.name, "ms": ms, "tflops": fl["total"] / ms / 1e9, "flops": fl["total"],
            "index": {"ms": idx_ms, "tflops": fl["index"] / idx_ms / 1e9 if idx_ms else None,
                      "frac_of_bf16_peak": fl["index"] / idx_ms / 1e9 / pk if idx_ms else None},
            "attn": {"ms": attn_ms, "tflops": fl["attn"] / attn_ms / 1e9 if attn_ms else None,
                     "frac_of_bf16_peak": fl["attn"] / attn_ms / 1e9 / pk if attn_ms else None},
            "stages_ms": {k: round(v[0] / reps, 4) for k, v in prof.items()},
            "peak_tflops": pk, "peak_source": peaks["source"]}


# ----------------------------------------------------------------------------- the oracle on the host
def oracle_setup(wl, requests):
    """fp64 caches of the sampled requests, built by the oracle itself (not timed)."""
    from oracle import csa_oracle as O
    sh = synth.gen_shared(wl)
    o = O.OracleConfig(H=wl.H, d=wl.d, d_rope=wl.d_rope, H_idx=wl.H_idx, d_idx=wl.d_idx, ratio=wl.ratio,
                       top_k=wl.top_k, window=wl.window)
    items = []
    for b in requests:
        r = synth.gen_request(wl, b)
        n = wl.n_entries
        ckv = O.compress(r["kv"], r["gate"], sh["bias"], wl.ratio, n)
        cidx = None if wl.hca else O.compress(r["idx_k"], r["idx_gate"], sh["idx_bias"], wl.ratio, n)
        items.append((r, ckv, cidx))
    return o, sh, items


def oracle_step(o, sh, item, t):
    """One decode step of one request in the oracle: compress-on-close of entry t//m, then
    indexer, top-k and sparse attention."""
    from oracle import csa_oracle as O
    r, ckv, cidx = item
    m = o.ratio
    if (t + 1) % m == 0:
        e = t // m
        lo, hi = (e - 1) * m, (e + 1) * m
        for src, g, bias, cache in ((r["kv"], r["gate"], sh["bias"], ckv),
                                    (r["idx_k"], r["idx_gate"], sh["idx_bias"], cidx)):
            if cache is None:
                continue
            x = O.pool_window(src[lo:hi], g[lo:hi], bias)
            cache[e] = O.rope(O.rms_norm(x, o.rms_eps), e * m, o.d_rope, o.rope_base)
    return O.decode_step(t, r["q"][0], None if o.hca else r["q_idx"][0], None if o.hca else r["w"][0],
                         sh["sink"], r["kv"], ckv, cidx, o)


def host_cores() -> dict:
    info = {"affinity_cores": len(os.sched_getaffinity(0))}
    try:
        from threadpoolctl import threadpool_info
        info["blas_threads"] = max((p.get("num_threads", 1) for p in threadpool_info()), default=1)
    except Exception:
        info["blas_threads"] = None
    return info


def run_cpu_baseline(budget_s: float, n_req: int = 2) -> dict:
    wl = DECODE_WL
    o, sh, items = oracle_setup(wl, list(range(n_req)))
    oracle_step(o, sh, items[0], wl.t)                    # warm-up
    done, t0 = 0, time.perf_counter()
    while True:
        oracle_step(o, sh, items[done % n_req], wl.t)
        done += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    hc = host_cores()
    return {"value": done / el, "unit": "query-tokens/s", "cores": hc["blas_threads"] or hc["affinity_cores"],
            "kind": "oracle", "host": hc,
            "sample": f"{done} single-request decode steps (requests 0..{n_req - 1} of the B=32, N=65,536 "
                      f"workload, fp64 NumPy; caches prebuilt untimed), {el:.1f} s; matmuls use the BLAS "
                      f"threads, element-wise NumPy one thread"}


def run_reference(args, world, rank) -> None:
    if rank != 0:
        return
    wl = DECODE_WL
    n_req = 2
    o, sh, items = oracle_setup(wl, list(range(n_req)))
    for i in range(args.warmup):
        oracle_step(o, sh, items[i % n_req], wl.t)
    t0 = time.perf_counter()
    for i in range(args.steps):
        oracle_step(o, sh, items[i % n_req], wl.t)
    el = time.perf_counter() - t0
    hc = host_cores()
    v = args.steps / el
    line = {"metric": METRIC, "impl": "reference", "value": v, "unit": "query-tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": dict(decode_config(world), timing="host wall clock around the oracle's decode steps",
                           l2="not applicable (host)"),
            "cpu_baseline": {"value": v, "unit": "query-tokens/s", "kind": "oracle",
                             "cores": hc["blas_threads"] or hc["affinity_cores"],
                             "sample": f"each step = one request's decode step (requests 0..{n_req - 1} of the "
                                       f"workload), fp64 NumPy oracle on the host; caches prebuilt untimed"},
            "e2e": {"value": v, "unit": "query-tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


METRIC = "CSA decode query-tokens/s (N=65,536, B=32, H=64, top-k 512, W=128, bf16)"


def headline_wl(args=None) -> synth.Workload:
    """The decode workload of the headline leg (B=32, N=65,536; --B and --storage change it)."""
    wl = FP4_DECODE_WL if args is not None and getattr(args, "storage", "bf16") == "fp4" else DECODE_WL
    return dataclasses.replace(wl, B=args.B) if args is not None and args.B else wl


def decode_config(world, args=None) -> dict:
    wl = headline_wl(args)
    R = args.rotations if args else ROTATIONS
    B = args.B if args and args.B else wl.B
    return {"workload": wl.name, "B_per_gpu": B, "N": wl.N, "t": wl.t, "H": wl.H, "H_idx": wl.H_idx,
            "top_k": wl.top_k, "window": wl.window, "ratio": wl.ratio, "parallelism": f"requests x{world}",
            "l2": f"inputs rotated over {R} device copies (~{R * 153 * B // 32} MB touched per cycle; "
                  f"L2 is 126 MB)", "timing": "CUDA graph of one csa_decode call per step, CUDA events"}


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: 5000 for the GPU arm, 100 for the reference arm, whose "
                         "step is a fp64 host decode step of about 50 ms)")
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--prefill-reps", type=int, default=3)
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--cpu-budget-extra", type=float, default=3.0,
                    help="seconds of oracle work beside each of the other decode workloads")
    ap.add_argument("--no-workloads", action="store_true", help="skip the other decode workloads")
    ap.add_argument("--workload", default=None, choices=("0", "1", "3", "4", "1fp4"),
                    help="run only this decode workload's leg (with --wl-B / --wl-N to reduce it) and print it "
                         "(1fp4: the headline decode over FP4 / FP8 caches)")
    ap.add_argument("--wl-B", type=int, default=0, help="requests of the --workload leg (default: the workload's)")
    ap.add_argument("--wl-N", type=int, default=0,
                    help="raw tokens per request of the --workload leg (default: the workload's; the query "
                         "sits at the last token)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--B", type=int, default=0, help="requests per GPU (default: the workload's 32)")
    ap.add_argument("--rotations", type=int, default=ROTATIONS, help="device input copies cycled between steps")
    ap.add_argument("--storage", choices=("bf16", "fp4"), default="bf16",
                    help="compressed-cache storage of the headline decode leg (fp4: FP4 E2M1 + FP8 E4M3)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.steps is None:
        args.steps = 100 if args.impl == "reference" else 5000

    if args.impl == "reference":
        world = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        run_reference(args, world, rank)
        return

    import torch
    world, rank, local = dist_setup()
    device = torch.device("cuda", torch.cuda.current_device())
    peaks = load_peaks()
    if args.workload is not None:                 # one decode workload, possibly reduced
        wl = FP4_DECODE_WL if args.workload == "1fp4" else synth.WORKLOADS[int(args.workload)]
        kw = {}
        if args.wl_B:
            kw["B"] = args.wl_B
        if args.wl_N:
            kw.update(N=args.wl_N, t=args.wl_N - 1)
        wl = dataclasses.replace(wl, **kw)
        print(json.dumps(run_decode_workload(wl, args, device, peaks)), flush=True)
        return
    # the host-side oracle baseline runs first (rank 0, N = 1), before the GPU is busy
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = run_cpu_baseline(args.cpu_budget)
    dec = run_decode(args, world, rank, device, peaks)
    pre = None if args.no_prefill else run_prefill(args, device, peaks)
    extra = None
    if rank == 0 and not args.no_workloads:
        extra = {w.name: run_decode_workload(w, args, device, peaks) for w in EXTRA_WORKLOADS.values()}
    if rank == 0:
        line = {"metric": METRIC, "value": dec["value"], "unit": "query-tokens/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": dec["ms_per_step"],
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                "data": "synthetic", "config": decode_config(world, args),
                "hbm_gbs": dec["hbm_gbs"], "hbm_frac_of_measured": dec["hbm_frac_of_measured"],
                "roofline": dec["roofline"], "cpu_baseline": cpu, "e2e": dec["e2e"],
                "gpu_launches": dec["gpu_launches"], "clocks": dec["clocks"],
                "detail": {k: dec[k] for k in ("step_bytes", "step_flops", "stage_sum_ms_per_step",
                                               "stages_ms_per_step", "stage_launches", "setup_s")},
                "prefill": pre, "workloads": extra}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
