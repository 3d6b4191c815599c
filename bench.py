#!/usr/bin/env python3
"""Benchmark of the W4A16 group-64 skinny GEMM on GB300.

One step = one w4a16_mm call of the tied LM head 262144x2560 at M = 1: the
largest single-GPU configuration of the workload set, streaming 377.5 MB of
packed weights, scales and biases.  The metric is achieved HBM GB/s over the
algorithmic bytes (codes + scales + biases + activations + outputs, read or
written once; tiny-llm "Week 2 Day 2: Keep W4 Packed", section "Revisit the
Decode Roofline") and its fraction of the measured GB300 copy bandwidth.

Timing: the weights are replicated into enough copies that one pass over
them is > 3x the L2 size, and step s uses copy s mod L, so every step streams
its weights from HBM (no L2 flush needed).  The timed region is K eager
back-to-back calls on one stream between CUDA events (queued behind a short
spin so the host never starves the GPU), bracketed by a barrier and a
synchronize; consecutive calls overlap by programmatic dependent launch, as
they do in a decode loop.  The line also reports the single-call cold
latency: the median of isolated calls, each after a write of twice the L2
size and bracketed by its own events.  SM clocks are sampled with nvidia-smi
around a load phase and the timed region.  The decode-layer projection set
and the other configurations are context numbers under "extras".

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
Under torchrun (N > 1) every rank runs its own independent replica (weak
scaling, no collective on the data path); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
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
sys.path.insert(0, ROOT)

METRIC = "achieved HBM GB/s and % of GB300 peak for W4A16 GEMV/skinny-GEMM (M=1..k+1)"
UNIT = "GB/s"
HEAD_N, HEAD_K = 262144, 2560
WORKLOAD = "W4A16 g64 tied LM head 262144x2560 at M=1 (w4a16_mm; 377.5 MB of packed weights, scales and biases)"
CONFIG = {"workload": WORKLOAD, "M": 1, "N": HEAD_N, "K": HEAD_K, "group_size": 64}
DECODE_LAYER = [("q", 2048, 2560), ("k", 512, 2560), ("v", 512, 2560), ("o", 2560, 2048),
                ("gate", 10240, 2560), ("up", 10240, 2560), ("down", 2560, 10240)]
# The launches of one decode-layer step (an extra).  A decoder layer's q/k/v
# projections are independent given their input, as are gate/up; they go
# through one w4a16_mm_group call each.  o and down depend on earlier results
# (attention, the gated activation) and run as their own w4a16_mm calls.
LAUNCHES = [("qkv", ("q", "k", "v")), ("o", ("o",)), ("gate_up", ("gate", "up")), ("down", ("down",))]
# Single workloads for --case: name -> (N, K, E)
CASES = {"q": (2048, 2560, 1), "kv": (512, 2560, 1), "o": (2560, 2048, 1), "gate": (10240, 2560, 1),
         "down": (2560, 10240, 1), "wide_up": (12288, 1536, 1), "wide_down": (1536, 12288, 1),
         "lm_head_1536": (262144, 1536, 1), "lm_head_2560": (262144, 2560, 1), "dense_16384": (16384, 16384, 1),
         "routed": (6144, 2048, 8), "tail_k_gate": (9216, 2304, 1), "tail_k_q": (2048, 2304, 1), "tail_k_head": (256000, 2304, 1),
         "stq1_16384": (16384, 16384, 1), "stq1_expert": (6144, 2048, 1), "stq1_routed": (6144, 2048, 8)}
FALLBACK_HBM_GBS = 6800.0
DOMINANT_KERNEL = "tc_stream_kernel"  # the persistent grid runs every step (the only kernel)
NOMINAL_HBM_GBS = 8000.0


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--kernel", default="auto", help="auto | simt | tc | vanilla")
    ap.add_argument("--no-extras", action="store_true", help="skip the per-config context measurements")
    ap.add_argument("--no-workspace", action="store_true",
                    help="run the calls through w4a16_mm without a workspace (w4a16_mm_ws otherwise)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="CPU work budget of the oracle baseline")
    ap.add_argument("--case", default=None,
                    help="time one workload alone instead of the step: " + ", ".join(sorted(CASES)) +
                         " (with --M; eager launches over rotating cold copies; handy under ncu)")
    ap.add_argument("--M", type=int, default=1, help="activation rows for --case")
    return ap.parse_args()


# ---- distributed plumbing ---------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend=None):
    """The process group of a torchrun launch (None for one process): NCCL on
    GPUs, gloo where there is none (the CPU tests of the multi-rank path)."""
    if world <= 1:
        return None
    import torch
    import torch.distributed as dist
    if backend is None:
        backend = "nccl" if torch.cuda.is_available() else "gloo"
    dist.init_process_group(backend=backend)
    return dist


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, v: float) -> float:
    if dist is None:
        return v
    import torch
    device = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_gbps(world: int, step_bytes: int, steps: int, ms_max: float) -> float:
    """Whole-job throughput: the bytes every rank streamed over the slowest
    rank's time (each rank runs its own replica of the step)."""
    return world * step_bytes * steps / (ms_max * 1e-3) / 1e9


# ---- peaks, clocks, ncu traffic ----------------------------------------------------

def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampler running during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_id: str | None):
        self.device_id = device_id
        self.proc = None
        self.lines: list[str] = []

    def __enter__(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
        if self.device_id:
            cmd += ["-i", self.device_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# The translation unit of the dominant kernel and the headers it includes.
DOMINANT_SOURCES = ("common.cuh", "launch.h", "route.cuh", "tc.cu")


def kernel_source_sha() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "skinny_gemm_gb300", "csrc")
    for name in DOMINANT_SOURCES:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str):
    """Per-launch DRAM bytes (read + write) of `kernel` on the bench workload,
    from the committed ncu summary (profiles/traffic.txt: one line per kernel,
    `name source_sha bytes_per_launch`), or None when that capture predates
    the current kernel sources."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    try:
        with open(path) as f:
            for line in f:
                parts = line.split()
                if len(parts) >= 3 and parts[0] == kernel and not line.startswith("#"):
                    return int(parts[2]) if parts[1] == kernel_source_sha() else None
    except OSError:
        return None
    return None


# ---- workload -------------------------------------------------------------------------

def layer_bytes(M=1):
    from skinny_gemm_gb300 import roofline
    return sum(roofline.mm_bytes(M, N, K) for _, N, K in DECODE_LAYER)


def build_layers(torch, ops, synth, copies: int, seed: int):
    """`copies` device copies of one seeded decode layer, plus inputs and outputs."""
    host = {name: synth.make_weights(seed + i, N, K) for i, (name, N, K) in enumerate(DECODE_LAYER)}
    base = {name: ops.W4Matrix.from_host(hw) for name, hw in host.items()}
    layers = [base]
    for _ in range(copies - 1):
        layers.append({n: ops.W4Matrix(w.Wq.clone(), w.scales.clone(), w.biases.clone(), w.N, w.K)
                       for n, w in base.items()})
    xs = {name: torch.from_numpy(synth.make_x(seed + 100 + i, 1, K).view(np.int16)).view(torch.bfloat16).cuda()
          for i, (name, N, K) in enumerate(DECODE_LAYER)}
    ys = {name: torch.empty(1, N, dtype=torch.bfloat16, device="cuda") for name, N, K in DECODE_LAYER}
    return layers, xs, ys


def measure_decode_layer(torch, ops, synth, roofline, l2, steps, warmup, peak):
    """The decode-layer projection set at M = 1 as four launches (qkv group,
    o, gate/up group, down) replayed as CUDA graphs over rotating layer
    copies; plus the same layer as seven w4a16_mm calls."""
    step_bytes = layer_bytes(1)
    weight_bytes = sum(roofline.weight_bytes(N, K) for _, N, K in DECODE_LAYER)
    copies = max(2, math.ceil(3 * l2 / weight_bytes))
    layers, xs, ys = build_layers(torch, ops, synth, copies, seed=0)
    stream = torch.cuda.Stream()
    dims = {name: (N, K) for name, N, K in DECODE_LAYER}

    def enqueue_layer(layer, launches):
        for _, names in launches:
            if len(names) == 1:
                ops.mm(xs[names[0]], layer[names[0]], out=ys[names[0]])
            else:
                ops.mm_group([xs[n] for n in names], [layer[n] for n in names], [ys[n] for n in names])

    out = {"matrices": [f"{n} {N}x{K}" for n, N, K in DECODE_LAYER], "bytes_per_step": step_bytes,
           "weight_copies": copies}
    for label, launches in (("grouped", LAUNCHES), ("ungrouped", [(n, (n,)) for n, _, _ in DECODE_LAYER])):
        graphs = []
        with torch.cuda.stream(stream):
            for layer in layers:
                enqueue_layer(layer, launches)
            torch.cuda.synchronize()
            for layer in layers:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    enqueue_layer(layer, launches)
                graphs.append(g)
            for s_ in range(warmup):
                graphs[s_ % len(graphs)].replay()
        torch.cuda.synchronize()
        a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n = max(1, min(steps, 5000))
        with torch.cuda.stream(stream):
            a_.record()
            for s_ in range(n):
                graphs[s_ % len(graphs)].replay()
            b_.record()
        torch.cuda.synchronize()
        ms = a_.elapsed_time(b_) / n
        gb = step_bytes / (ms * 1e-3) / 1e9
        out[label] = {"launches_per_step": len(launches), "us_per_step": round(1e3 * ms, 3), "GBps": round(gb, 1),
                      "frac": round(gb / peak, 4),
                      "launches": [("w4a16_mm_group" if len(nm) > 1 else "w4a16_mm") + f"({', '.join(nm)})"
                                   for _, nm in launches]}
        del graphs
    del layers
    return out


def head_copies(torch, ops, synth, roofline, l2, seed):
    """Rotating device copies of the seeded LM head (> 3x L2 in total)."""
    hw = synth.make_weights(seed, HEAD_N, HEAD_K)
    base = ops.W4Matrix.from_host(hw)
    copies = max(2, math.ceil(3 * l2 / roofline.weight_bytes(HEAD_N, HEAD_K)))
    ws = [base] + [ops.W4Matrix(base.Wq.clone(), base.scales.clone(), base.biases.clone(), HEAD_N, HEAD_K)
                   for _ in range(copies - 1)]
    torch.cuda.synchronize()  # the weights are written before any call reads them (overlapped launches)
    return hw, ws


def run_ours(args, world, rank, local):
    import torch
    from skinny_gemm_gb300 import ops, roofline, synth

    torch.cuda.set_device(local)
    dist = init_dist(world)
    props = torch.cuda.get_device_properties(local)
    l2 = int(getattr(props, "L2_cache_size", 126 * 2**20))
    N, K = HEAD_N, HEAD_K
    step_bytes = roofline.mm_bytes(1, N, K)
    wsel = None if args.no_workspace else "auto"
    hw, ws = head_copies(torch, ops, synth, roofline, l2, seed=1000 * rank + 1)
    copies = len(ws)
    x = torch.from_numpy(synth.make_x(1000 * rank + 2, 1, K).view(np.int16)).view(torch.bfloat16).cuda()
    y = torch.empty(1, N, dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.Stream()
    plan = ops.get_plan(N, K)

    def call(s_):
        ops.mm(x, ws[s_ % copies], out=y, workspace=wsel)

    with torch.cuda.stream(stream):
        for s_ in range(max(3, args.warmup)):
            call(s_)
    torch.cuda.synchronize()

    device_id = getattr(props, "uuid", None)
    device_id = f"GPU-{device_id}" if device_id is not None and not str(device_id).startswith("GPU-") else device_id
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(str(device_id) if device_id else None)
    with sampler:
        # untimed load phase of about half a second, so the clock samples are taken under load
        with torch.cuda.stream(stream):
            t0 = time.perf_counter()
            i = 0
            while time.perf_counter() - t0 < 0.5:
                for _ in range(64):
                    call(i)
                    i += 1
                torch.cuda.current_stream().synchronize()
        barrier(dist)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            torch.cuda._sleep(20_000_000)  # the host queues the calls while the GPU spins
            t_start.record()
            for s_ in range(args.steps):
                call(s_)
            t_end.record()
        torch.cuda.synchronize()
        barrier(dist)
    ms_total = max_over_ranks(dist, t_start.elapsed_time(t_end))
    ms_per_step = ms_total / args.steps
    value = aggregate_gbps(world, step_bytes, args.steps, ms_total)
    peak, peak_kind = measured_peak()
    launch_us = 1e3 * ms_per_step  # one launch per step
    achieved = step_bytes / (launch_us * 1e-6) / 1e9

    cold = single_call_cold(torch, lambda i: call(i), stream, l2, reps=60)
    e2e = measure_e2e(torch, ops, ws, args.steps, step_bytes, world, dist, wsel)
    extras = None if args.no_extras else measure_extras(torch, ops, synth, roofline, l2, peak, args)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args.cpu_seconds, hw)

    if rank == 0:
        clocks = sampler.summary()
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_per_step, 6), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "accumulate": "f32", "data": "synthetic",
            "config": dict(CONFIG),
            "setup": {"api": "w4a16_mm_ws (the binding's per-stream workspace)" if wsel else "w4a16_mm (no workspace)",
                      "plan": plan, "parallelism": f"replicas x{world}",
                      "l2_policy": f"inputs larger than L2: {copies} rotating weight copies "
                                   f"({copies * roofline.weight_bytes(N, K) / 1e6:.0f} MB > 3x L2 {l2 / 1e6:.0f} MB)",
                      "launch": "eager back-to-back calls on one stream, programmatic dependent launch"},
            "roofline": {"bound": "hbm", "kernel": DOMINANT_KERNEL, "achieved": round(achieved, 1), "peak": peak,
                         "unit": "GB/s", "frac": round(achieved / peak, 4),
                         "traffic": ncu_traffic(DOMINANT_KERNEL),
                         "algorithmic_bytes_per_launch": step_bytes,
                         "launch_us": round(launch_us, 3),
                         "peak_kind": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
                         if peak_kind == "measured" else "fallback 6.8 TB/s",
                         "frac_of_nominal_8TBps": round(achieved / NOMINAL_HBM_GBS, 4),
                         "launches_timed": args.steps,
                         "timing": "CUDA events around the timed region on the launching stream; "
                                   "average launch = region / launches (one launch per step)"},
            "single_call_cold": cold,
            "e2e": e2e,
            "gpu_launches": args.steps,
            "clocks": clocks,
        }
        if cpu is not None:
            line["cpu_baseline"] = cpu
        if extras is not None:
            line["extras"] = extras
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def single_call_cold(torch, call, stream, l2, reps=60):
    """Median latency of isolated calls: before each, a write of twice the L2
    size (the previous call's lines are gone and no kernel of ours runs
    before it), then events around the call alone."""
    from skinny_gemm_gb300 import roofline
    flush = torch.empty(2 * l2, dtype=torch.uint8, device="cuda")
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    with torch.cuda.stream(stream):
        for i, (a, b) in enumerate(evs):
            flush.fill_(i & 0xFF)
            a.record()
            call(i)
            b.record()
    torch.cuda.synchronize()
    us = sorted(1e3 * a.elapsed_time(b) for a, b in evs)
    med = statistics.median(us)
    nb = roofline.mm_bytes(1, HEAD_N, HEAD_K)
    peak, _ = measured_peak()
    del flush
    return {"us_median": round(med, 3), "us_min": round(us[0], 3), "us_max": round(us[-1], 3), "calls": reps,
            "GBps": round(nb / (med * 1e-6) / 1e9, 1), "frac": round(nb / (med * 1e-6) / 1e9 / peak, 4),
            "method": f"fill of {2 * l2 / 1e6:.0f} MB (2x L2) before each call, events around the call alone"}


def measure_e2e(torch, ops, ws, steps, step_bytes, world, dist, wsel):
    """Through the public API with HOST buffers, every step: pinned host ->
    device copy of the activation row, one LM-head call, device -> pinned
    host copy of the 262144 logits, and the synchronisation that read
    implies."""
    K, N = HEAD_K, HEAD_N
    h_in = torch.empty(1, K, dtype=torch.bfloat16, pin_memory=True)
    h_out = torch.empty(1, N, dtype=torch.bfloat16, pin_memory=True)
    h_in.copy_(torch.randn(1, K).to(torch.bfloat16))
    d_in = torch.empty(1, K, dtype=torch.bfloat16, device="cuda")
    d_out = torch.empty(1, N, dtype=torch.bfloat16, device="cuda")
    n = max(1, min(steps, 2000))

    def step(s_):
        d_in.copy_(h_in, non_blocking=True)
        ops.mm(d_in, ws[s_ % len(ws)], out=d_out, workspace=wsel)
        h_out.copy_(d_out, non_blocking=True)
        torch.cuda.current_stream().synchronize()

    for s_ in range(min(20, n)):
        step(s_)
    barrier(dist)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for s_ in range(n):
        step(s_)
    dt = max_over_ranks(dist, time.perf_counter() - t0)
    return {"value": round(world * step_bytes * n / dt / 1e9, 2), "unit": UNIT,
            "h2d_bytes_per_step": int(h_in.numel() * 2), "d2h_bytes_per_step": int(h_out.numel() * 2),
            "steps": n, "ms_per_step": round(1e3 * dt / n, 4),
            "api": "skinny_gemm_gb300.ops.mm (eager, the C ABI through ctypes) with host copies"}


def time_graph_launches(torch, fn_list, reps, min_calls=32):
    """Average time per call: fn_list (one call each), repeated to at least
    min_calls calls, captured in one graph and replayed reps times.  The
    repetition keeps the replay boundary (where a launch cannot overlap the
    previous one) rare, as it is in a decode loop."""
    rounds = max(1, -(-min_calls // len(fn_list)))
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for fn in fn_list:
            fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(rounds):
            for fn in fn_list:
                fn()
    with torch.cuda.stream(stream):
        for _ in range(3):
            g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        a.record()
        for _ in range(reps):
            g.replay()
        b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / (reps * rounds * len(fn_list))  # ms per call


def measure_extras(torch, ops, synth, roofline, l2, peak, args):
    """Context numbers on the other workloads (M = 1..8), cold weights; each
    timed as CUDA-graph replays of at least 32 calls over rotating copies."""
    out = {}

    def cold_set(N, K, seed):
        wb = roofline.weight_bytes(N, K)
        copies = max(1, math.ceil(3 * l2 / wb))
        hw = synth.make_weights(seed, N, K)
        base = ops.W4Matrix.from_host(hw)
        ws = [base] + [ops.W4Matrix(base.Wq.clone(), base.scales.clone(), base.biases.clone(), N, K)
                       for _ in range(copies - 1)]
        torch.cuda.synchronize()
        return ws

    def timed(ws, M, N, K, reps, **kw):
        x = torch.randn(M, K, device="cuda").to(torch.bfloat16)
        y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        ms = time_graph_launches(torch, [lambda w=w: ops.mm(x, w, out=y, **kw) for w in ws], reps)
        g = roofline.mm_bytes(M, N, K) / (ms * 1e-3) / 1e9
        return {"us": round(1e3 * ms, 3), "GBps": round(g, 1), "frac": round(g / peak, 4)}

    out["decode_layer"] = measure_decode_layer(torch, ops, synth, roofline, l2, min(args.steps, 2000),
                                               max(3, min(args.warmup, 50)), peak)
    verify = {}
    for (N, K) in [(10240, 2560), (2560, 10240), (12288, 1536), (1536, 12288)]:
        ws = cold_set(N, K, 7)
        t = {M: timed(ws, M, N, K, 20) for M in (1, 3, 5, 7)}
        verify[f"{N}x{K}"] = {f"M{M}_us": t[M]["us"] for M in t}
        verify[f"{N}x{K}"].update({f"M{M}_GBps": t[M]["GBps"] for M in t})
        verify[f"{N}x{K}"]["t5_over_t1"] = round(t[5]["us"] / t[1]["us"], 3)
        del ws
    out["verify"] = verify
    lm, lm_argmax = {}, {}
    for (N, K) in [(262144, 1536), (262144, 2560)]:
        ws = cold_set(N, K, 8)
        for M in (1, 3):
            lm[f"{N}x{K}_M{M}"] = timed(ws, M, N, K, 10)
        lm[f"{N}x{K}_M1_no_workspace"] = timed(ws, 1, N, K, 10, workspace=None)
        # greedy head: w4a16_mm_argmax against w4a16_mm followed by torch.argmax over the logits
        for M in (1, 3):
            x = torch.randn(M, K, device="cuda").to(torch.bfloat16)
            y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
            idx = torch.empty(M, dtype=torch.int32, device="cuda")
            val = torch.empty(M, dtype=torch.bfloat16, device="cuda")
            fused = [lambda w=w: ops.mm_argmax(x, w, idx=idx, val=val) for w in ws]
            unfused = [lambda w=w: (ops.mm(x, w, out=y), torch.argmax(y, dim=-1)) for w in ws]
            ms_f = time_graph_launches(torch, fused, 10)
            ms_u = time_graph_launches(torch, unfused, 10)
            g = (roofline.mm_bytes(M, N, K) - 2 * M * N + 6 * M) / (ms_f * 1e-3) / 1e9  # no logits, idx + val out
            lm_argmax[f"{N}x{K}_M{M}"] = {"us": round(1e3 * ms_f, 2), "GBps": round(g, 1), "frac": round(g / peak, 4),
                                          "mm_then_torch_argmax_us": round(1e3 * ms_u, 2)}
        if K == 2560:  # the tied table as embeddings: a decode step's rows and a prefill's
            emb = {}
            for T in (8, 4096):
                ids = torch.from_numpy(synth.make_ids(1, T, N)).cuda()
                e_out = torch.empty(T, K, dtype=torch.bfloat16, device="cuda")
                ms_e = time_graph_launches(torch, [lambda w=w: ops.embed(ids, w, out=e_out) for w in ws], 10)
                nb = T * K * (0.5 + 4 / 64) + T * K * 2 + 4 * T
                emb[f"T{T}"] = {"us": round(1e3 * ms_e, 3), "GBps": round(nb / (ms_e * 1e-3) / 1e9, 1),
                                "frac": round(nb / (ms_e * 1e-3) / 1e9 / peak, 4)}
            out["embed_262144x2560"] = emb
        del ws
    out["lm_head"] = lm
    out["lm_head_argmax"] = lm_argmax
    dense = {}
    ws = cold_set(16384, 16384, 9)
    for M in (1, 2, 4, 8):
        dense[f"M{M}"] = timed(ws, M, 16384, 16384, 10)
    dense["M1_no_workspace"] = timed(ws, 1, 16384, 16384, 10, workspace=None)
    del ws
    out["dense_16384"] = dense
    # routed experts: 8 x 6144x2048, 8 tokens, ids uniform on 0..7 (seed 0)
    E, N, K, T = 8, 6144, 2048, 8
    hw = synth.make_weights(0, N, K, E)
    base = ops.W4Matrix.from_host(hw)
    copies = max(1, math.ceil(3 * l2 / base.nbytes))
    ws = [base] + [ops.W4Matrix(base.Wq.clone(), base.scales.clone(), base.biases.clone(), N, K, E)
                   for _ in range(copies - 1)]
    ids_np = synth.make_ids(0, T, E)
    ids = torch.from_numpy(ids_np).cuda()
    x = torch.randn(T, K, device="cuda").to(torch.bfloat16)
    y = torch.empty(T, N, dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    ms = time_graph_launches(torch, [lambda w=w: ops.mm_id(x, w, ids, out=y) for w in ws], 20)
    nb, touched = roofline.mm_id_bytes(ids_np, T, N, K, E)
    # bytes read on speculation before the ids are known: the first 512-code
    # stage of every expert, of which the untouched experts' are never used
    spec = E * N * (512 // 2 + 512 // 64 * 4)
    out["routed"] = {"experts_touched": touched, "bytes": nb, "us": round(1e3 * ms, 2),
                     "GBps": round(nb / (ms * 1e-3) / 1e9, 1), "frac": round(nb / (ms * 1e-3) / 1e9 / peak, 4),
                     "l2_prefetch_bytes": spec, "l2_prefetch_wasted_bytes": (E - touched) * N * (512 // 2 + 512 // 64 * 4)}
    del ws
    # K % 512 != 0 (a hidden-2304 gate 9216x2304 and a 256000x2304 LM head), M = 1 and 5: the
    # tensor-core kernels on K padded to whole stages (the default) against the CUDA-core family
    tail = {}
    for (N, K) in [(9216, 2304), (256000, 2304)]:
        ws = cold_set(N, K, 10)
        t1, t5 = timed(ws, 1, N, K, 20), timed(ws, 5, N, K, 20)
        s1, s5 = timed(ws, 1, N, K, 20, kernel="simt"), timed(ws, 5, N, K, 20, kernel="simt")
        tail[f"{N}x{K}"] = {"kernel": ops.get_plan(N, K)["kernel"], "M1": t1, "M5": t5,
                            "t5_over_t1": round(t5["us"] / t1["us"], 3), "simt_M1": s1, "simt_M5": s5}
        del ws
    out["tail_k"] = tail
    # group-128 tables on the 262144x2560 head: read natively (0.53125 B per
    # weight) against their expansion to group 64 (0.5625 B per weight)
    N, K = 262144, 2560
    hw = synth.make_weights(12, N, K)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()  # noqa: E731
    s128, b128 = dev(hw.scales[:, ::2]), dev(hw.biases[:, ::2])
    nat = ops.W4Matrix(torch.from_numpy(hw.Wq.view(np.int32)).cuda(), s128, b128, N, K, group=128)
    copies = max(2, math.ceil(3 * l2 / (N * K * 0.53125)))
    nats = [nat] + [ops.W4Matrix(nat.Wq.clone(), s128.clone(), b128.clone(), N, K, group=128)
                    for _ in range(copies - 1)]
    exps = [ops.W4Matrix.from_group(w.Wq, w.scales, w.biases, N, K, 128) for w in nats]
    torch.cuda.synchronize()
    g128 = {}
    for M in (1, 3):
        nb_nat = N * K // 2 + 4 * N * (K // 128) + 2 * M * K + 2 * M * N
        tn, te = timed(nats, M, N, K, 10), timed(exps, M, N, K, 10)
        g = nb_nat / (tn["us"] * 1e-6) / 1e9
        g128[f"{N}x{K}_M{M}"] = {"native_us": tn["us"], "native_GBps": round(g, 1), "native_frac": round(g / peak, 4),
                                 "native_bytes": nb_nat, "expanded_to_g64_us": te["us"],
                                 "expanded_bytes": roofline.mm_bytes(M, N, K)}
    del nats, exps
    out["group128"] = g128
    # many activation rows: the tcgen05 prefill kernel (the default above 32
    # rows) against the skinny tile kernel taking them eight at a time
    pre = {}
    for (N, K) in [(10240, 2560), (12288, 1536)]:
        ws = cold_set(N, K, 11)
        t = {M: timed(ws, M, N, K, 10) for M in (1, 8, 16, 32, 64, 128, 256)}
        row = {f"M{M}_us": t[M]["us"] for M in t}
        row.update({f"t{M}_over_t1": round(t[M]["us"] / t[1]["us"], 3) for M in (16, 32, 64, 128, 256)})
        flops = {M: 2.0 * M * N * K / (t[M]["us"] * 1e-6) / 1e12 for M in (64, 128, 256)}
        row.update({f"M{M}_TFLOPs": round(v, 1) for M, v in flops.items()})
        for M in (16, 32):  # below the switch: the prefill kernel selected explicitly
            row[f"M{M}_prefill_kernel_us"] = timed(ws, M, N, K, 10, kernel="tc_prefill")["us"]
        for M in (64, 128):  # above it: the skinny tile kernel, eight rows at a time
            row[f"M{M}_tile_kernel_us"] = timed(ws, M, N, K, 10, kernel="tc_tile")["us"]
        pre[f"{N}x{K}"] = row
        del ws
    out["prefill"] = pre
    out["stq1"] = measure_stq1(torch, ops, synth, roofline, l2, peak)
    return out


# ---- the oracle as the CPU baseline / reference arm --------------------------------------

def oracle_head_pass(oracle, hw, xb, ncols: int, threads: int) -> int:
    """The oracle on the first `ncols` output columns of the LM head at M = 1;
    returns their algorithmic bytes."""
    from skinny_gemm_gb300 import roofline
    cols = np.arange(ncols, dtype=np.int64)
    oracle.mm(xb, hw.Wq, hw.scales, hw.biases, 1, hw.N, hw.K, cols=cols, threads=threads)
    return roofline.mm_bytes(1, ncols, hw.K)


def oracle_one_core(oracle, synth, roofline, seconds: float) -> dict:
    """The oracle on one core on the two smallest configurations: the tiny
    256x512 matvec and the decode-layer projection set, both at M = 1."""
    out = {}
    sets = {"tiny_256x512": [(256, 512)], "decode_layer_set": [(N, K) for _, N, K in DECODE_LAYER]}
    for name, shapes in sets.items():
        mats = [(synth.make_weights(3 + i, N, K), synth.make_x(4 + i, 1, K)) for i, (N, K) in enumerate(shapes)]
        t0, passes, nbytes = time.perf_counter(), 0, 0
        while True:
            for hw, xb in mats:
                oracle.mm(xb, hw.Wq, hw.scales, hw.biases, 1, hw.N, hw.K, threads=1)
                nbytes += roofline.mm_bytes(1, hw.N, hw.K)
            passes += 1
            if time.perf_counter() - t0 >= seconds:
                break
        dt = time.perf_counter() - t0
        out[name] = {"GBps": round(nbytes / dt / 1e9, 5), "s_per_pass": round(dt / passes, 4), "passes": passes}
    out["cores"] = 1
    return out


def cpu_baseline(seconds: float, hw):
    import oracle
    from skinny_gemm_gb300 import roofline, synth
    xb = synth.make_x(2, 1, hw.K)
    threads = oracle.host_threads()
    t0 = time.perf_counter()
    nbytes, passes = 0, 0
    while True:
        nbytes += oracle_head_pass(oracle, hw, xb, hw.N, threads)
        passes += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    one = oracle_one_core(oracle, synth, roofline, 1.0)
    return {"value": round(nbytes / dt / 1e9, 4), "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{passes} full fp64 oracle passes over the 262144x2560 LM head at M=1 ({dt:.1f} s)",
            "one_core": one}


def run_reference(args, world, rank, local):
    if rank != 0:
        return
    import oracle
    from skinny_gemm_gb300 import synth
    hw = synth.make_weights(1, HEAD_N, HEAD_K)
    xb = synth.make_x(2, 1, HEAD_K)
    threads = oracle.host_threads()
    # size each step so warm-up + timed steps take about two minutes of CPU time
    t0 = time.perf_counter()
    probe = 2048
    oracle_head_pass(oracle, hw, xb, probe, threads)
    per_col = (time.perf_counter() - t0) / probe
    budget = 120.0 / max(1, args.steps + args.warmup)
    ncols = int(min(HEAD_N, max(64, budget / max(per_col, 1e-12))))
    for _ in range(args.warmup):
        oracle_head_pass(oracle, hw, xb, ncols, threads)
    t0 = time.perf_counter()
    nbytes = 0
    for _ in range(args.steps):
        nbytes += oracle_head_pass(oracle, hw, xb, ncols, threads)
    dt = time.perf_counter() - t0
    value = nbytes / dt / 1e9
    sample = f"first {ncols} of the 262144 output columns of the LM head per step, fp64 oracle"
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * dt / args.steps, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": dict(CONFIG),
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_case(args):
    """One workload, `steps` eager launches round-robin over cold copies."""
    import torch
    from skinny_gemm_gb300 import ops, roofline, synth
    N, K, E = CASES[args.case]
    M = args.M
    l2 = int(getattr(torch.cuda.get_device_properties(0), "L2_cache_size", 126 * 2**20))
    if args.case.startswith("stq1"):
        run_stq1_case(args, torch, ops, roofline, synth, N, K, E, M, l2)
        return
    hw = synth.make_weights(11, N, K, E)
    base = ops.W4Matrix.from_host(hw)
    copies = max(1, math.ceil(3 * l2 / base.nbytes))
    ws = [base] + [ops.W4Matrix(base.Wq.clone(), base.scales.clone(), base.biases.clone(), N, K, E)
                   for _ in range(copies - 1)]
    x = torch.randn(M, K, device="cuda").to(torch.bfloat16)
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    if E > 1:
        ids_np = synth.make_ids(0, M, E)
        ids = torch.from_numpy(ids_np).cuda()
        call = lambda w: ops.mm_id(x, w, ids, out=y, kernel=args.kernel)  # noqa: E731
        nbytes = roofline.mm_id_bytes(ids_np, M, N, K, E)[0]
    else:
        wsel = None if args.no_workspace else "auto"
        call = lambda w: ops.mm(x, w, out=y, kernel=args.kernel, workspace=wsel)  # noqa: E731
        nbytes = roofline.mm_bytes(M, N, K)
    for i in range(args.warmup):
        call(ws[i % copies])
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda._sleep(20_000_000)  # queue the launches behind a spin so the CPU never starves the GPU
    a.record()
    for i in range(args.steps):
        call(ws[i % copies])
    b.record()
    torch.cuda.synchronize()
    us = 1e3 * a.elapsed_time(b) / args.steps
    print(json.dumps({"case": args.case, "M": M, "N": N, "K": K, "E": E, "us_per_call": round(us, 3),
                      "GBps": round(nbytes / (us * 1e-6) / 1e9, 1), "plan": ops.get_plan(N, K, args.kernel)}))


def stq1_cold_set(torch, ops, synth, N, K, E, l2, seed):
    base = ops.STQ1Matrix.from_host(synth.make_stq1(seed, N, K, E), N, K, E)
    copies = max(1, math.ceil(3 * l2 / base.packed.numel()))
    return [base] + [ops.STQ1Matrix(base.packed.clone(), N, K, E) for _ in range(copies - 1)]


def run_stq1_case(args, torch, ops, roofline, synth, N, K, E, M, l2):
    """An STQ1_0 workload alone: eager launches round-robin over cold copies."""
    ws = stq1_cold_set(torch, ops, synth, N, K, E, l2, 12)
    copies = len(ws)
    x = torch.randn(M, K, device="cuda")
    y = torch.empty(M, N, device="cuda")
    if E > 1:
        ids_np = synth.make_ids(0, M, E)
        ids = torch.from_numpy(ids_np).cuda()
        call = lambda w: ops.stq1_mm_id(x, w, ids, out=y)  # noqa: E731
        nbytes = roofline.stq1_mm_id_bytes(ids_np, M, N, K, E)[0]
    else:
        call = lambda w: ops.stq1_mm(x, w, out=y)  # noqa: E731
        nbytes = roofline.stq1_mm_bytes(M, N, K)
    for i in range(args.warmup):
        call(ws[i % copies])
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda._sleep(20_000_000)
    a.record()
    for i in range(args.steps):
        call(ws[i % copies])
    b.record()
    torch.cuda.synchronize()
    us = 1e3 * a.elapsed_time(b) / args.steps
    print(json.dumps({"case": args.case, "M": M, "N": N, "K": K, "E": E, "us_per_call": round(us, 3),
                      "GBps": round(nbytes / (us * 1e-6) / 1e9, 1), "plan": ops.stq1_get_plan(N, K)}))


def measure_stq1(torch, ops, synth, roofline, l2, peak):
    """STQ1_0 ternary workloads of the Hy4 page: the 16384^2 matvec of its
    bandwidth table, the 6144x2048 expert at batch 1..8, eight routed experts."""
    out = {}

    def timed(ws, M, N, K, reps):
        x = torch.randn(M, K, device="cuda")
        y = torch.empty(M, N, device="cuda")
        ms = time_graph_launches(torch, [lambda w=w: ops.stq1_mm(x, w, out=y) for w in ws], reps)
        g = roofline.stq1_mm_bytes(M, N, K) / (ms * 1e-3) / 1e9
        return {"us": round(1e3 * ms, 2), "GBps": round(g, 1), "frac": round(g / peak, 4)}

    for (N, K, Ms) in [(16384, 16384, (1, 2)), (6144, 2048, (1, 2, 4, 5, 8))]:
        ws = stq1_cold_set(torch, ops, synth, N, K, 1, l2, 10)
        for M in Ms:
            out[f"{N}x{K}_M{M}"] = timed(ws, M, N, K, 10)
        del ws
    E, N, K, T = 8, 6144, 2048, 8
    ws = stq1_cold_set(torch, ops, synth, N, K, E, l2, 0)
    ids_np = synth.make_ids(0, T, E)
    ids = torch.from_numpy(ids_np).cuda()
    x = torch.randn(T, K, device="cuda")
    y = torch.empty(T, N, device="cuda")
    ms = time_graph_launches(torch, [lambda w=w: ops.stq1_mm_id(x, w, ids, out=y) for w in ws], 20)
    nb, touched = roofline.stq1_mm_id_bytes(ids_np, T, N, K, E)
    out["routed_8x6144x2048_T8"] = {"experts_touched": touched, "us": round(1e3 * ms, 2),
                                    "GBps": round(nb / (ms * 1e-3) / 1e9, 1),
                                    "frac": round(nb / (ms * 1e-3) / 1e9 / peak, 4)}
    return out


def main():
    args = parse_args()
    world, rank, local = dist_env()
    if args.case:
        run_case(args)
        return
    if args.impl == "reference":
        run_reference(args, world, rank, local)
    else:
        run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
