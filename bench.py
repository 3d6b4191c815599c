#!/usr/bin/env python3
"""Benchmark of the W4A16 group-64 skinny GEMM on GB300.

One step = the decode-layer projection set of a hidden-2560 model at M = 1
(q 2048x2560, k 512x2560, v 512x2560, o 2560x2048, gate 10240x2560,
up 10240x2560, down 2560x10240), i.e. seven w4a16_mm calls streaming 51.6 MB
of packed weights.  The metric is achieved HBM GB/s over the algorithmic
bytes (codes + scales + biases + activations + outputs, read or written once;
tiny-llm "Week 2 Day 2: Keep W4 Packed", section "Revisit the Decode
Roofline") and its fraction of the measured GB300 copy bandwidth.

Timing: the layer weights are replicated into enough copies that one pass
over them is > 3x the L2 size, and step s uses copy s mod L, so every step
streams its weights from HBM (no L2 flush needed).  Each copy's seven calls
are captured once in a CUDA graph; the timed region replays K graphs between
CUDA events on the launching stream, bracketed by a barrier and a
synchronize.  Per-launch durations (roofline) come from a second pass over
twin graphs that carry event nodes between the launches.  SM clocks are
sampled with nvidia-smi during the timed region.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
Under torchrun (N > 1) every rank runs its own independent layers (weak
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
DECODE_LAYER = [("q", 2048, 2560), ("k", 512, 2560), ("v", 512, 2560), ("o", 2560, 2048),
                ("gate", 10240, 2560), ("up", 10240, 2560), ("down", 2560, 10240)]
WORKLOAD = ("W4A16 g64 decode-layer projection set at M=1, hidden 2560: q 2048x2560, k 512x2560, "
            "v 512x2560, o 2560x2048, gate 10240x2560, up 10240x2560, down 2560x10240")
# The launches of one step.  A decoder layer's q/k/v projections are
# independent given their input, as are gate/up; they go through one
# w4a16_mm_group call each.  o and down depend on earlier results (attention,
# the gated activation) and run as their own w4a16_mm calls.
LAUNCHES = [("qkv", ("q", "k", "v")), ("o", ("o",)), ("gate_up", ("gate", "up")), ("down", ("down",))]
# Single workloads for --case: name -> (N, K, E)
CASES = {"q": (2048, 2560, 1), "kv": (512, 2560, 1), "o": (2560, 2048, 1), "gate": (10240, 2560, 1),
         "down": (2560, 10240, 1), "wide_up": (12288, 1536, 1), "wide_down": (1536, 12288, 1),
         "lm_head_1536": (262144, 1536, 1), "lm_head_2560": (262144, 2560, 1), "dense_16384": (16384, 16384, 1),
         "routed": (6144, 2048, 8),
         "stq1_16384": (16384, 16384, 1), "stq1_expert": (6144, 2048, 1), "stq1_routed": (6144, 2048, 8)}
FALLBACK_HBM_GBS = 6800.0
DOMINANT_KERNEL = "tc_tile_kernel"  # runs every projection of the decode-layer step
NOMINAL_HBM_GBS = 8000.0


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--kernel", default="auto", help="auto | simt | tc | vanilla")
    ap.add_argument("--no-extras", action="store_true", help="skip the per-config context measurements")
    ap.add_argument("--ungrouped", action="store_true", help="time the layer as seven w4a16_mm calls")
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


def run_ours(args, world, rank, local):
    import torch
    from skinny_gemm_gb300 import ops, roofline, synth

    torch.cuda.set_device(local)
    dist = init_dist(world)
    props = torch.cuda.get_device_properties(local)
    l2 = int(getattr(props, "L2_cache_size", 126 * 2**20))
    kernel = args.kernel
    plan = ops.get_plan(10240, 2560, kernel)
    step_bytes = layer_bytes(1)
    weight_bytes = sum(roofline.weight_bytes(N, K) for _, N, K in DECODE_LAYER)
    copies = max(2, math.ceil(3 * l2 / weight_bytes))
    layers, xs, ys = build_layers(torch, ops, synth, copies, seed=1000 * rank)

    stream = torch.cuda.Stream()
    try:
        make_ev = lambda: torch.cuda.Event(enable_timing=True, external=True)  # noqa: E731
        make_ev()
        external_ok = True
    except TypeError:
        make_ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
        external_ok = False

    grouped = not args.ungrouped and args.kernel == "auto"
    launches = LAUNCHES if grouped else [(name, (name,)) for name, _, _ in DECODE_LAYER]

    def enqueue_layer(layer, evs=None, launches=launches):
        for i, (_, names) in enumerate(launches):
            if evs is not None:
                evs[i].record()
            if len(names) == 1:
                ops.mm(xs[names[0]], layer[names[0]], out=ys[names[0]], kernel=kernel)
            else:
                ops.mm_group([xs[n] for n in names], [layer[n] for n in names], [ys[n] for n in names])
        if evs is not None:
            evs[len(launches)].record()

    graphs, ev_graphs, graph_events = [], [], []
    with torch.cuda.stream(stream):
        for layer in layers:  # eager warm-up of every launch before capture
            enqueue_layer(layer)
        torch.cuda.synchronize()
        for layer in layers:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                enqueue_layer(layer)
            graphs.append(g)
            if external_ok:  # a twin graph with event nodes between the launches
                ge = torch.cuda.CUDAGraph()
                evs = [make_ev() for _ in range(len(launches) + 1)]
                with torch.cuda.graph(ge, stream=stream):
                    enqueue_layer(layer, evs)
                ev_graphs.append(ge)
                graph_events.append(evs)
    torch.cuda.synchronize()

    def replay(s):
        graphs[s % len(graphs)].replay()

    with torch.cuda.stream(stream):
        for s in range(args.warmup):
            replay(s)
    torch.cuda.synchronize()

    device_id = getattr(props, "uuid", None)
    device_id = f"GPU-{device_id}" if device_id is not None and not str(device_id).startswith("GPU-") else device_id
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(str(device_id) if device_id else None)
    with sampler:
        barrier(dist)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            t_start.record()
            for s in range(args.steps):
                replay(s)
            t_end.record()
        torch.cuda.synchronize()
        barrier(dist)
    ms_total = max_over_ranks(dist, t_start.elapsed_time(t_end))
    ms_per_step = ms_total / args.steps
    value = aggregate_gbps(world, step_bytes, args.steps, ms_total)

    dims = {name: (N, K) for name, N, K in DECODE_LAYER}

    def launch_bytes(names):
        return sum(roofline.mm_bytes(1, *dims[n]) for n in names)

    # Per-launch durations, from a second pass over the same rotating layers
    # whose graphs carry event nodes between launches.
    launch_ms = []
    if external_ok:
        with torch.cuda.stream(stream):
            for rep in range(3):
                for ge in ev_graphs:
                    ge.replay()
        torch.cuda.synchronize()
        for evs in graph_events:
            launch_ms.append([evs[i].elapsed_time(evs[i + 1]) for i in range(len(launches))])
    else:  # eager launches queued behind a spin kernel, so events bracket only the kernels
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(len(launches) + 1)]
        with torch.cuda.stream(stream):
            for layer in layers:
                torch.cuda._sleep(50_000_000)
                enqueue_layer(layer, evs)
                torch.cuda.synchronize()
                launch_ms.append([evs[i].elapsed_time(evs[i + 1]) for i in range(len(launches))])
    peak, peak_kind = measured_peak()
    # The dominant kernel is every launch of the step (the tile kernel runs all
    # of them), and programmatic dependent launch overlaps each launch with its
    # neighbours, so its average launch duration is the timed region over the
    # launches in it, and its achieved rate is the step's algorithmic bytes
    # over the step time.
    launches_per_step = len(launches)
    launch_us = 1e3 * ms_total / (args.steps * launches_per_step)
    achieved = step_bytes / (launches_per_step * launch_us * 1e-6) / 1e9
    per_launch = {}
    for i, (lname, names) in enumerate(launches):
        us = 1e3 * sum(r[i] for r in launch_ms) / len(launch_ms)
        per_launch[lname] = {"matrices": [f"{n} {dims[n][0]}x{dims[n][1]}" for n in names], "us": round(us, 3),
                             "GBps": round(launch_bytes(names) / (us * 1e-6) / 1e9, 1)}

    # The same layer as seven separate w4a16_mm calls (context for the grouping).
    ungrouped = None
    if grouped and not args.no_extras:
        seven = [(name, (name,)) for name, _, _ in DECODE_LAYER]
        g7 = []
        with torch.cuda.stream(stream):
            for layer in layers:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    enqueue_layer(layer, launches=seven)
                g7.append(g)
            for s_ in range(args.warmup):
                g7[s_ % len(g7)].replay()
        torch.cuda.synchronize()
        a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n7 = max(1, min(args.steps, 5000))
        with torch.cuda.stream(stream):
            a_.record()
            for s_ in range(n7):
                g7[s_ % len(g7)].replay()
            b_.record()
        torch.cuda.synchronize()
        ms7 = a_.elapsed_time(b_) / n7
        ungrouped = {"launches_per_step": 7, "ms_per_step": round(ms7, 6),
                     "GBps": round(step_bytes / (ms7 * 1e-3) / 1e9, 2)}
        del g7

    e2e = measure_e2e(torch, ops, layers, args.steps, kernel, step_bytes, world, dist, launches)
    extras = None if args.no_extras else measure_extras(torch, ops, synth, roofline, l2, kernel, peak)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args.cpu_seconds)

    if rank == 0:
        clocks = sampler.summary()
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_per_step, 6), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "accumulate": "f32", "data": "synthetic",
            "config": {"workload": WORKLOAD, "M": 1, "group_size": 64, "bytes_per_step": step_bytes,
                       "kernel": plan["kernel"], "plan": plan,
                       "l2_policy": f"inputs larger than L2: {copies} rotating layer copies "
                                    f"({copies * weight_bytes / 1e6:.0f} MB > 3x L2 {l2 / 1e6:.0f} MB)",
                       "cuda_graphs": True, "parallelism": f"replicas x{world}",
                       "launches": [f"{ln}: " + ("w4a16_mm_group" if len(nm) > 1 else "w4a16_mm") + f"({', '.join(nm)})"
                                    for ln, nm in launches]},
            "roofline": {"bound": "hbm", "kernel": DOMINANT_KERNEL, "achieved": round(achieved, 1), "peak": peak,
                         "unit": "GB/s", "frac": round(achieved / peak, 4),
                         "traffic": ncu_traffic(DOMINANT_KERNEL),
                         "algorithmic_bytes_per_launch": round(step_bytes / launches_per_step),
                         "launch_us": round(launch_us, 3),
                         "peak_kind": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
                         if peak_kind == "measured" else "fallback 6.8 TB/s",
                         "frac_of_nominal_8TBps": round(achieved / NOMINAL_HBM_GBS, 4),
                         "launches_timed": args.steps * launches_per_step,
                         "timing": "CUDA events around the timed region on the launching stream; "
                                   "average launch = region / launches (launches overlap)"},
            "per_launch_serialised": {
                "timing": ("event nodes between the launches of twin graphs, replayed after the timed region; "
                           "the event nodes stop the launches from overlapping, so these are upper bounds"
                           if external_ok else "events behind a spin kernel"),
                **per_launch},
            "ungrouped_layer": ungrouped,
            "e2e": e2e,
            "gpu_launches": args.steps * launches_per_step,
            "clocks": clocks,
        }
        if cpu is not None:
            line["cpu_baseline"] = cpu
        if extras is not None:
            line["extras"] = extras
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def measure_e2e(torch, ops, layers, steps, kernel, step_bytes, world, dist, launches):
    """Through the public API, every step: pinned host -> device copy of the
    step's activations, the layer's calls (the same launches as the timed
    region), device -> pinned host read of the outputs (with the
    synchronisation that read implies)."""
    k_in = [K for _, N, K in DECODE_LAYER]
    n_out = [N for _, N, K in DECODE_LAYER]
    h_in = torch.empty(sum(k_in), dtype=torch.bfloat16, pin_memory=True)
    h_out = torch.empty(sum(n_out), dtype=torch.bfloat16, pin_memory=True)
    h_in.copy_(torch.randn(sum(k_in)).to(torch.bfloat16))
    d_in = torch.empty(sum(k_in), dtype=torch.bfloat16, device="cuda")
    d_out = torch.empty(sum(n_out), dtype=torch.bfloat16, device="cuda")
    ins, outs, a, b = [], [], 0, 0
    for K, N in zip(k_in, n_out):
        ins.append(d_in[a:a + K].view(1, K))
        outs.append(d_out[b:b + N].view(1, N))
        a, b = a + K, b + N
    n = max(1, min(steps, 5000))

    idx = {name: i for i, (name, N, K) in enumerate(DECODE_LAYER)}

    def step(s):
        d_in.copy_(h_in, non_blocking=True)
        layer = layers[s % len(layers)]
        for _, names in launches:
            if len(names) == 1:
                ops.mm(ins[idx[names[0]]], layer[names[0]], out=outs[idx[names[0]]], kernel=kernel)
            else:
                ops.mm_group([ins[idx[n]] for n in names], [layer[n] for n in names], [outs[idx[n]] for n in names])
        h_out.copy_(d_out, non_blocking=True)
        torch.cuda.current_stream().synchronize()

    for s in range(min(50, n)):
        step(s)
    barrier(dist)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for s in range(n):
        step(s)
    dt = max_over_ranks(dist, time.perf_counter() - t0)
    return {"value": round(world * step_bytes * n / dt / 1e9, 2), "unit": UNIT,
            "h2d_bytes_per_step": int(h_in.numel() * 2), "d2h_bytes_per_step": int(h_out.numel() * 2),
            "steps": n, "ms_per_step": round(1e3 * dt / n, 4),
            "api": "skinny_gemm_gb300.ops.mm / mm_group (eager, the C ABI through ctypes)"}


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


def measure_extras(torch, ops, synth, roofline, l2, kernel, peak):
    """Context numbers on the other workloads (M = 1..8), cold weights."""
    out = {}

    def cold_set(N, K, seed):
        wb = roofline.weight_bytes(N, K)
        copies = max(1, math.ceil(3 * l2 / wb))
        hw = synth.make_weights(seed, N, K)
        base = ops.W4Matrix.from_host(hw)
        ws = [base] + [ops.W4Matrix(base.Wq.clone(), base.scales.clone(), base.biases.clone(), N, K)
                       for _ in range(copies - 1)]
        return ws

    def gbps(ws, M, N, K, reps):
        x = torch.randn(M, K, device="cuda").to(torch.bfloat16)
        y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        fns = [lambda w=w: ops.mm(x, w, out=y, kernel=kernel) for w in ws]
        ms = time_graph_launches(torch, fns, reps)
        return ms, roofline.mm_bytes(M, N, K) / (ms * 1e-3) / 1e9

    verify = {}
    for (N, K) in [(10240, 2560), (2560, 10240), (12288, 1536), (1536, 12288)]:
        ws = cold_set(N, K, 7)
        t = {M: gbps(ws, M, N, K, 20) for M in (1, 3, 5, 7)}
        verify[f"{N}x{K}"] = {f"M{M}_us": round(1e3 * t[M][0], 3) for M in t}
        verify[f"{N}x{K}"].update({f"M{M}_GBps": round(t[M][1], 1) for M in t})
        verify[f"{N}x{K}"]["t5_over_t1"] = round(t[5][0] / t[1][0], 3)
        del ws
    out["verify"] = verify
    lm, lm_argmax = {}, {}
    for (N, K) in [(262144, 1536), (262144, 2560)]:
        ws = cold_set(N, K, 8)
        for M in (1, 3):
            ms, g = gbps(ws, M, N, K, 10)
            lm[f"{N}x{K}_M{M}"] = {"us": round(1e3 * ms, 2), "GBps": round(g, 1), "frac": round(g / peak, 4)}
        # greedy head: w4a16_mm_argmax against w4a16_mm followed by torch.argmax over the logits
        for M in (1, 3):
            x = torch.randn(M, K, device="cuda").to(torch.bfloat16)
            y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
            idx = torch.empty(M, dtype=torch.int32, device="cuda")
            val = torch.empty(M, dtype=torch.bfloat16, device="cuda")
            fused = [lambda w=w: ops.mm_argmax(x, w, idx=idx, val=val) for w in ws]
            unfused = [lambda w=w: (ops.mm(x, w, out=y, kernel=kernel), torch.argmax(y, dim=-1)) for w in ws]
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
        ms, g = gbps(ws, M, 16384, 16384, 10)
        dense[f"M{M}"] = {"us": round(1e3 * ms, 2), "GBps": round(g, 1), "frac": round(g / peak, 4)}
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
    fns = [lambda w=w: ops.mm_id(x, w, ids, out=y, kernel=kernel) for w in ws]
    ms = time_graph_launches(torch, fns, 20)
    nb, touched = roofline.mm_id_bytes(ids_np, T, N, K, E)
    out["routed"] = {"experts_touched": touched, "bytes": nb, "us": round(1e3 * ms, 2),
                     "GBps": round(nb / (ms * 1e-3) / 1e9, 1), "frac": round(nb / (ms * 1e-3) / 1e9 / peak, 4)}
    del ws
    out["stq1"] = measure_stq1(torch, ops, synth, roofline, l2, peak)
    return out


# ---- the oracle as the CPU baseline / reference arm --------------------------------------

def oracle_layer_pass(oracle, host, xs, cols_frac: float, threads: int):
    """One oracle pass over a column sample of the decode layer; returns algorithmic bytes."""
    from skinny_gemm_gb300 import roofline
    total = 0
    for name, N, K in DECODE_LAYER:
        hw = host[name]
        nc = max(1, int(round(N * cols_frac)))
        cols = np.arange(nc, dtype=np.int64)
        oracle.mm(xs[name], hw.Wq, hw.scales, hw.biases, 1, N, K, cols=cols, threads=threads)
        total += roofline.mm_bytes(1, nc, K)
    return total


def cpu_baseline(seconds: float):
    import oracle
    from skinny_gemm_gb300 import synth
    host = {name: synth.make_weights(i, N, K) for i, (name, N, K) in enumerate(DECODE_LAYER)}
    xs = {name: synth.make_x(100 + i, 1, K) for i, (name, N, K) in enumerate(DECODE_LAYER)}
    threads = oracle.host_threads()
    t0 = time.perf_counter()
    nbytes = oracle_layer_pass(oracle, host, xs, 1.0, threads)
    passes = 1
    while time.perf_counter() - t0 < seconds:
        nbytes += oracle_layer_pass(oracle, host, xs, 1.0, threads)
        passes += 1
    dt = time.perf_counter() - t0
    return {"value": round(nbytes / dt / 1e9, 4), "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{passes} full fp64 oracle passes over the decode-layer set at M=1 ({dt:.1f} s)"}


def run_reference(args, world, rank, local):
    if rank != 0:
        return
    import oracle
    from skinny_gemm_gb300 import synth
    host = {name: synth.make_weights(i, N, K) for i, (name, N, K) in enumerate(DECODE_LAYER)}
    xs = {name: synth.make_x(100 + i, 1, K) for i, (name, N, K) in enumerate(DECODE_LAYER)}
    threads = oracle.host_threads()
    # size each step so warm-up + timed steps take about two minutes of CPU time
    t0 = time.perf_counter()
    oracle_layer_pass(oracle, host, xs, 0.01, threads)
    per_frac = (time.perf_counter() - t0) / 0.01
    budget = 120.0 / max(1, args.steps + args.warmup)
    frac = min(1.0, max(1e-4, budget / max(per_frac, 1e-9)))
    for _ in range(args.warmup):
        oracle_layer_pass(oracle, host, xs, frac, threads)
    t0 = time.perf_counter()
    nbytes = 0
    for _ in range(args.steps):
        nbytes += oracle_layer_pass(oracle, host, xs, frac, threads)
    dt = time.perf_counter() - t0
    value = nbytes / dt / 1e9
    sample = f"first {frac:.4%} of the output columns of each decode-layer matrix per step, fp64 oracle"
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * dt / args.steps, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": WORKLOAD, "M": 1, "group_size": 64},
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
        call = lambda w: ops.mm(x, w, out=y, kernel=args.kernel)  # noqa: E731
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
