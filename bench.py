#!/usr/bin/env python3
"""Benchmark of the NF4 weight-only linear layer on one GB300 (or N independent replicas).

Headline: NF4 GEMV (M = 1) HBM GB/s on the packed bytes over one decode pass of the 3B-shaped
workload (hidden 2048, 36 layers x 7 linears, 1.474 GB of codes + scales resident in HBM).  A step
is one pass over all 252 linears, replayed from a CUDA graph.  The prefill contractions (M = 32 and
M = 512 on the 20B-shaped linears) are timed after the headline loop and reported as extra keys.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
For N > 1 launch with torch.distributed.run; each rank runs a full replica (weak scaling).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from nf4_weight_only_gb300 import workloads as W  # noqa: E402

METRIC = "NF4 GEMV HBM GB/s (M=1) & % of peak; prefill TFLOP/s at M=32/512"


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            d = json.load(fh)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in getattr(self, "lines", []):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = max(mx, float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx or None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------------------------------------
# our arm
# ------------------------------------------------------------------------------------------------
def build_weights(nf4, synth, wl: W.Workload, dev):
    """Quantize every linear of every layer on the device (fp32 weights drawn there, then freed)."""
    mats = []
    for layer in range(wl.layers):
        for li, lin in enumerate(wl.linears):
            w = synth.device_weights(wl.seed * 100003 + layer * 16 + li, lin.n, lin.k, dev,
                                     outlier_frac=wl.outlier_frac)
            codes, scales = nf4.quantize(w)
            del w
            mats.append((lin, codes, scales))
    torch.cuda.synchronize()
    return mats


def time_graph(graph, stream, steps, warmup, flush=None):
    for _ in range(warmup):
        graph.replay()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    times = []
    for _ in range(steps):
        if flush is not None:
            flush()
        with torch.cuda.stream(stream):
            start.record(stream)
            graph.replay()
            end.record(stream)
        end.synchronize()
        times.append(start.elapsed_time(end) / 1e3)
    return times


def run_ours(args, rank, world):
    import nf4_weight_only_gb300 as nf4
    from nf4_weight_only_gb300 import build, synth

    build.build()
    nf4.load()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    pk = peaks()
    wl = W.DECODE_3B
    mats = build_weights(nf4, synth, wl, dev)
    xs = {k: synth.device_activations_bf16(77 + k, 1, k, dev) for k in {l.k for l in wl.linears}}
    ys = [torch.empty((1, lin.n), dtype=torch.bfloat16, device=dev) for lin, _, _ in mats]
    stream = torch.cuda.Stream(device=dev)

    def step():
        for (lin, codes, scales), y in zip(mats, ys):
            nf4.nf4_linear(xs[lin.k], codes, scales, y, stream)

    with torch.cuda.stream(stream):
        step()  # first call per device builds its constant table outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    torch.cuda.synchronize()

    packed = wl.packed_bytes_per_pass()
    algo = packed + sum(2 * lin.k + 2 * lin.n for lin, _, _ in mats)  # + x reads and y writes
    launches = len(mats)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clk:
        t0 = time.perf_counter()
        times = time_graph(graph, stream, args.steps, args.warmup)
        wall = time.perf_counter() - t0
    clocks = clk.summary()
    step_s = max(times) if args.steps == 1 else statistics.median(times)
    total_s = sum(times)
    if world > 1:
        t = torch.tensor([total_s], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        total_s = float(t.item())
    gbs = packed * args.steps * world / total_s / 1e9
    per_launch_s = total_s / args.steps / launches
    achieved = (algo / launches) / per_launch_s / 1e9

    # end to end: pinned host x in, every y out, through the same C-ABI calls (no graph)
    xs_host = {k: v.cpu().pin_memory() for k, v in xs.items()}
    ys_host = [torch.empty_like(y, device="cpu").pin_memory() for y in ys]
    with torch.cuda.stream(stream):
        for _ in range(2):
            for k, h in xs_host.items():
                xs[k].copy_(h, non_blocking=True)
            graph.replay()
            for y, h in zip(ys, ys_host):
                h.copy_(y, non_blocking=True)
    torch.cuda.synchronize()
    e2e_steps = max(3, min(args.steps, 20))
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for _ in range(e2e_steps):
            for k, h in xs_host.items():
                xs[k].copy_(h, non_blocking=True)
            graph.replay()
            for y, h in zip(ys, ys_host):
                h.copy_(y, non_blocking=True)
    torch.cuda.synchronize()
    e2e_s = (time.perf_counter() - t0) / e2e_steps
    h2d = sum(2 * k for k in xs_host)
    d2h = sum(2 * y.numel() for y in ys)

    prefill = prefill_bench(nf4, synth, dev, pk) if not args.skip_prefill else None

    result = {
        "metric": METRIC, "value": round(gbs, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_s * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": wl.name, "linears_per_step": launches, "packed_bytes_per_step": packed,
                   "l2": "inputs larger than L2 (1.47 GB of packed weights per step)",
                   "graph": "one CUDA graph per step", "peak_source": pk["source"]},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / pk["hbm_gbs"], 4), "traffic": None,
                     "kernel": "gemv_kernel<1,1>", "note": "per-launch average over the timed steps, gaps included"},
        "e2e": {"value": round(packed / e2e_s / 1e9, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": launches * args.steps,
        "clocks": clocks,
    }
    if prefill is not None:
        result["prefill"] = prefill
    return result


def prefill_bench(nf4, synth, dev, pk):
    """TFLOP/s of the four 20B-shaped prefill linears at M = 32 and M = 512."""
    wl = W.PREFILL_20B
    mats = []
    for li, lin in enumerate(wl.linears):
        w = synth.device_weights(wl.seed * 100003 + li, lin.n, lin.k, dev, outlier_frac=wl.outlier_frac)
        mats.append((lin,) + tuple(nf4.quantize(w)))
        del w
    out = {}
    stream = torch.cuda.Stream(device=dev)
    for m in wl.tokens:
        xs = {k: synth.device_activations_bf16(99 + k, m, k, dev) for k in {l.k for l, _, _ in mats}}
        ys = [torch.empty((m, lin.n), dtype=torch.bfloat16, device=dev) for lin, _, _ in mats]

        def step():
            for (lin, codes, scales), y in zip(mats, ys):
                nf4.nf4_linear(xs[lin.k], codes, scales, y, stream)

        with torch.cuda.stream(stream):
            step()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            step()
        times = time_graph(graph, stream, 10, 3)
        t = statistics.median(times)
        flops = sum(2.0 * m * lin.n * lin.k for lin, _, _ in mats)
        tf = flops / t / 1e12
        packed = sum(lin.n * (lin.k // 2 + lin.k // 64 * 2) for lin, _, _ in mats)
        out[f"M{m}"] = {"tflops": round(tf, 2), "frac_of_bf16_peak": round(tf / pk["bf16_tflops"], 4),
                        "packed_gbs": round(packed / t / 1e9, 1), "ms": round(t * 1e3, 4)}
    return out


# ------------------------------------------------------------------------------------------------
# the oracle on the host cores (cpu_baseline and --impl reference)
# ------------------------------------------------------------------------------------------------
def oracle_sample(seconds_budget: float = 15.0):
    """Time the oracle's fp64 linear on one 3B-shaped layer (7 linears, M = 1) and scale it to
    packed GB/s.  Returns (GB/s, threads, description)."""
    import oracle
    from nf4_weight_only_gb300 import synth
    o = oracle.default()
    wl = W.DECODE_3B
    threads = os.cpu_count() or 1
    prepared = []
    for li, lin in enumerate(wl.linears):
        w = synth.weights(wl.seed * 100003 + li, lin.n, lin.k)
        codes, scales = o.quantize(w)
        prepared.append((lin, codes, scales, synth.activations_bf16(77 + lin.k, 1, lin.k)))
    packed = sum(lin.n * (lin.k // 2 + lin.k // 64 * 2) for lin, *_ in prepared)
    reps, total = 0, 0.0
    while total < seconds_budget and reps < 50:
        t0 = time.perf_counter()
        for lin, codes, scales, x in prepared:
            o.linear(x, codes, scales, nthreads=threads)
        total += time.perf_counter() - t0
        reps += 1
    gbs = packed * reps / total / 1e9
    return gbs, threads, f"{reps} pass(es) over one 3B-shaped layer (7 linears, {packed/1e6:.1f} MB packed), M=1, fp64"


def run_reference(args, rank, world):
    if rank != 0:
        return None
    budget = max(5.0, min(60.0, 10.0 * args.steps / max(args.steps, 1)))
    gbs, cores, sample = oracle_sample(budget)
    wl = W.DECODE_3B
    step_s = wl.packed_bytes_per_pass() / (gbs * 1e9)
    return {
        "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_s * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
        "config": {"workload": wl.name},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--skip-prefill", action="store_true")
    ap.add_argument("--skip-cpu-baseline", action="store_true")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        backend = "gloo" if args.impl == "reference" else "nccl"
        if backend == "nccl":
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        torch.distributed.init_process_group(backend)
    if args.impl == "reference":
        res = run_reference(args, rank, world)
    else:
        res = run_ours(args, rank, world)
        if rank == 0 and res is not None and not args.skip_cpu_baseline:
            gbs, cores, sample = oracle_sample(15.0)
            res["cpu_baseline"] = {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                                   "sample": sample}
    if rank == 0 and res is not None:
        print(json.dumps(res))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
