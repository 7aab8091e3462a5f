#!/usr/bin/env python3
"""Benchmark of the NF4 weight-only linear layer on one GB300 (or N independent replicas).

Headline: NF4 GEMV (M = 1) HBM GB/s on the packed bytes over one decode pass of the 3B-shaped
workload (hidden 2048, 36 layers, 1.474 GB of codes + scales resident in HBM).  A step is one pass
over every linear of every layer in dependency order -- per layer q|k|v (one grouped launch, shared
input), o, gate|up (grouped), down: 144 launches chained with programmatic dependent launch and
replayed from one CUDA graph.  The 20B-shaped prefill (M = 32 and M = 512) is timed after the
headline loop and reported under "prefill".

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

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from nf4_weight_only_gb300 import workloads as W  # noqa: E402

METRIC = "NF4 GEMV HBM GB/s (M=1) & % of peak; prefill TFLOP/s at M=32/512"

# One decoder layer's linears in dependency order; names in one tuple read the same input.
LAYER_STEPS = (("q", "k", "v"), ("o",), ("gate", "up"), ("down",))


def decode_traffic_per_launch():
    """DRAM bytes per decode launch from the committed ncu launch-list summary (None if absent)."""
    import re
    path = os.path.join(ROOT, "profiles", "gemv_decode_3b_launch_list.md")
    try:
        with open(path) as fh:
            m = re.search(r"^traffic_bytes_per_launch:\s*(\d+)", fh.read(), re.M)
        return int(m.group(1)) if m else None
    except OSError:
        return None


def max_over_ranks(seconds: float, device) -> float:
    """The slowest rank's time (all ranks call it; device is where the process group's tensors live:
    the rank's GPU for NCCL, the CPU for gloo)."""
    t = torch.tensor([float(seconds)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank_step: float, steps: int, world: int, max_seconds: float) -> float:
    """Whole-job rate: the units every rank processed (weak scaling: each rank runs its own replica)
    divided by the slowest rank's time."""
    return units_per_rank_step * steps * world / max_seconds


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            d = json.load(fh)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]


def sample_clocks(gpu_index: int):
    """One nvidia-smi reading: SM clock, max SM clock, active throttle reasons (None if unavailable)."""
    try:
        out = subprocess.run(["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={CLOCK_FIELDS}",
                              "--format=csv,noheader,nounits"], capture_output=True, text=True, timeout=10).stdout
    except (OSError, subprocess.TimeoutExpired):
        return None
    parts = [p.strip() for p in out.strip().split(",")]
    if len(parts) < 9:
        return None
    try:
        return {"sm": float(parts[1]), "max": float(parts[2]),
                "reasons": [n for n, v in zip(REASONS, parts[5:9]) if v.lower().startswith("active")]}
    except ValueError:
        return None


def clocks_summary(samples):
    samples = [s for s in samples if s]
    if not samples:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
    return {"sm_mhz": statistics.median(s["sm"] for s in samples), "sm_max_mhz": max(s["max"] for s in samples),
            "reasons": sorted({r for s in samples for r in s["reasons"]}), "samples": len(samples)}


def timed_replays(graph, stream, steps, warmup, gpu_index):
    """`warmup` untimed replays, then exactly `steps` replays enqueued between CUDA events on
    `stream`; nvidia-smi is sampled while the device works through them.
    Returns (per-step seconds, total seconds, clock samples)."""
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            graph.replay()
    torch.cuda.synchronize()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    with torch.cuda.stream(stream):
        evs[0].record(stream)
        for i in range(steps):
            graph.replay()
            evs[i + 1].record(stream)
    samples = []
    while not evs[-1].query():
        samples.append(sample_clocks(gpu_index))
    torch.cuda.synchronize()
    per = [evs[i].elapsed_time(evs[i + 1]) / 1e3 for i in range(steps)]
    return per, evs[0].elapsed_time(evs[-1]) / 1e3, samples


def build_layers(nf4, synth, wl: W.Workload, dev):
    """Quantize every linear of every layer on the device (fp32 weights drawn there, then freed)."""
    layers = []
    for layer in range(wl.layers):
        mats = {}
        for li, lin in enumerate(wl.linears):
            w = synth.device_weights(wl.seed * 100003 + layer * 16 + li, lin.n, lin.k, dev,
                                     outlier_frac=wl.outlier_frac)
            codes, scales = nf4.quantize(w)
            del w
            mats[lin.name] = (lin, codes, scales)
        layers.append(mats)
    torch.cuda.synchronize()
    return layers


def run_ours(args, rank, world):
    import nf4_weight_only_gb300 as nf4
    from nf4_weight_only_gb300 import build, synth

    build.build()
    nf4.load()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    pk = peaks()
    wl = W.DECODE_3B
    layers = build_layers(nf4, synth, wl, dev)
    xs = {k: synth.device_activations_bf16(77 + k, 1, k, dev) for k in {l.k for l in wl.linears}}
    # every y is a view of one flat buffer (each n is a multiple of 8, so every view stays 16-byte
    # aligned), which the end-to-end step copies back to the host in one transfer
    y_flat = torch.empty(wl.layers * sum(lin.n for lin in wl.linears), dtype=torch.bfloat16, device=dev)
    ys, off = [], 0
    for m in layers:
        yl = {}
        for name, (lin, _, _) in m.items():
            yl[name] = y_flat[off:off + lin.n].view(1, lin.n)
            off += lin.n
        ys.append(yl)
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()  # x is drawn on the default stream

    def step():
        for mats, yl in zip(layers, ys):
            for names in LAYER_STEPS:
                lin = mats[names[0]][0]
                if len(names) == 1:
                    nf4.nf4_linear(xs[lin.k], mats[names[0]][1], mats[names[0]][2], yl[names[0]], stream)
                else:
                    nf4.nf4_linear_grouped(xs[lin.k], [mats[n][1] for n in names], [mats[n][2] for n in names],
                                           [yl[n] for n in names], stream)

    launches = wl.layers * len(LAYER_STEPS)
    with torch.cuda.stream(stream):
        step()  # the first call per device builds its constant table, outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    torch.cuda.synchronize()

    packed = wl.packed_bytes_per_pass()
    algo = packed + wl.layers * sum(2 * lin.k + 2 * lin.n for lin in wl.linears)  # + x reads, y writes
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    times, total_s, samples = timed_replays(graph, stream, args.steps, args.warmup, dev.index)
    if world > 1:
        torch.distributed.barrier()
        total_s = max_over_ranks(total_s, dev)
    clocks = clocks_summary(samples)
    step_s = statistics.median(times)
    gbs = job_throughput(packed, args.steps, world, total_s) / 1e9
    per_launch_s = total_s / args.steps / launches
    achieved = (algo / launches) / per_launch_s / 1e9

    # end to end: pinned host x in and every y out each step (one transfer of the flat y buffer),
    # around the same graph of C-ABI calls
    xs_host = {k: v.cpu().pin_memory() for k, v in xs.items()}
    y_host = torch.empty(y_flat.shape, dtype=y_flat.dtype).pin_memory()

    def e2e_step():
        for k, h in xs_host.items():
            xs[k].copy_(h, non_blocking=True)
        graph.replay()
        y_host.copy_(y_flat, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            e2e_step()
    torch.cuda.synchronize()
    e2e_steps = max(3, min(args.steps, 50))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        e1.record(stream)
    torch.cuda.synchronize()
    e2e_s = e0.elapsed_time(e1) / 1e3 / e2e_steps
    h2d = sum(2 * k for k in xs_host)
    d2h = 2 * y_flat.numel()

    prefill = prefill_bench(nf4, synth, dev, pk) if not args.skip_prefill else None
    embed = embed_bench(nf4, synth, dev, pk) if not args.skip_prefill else None
    codec = codec_bench(nf4, synth, dev, pk) if not args.skip_prefill else None
    overflow = overflow_bench(nf4, synth, dev) if not args.skip_prefill else None

    result = {
        "metric": METRIC, "value": round(gbs, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_s * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": wl.name, "launches_per_step": launches,
                   "launch_structure": "per layer: q|k|v grouped, o, gate|up grouped, down (PDL-chained)",
                   "packed_bytes_per_step": packed,
                   "l2": "inputs larger than L2 (1.47 GB of packed weights per step)",
                   "graph": "one CUDA graph per step", "peak_source": pk["source"]},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / pk["hbm_gbs"], 4), "traffic": decode_traffic_per_launch(),
                     "algorithmic_bytes_per_launch": int(algo / launches),
                     "kernel": "gemv_kernel<1,1,2|4> (CUDA-core GEMV, M = 1)",
                     "note": "algorithmic bytes (codes+scales+x+y) per launch / average launch time over the "
                             "timed steps, inter-launch gaps included; peak of measured"},
        "e2e": {"value": round(packed / e2e_s / 1e9, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": launches * args.steps,
        "clocks": clocks,
    }
    if prefill is not None:
        result["prefill"] = prefill
    if embed is not None:
        result["embed"] = embed
    if codec is not None:
        result.update(codec)  # "quantize" and "dequant"
    if overflow is not None:
        result["overflow"] = overflow
    return result


def overflow_bench(nf4, synth, dev, layers: int = 2, passes: int = 8):
    """Overflow streaming: `layers` 32B-shaped layers (7 linears each, M = 1) whose packed weights
    stay in pinned host memory, streamed through the two-slot ring.  Reported as packed GB/s
    against a plain host-to-device copy of the same bytes (the link's own rate)."""
    wl = W.SWEEP_32B
    mats = []
    for layer in range(layers):
        for li, lin in enumerate(wl.linears):
            w = synth.device_weights(wl.seed * 100003 + layer * 16 + li, lin.n, lin.k, dev)
            codes, scales = nf4.quantize(w)
            del w
            mats.append((lin, codes.cpu().pin_memory(), scales.cpu().pin_memory()))
            del codes, scales
    torch.cuda.synchronize()
    xs = {k: synth.device_activations_bf16(88 + k, 1, k, dev) for k in {l.k for l in wl.linears}}
    ys = [torch.empty((1, lin.n), dtype=torch.bfloat16, device=dev) for lin, _, _ in mats]
    ops = [(xs[lin.k], c, s, y) for (lin, c, s), y in zip(mats, ys)]
    packed = sum(c.numel() + 2 * s.numel() for _, c, s in mats)
    stream = torch.cuda.Stream(device=dev)
    ring = nf4.Ring(max(nf4.Ring.bytes_needed(lin.n, lin.k) for lin in wl.linears))
    try:
        for _ in range(2):
            ring.run(ops, stream)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(passes):
            ring.run(ops, stream)
        e1.record(stream)
        samples = []
        while not e1.query():
            samples.append(sample_clocks(dev.index))
        torch.cuda.synchronize()
        ring_s = e0.elapsed_time(e1) / 1e3 / passes
    finally:
        ring.close()
    # the link alone: one pinned buffer of the same size copied to the device
    host = torch.empty(packed, dtype=torch.uint8).pin_memory()
    devbuf = torch.empty(packed, dtype=torch.uint8, device=dev)
    with torch.cuda.stream(stream):
        devbuf.copy_(host, non_blocking=True)
        torch.cuda.synchronize()
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        for _ in range(passes):
            devbuf.copy_(host, non_blocking=True)
        c1.record(stream)
    torch.cuda.synchronize()
    copy_s = c0.elapsed_time(c1) / 1e3 / passes
    return {"workload": f"{layers} x 32B-shaped layer ({len(mats)} linears, M = 1) from pinned host memory",
            "packed_bytes_per_pass": packed, "gbs": round(packed / ring_s / 1e9, 1), "ms_per_pass": round(ring_s * 1e3, 3),
            "h2d_copy_gbs": round(packed / copy_s / 1e9, 1), "frac_of_h2d_copy": round(copy_s / ring_s, 4),
            "kernel": "nf4_ring_run (copy engine into two slots + the linear kernels)",
            "clocks": clocks_summary(samples)}


def embed_bench(nf4, synth, dev, pk, vocab: int = 151936, hidden: int = 2048, n_ids: int = 4096):
    """GB/s of `nf4_embed` gathering `n_ids` random rows of a 3B-shaped packed embedding table
    (ids read, codes and scales of each row read, bf16 rows written)."""
    w = synth.device_weights(31, vocab, hidden, dev)
    codes, scales = nf4.quantize(w)
    del w
    gen = torch.Generator(device="cpu").manual_seed(32)
    ids = torch.randint(0, vocab, (n_ids,), generator=gen, dtype=torch.int32).to(dev)
    out = torch.empty((n_ids, hidden), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)  # larger than L2, written before each launch
    iters = 50
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
    with torch.cuda.stream(stream):
        for _ in range(5):
            nf4.nf4_embed(ids, codes, scales, out, stream)
        for a, b in evs:
            flush.fill_(1)
            a.record(stream)
            nf4.nf4_embed(ids, codes, scales, out, stream)
            b.record(stream)
    samples = []
    while not evs[-1][1].query():
        samples.append(sample_clocks(dev.index))
    torch.cuda.synchronize()
    t = statistics.median(a.elapsed_time(b) / 1e3 for a, b in evs)
    algo = n_ids * (4 + hidden // 2 + hidden // 64 * 2 + 2 * hidden)
    gbs = algo / t / 1e9
    return {"workload": f"{n_ids} random ids of a {vocab} x {hidden} packed table", "gbs": round(gbs, 1),
            "frac_of_hbm": round(gbs / pk["hbm_gbs"], 4), "us": round(t * 1e6, 2),
            "algorithmic_bytes": algo, "kernel": "embed_kernel", "l2": "flushed (256 MB written) before each launch",
            "clocks": clocks_summary(samples)}


def codec_bench(nf4, synth, dev, pk, n: int = 16384, k: int = 16384):
    """GB/s of `nf4_quantize` (fp32 in, codes + scales out: 4.53 B/weight) and `nf4_dequant` (codes +
    scales in, bf16 out: 2.53 B/weight) on one n x k matrix; every buffer is larger than L2."""
    w = synth.device_weights(41, n, k, dev)
    codes = torch.empty((n, k // 2), dtype=torch.uint8, device=dev)
    scales = torch.empty((n, k // 64), dtype=torch.float16, device=dev)
    w_hat = torch.empty((n, k), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()
    out = {}
    for name, call, algo in (
            ("quantize", lambda: nf4.nf4_quantize(w, codes, scales, stream), n * k * 4 + n * k // 2 + n * (k // 64) * 2),
            ("dequant", lambda: nf4.nf4_dequant(codes, scales, w_hat, stream), n * k // 2 + n * (k // 64) * 2 + n * k * 2)):
        iters = 20
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
        with torch.cuda.stream(stream):
            for _ in range(3):
                call()
            for a, b in evs:
                a.record(stream)
                call()
                b.record(stream)
        samples = []
        while not evs[-1][1].query():
            samples.append(sample_clocks(dev.index))
        torch.cuda.synchronize()
        t = statistics.median(a.elapsed_time(b) / 1e3 for a, b in evs)
        gbs = algo / t / 1e9
        out[name] = {"workload": f"{n} x {k} matrix", "gbs": round(gbs, 1), "frac_of_hbm": round(gbs / pk["hbm_gbs"], 4),
                     "us": round(t * 1e6, 2), "algorithmic_bytes": algo,
                     "kernel": "quantize_kernel" if name == "quantize" else "dequant_kernel",
                     "l2": "every buffer larger than L2", "clocks": clocks_summary(samples)}
    del w, codes, scales, w_hat
    torch.cuda.empty_cache()
    return out


def prefill_bench(nf4, synth, dev, pk):
    """TFLOP/s of the four 20B-shaped prefill linears (gate|up grouped) at M = 32 and M = 512."""
    wl = W.PREFILL_20B
    mats = {}
    for li, lin in enumerate(wl.linears):
        w = synth.device_weights(wl.seed * 100003 + li, lin.n, lin.k, dev, outlier_frac=wl.outlier_frac)
        mats[lin.name] = (lin,) + tuple(nf4.quantize(w))
        del w
    out = {}
    stream = torch.cuda.Stream(device=dev)
    groups = (("gate", "up"), ("down",), ("qkv",))
    for m in wl.tokens:
        xs = {k: synth.device_activations_bf16(99 + k, m, k, dev) for k in {l.k for l in wl.linears}}
        ys = {name: torch.empty((m, lin.n), dtype=torch.bfloat16, device=dev) for name, (lin, _, _) in mats.items()}
        torch.cuda.synchronize()  # weights and x are made on the default stream

        def step():
            for names in groups:
                lin = mats[names[0]][0]
                nf4.nf4_linear_grouped(xs[lin.k], [mats[n][1] for n in names], [mats[n][2] for n in names],
                                       [ys[n] for n in names], stream)

        with torch.cuda.stream(stream):
            step()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            step()
        times, _, samples = timed_replays(graph, stream, 50, 5, dev.index)
        t = statistics.median(times)
        flops = sum(2.0 * m * lin.n * lin.k for lin, _, _ in mats.values())
        tf = flops / t / 1e12
        packed = sum(lin.n * (lin.k // 2 + lin.k // 64 * 2) for lin, _, _ in mats.values())
        out[f"M{m}"] = {"tflops": round(tf, 2), "frac_of_bf16_peak": round(tf / pk["bf16_tflops"], 4),
                        "frac_of_bf16_sustained": round(tf / pk["bf16_tflops_sustained"], 4),
                        "peak_note": "burst peak: 50 replays of a sub-millisecond graph; sustained beside it",
                        "kernel": f"stream_kernel<{32 if m <= 32 else 256}> (tcgen05, dequant into tensor memory)",
                        "packed_gbs": round(packed / t / 1e9, 1), "ms": round(t * 1e3, 4),
                        "clocks": clocks_summary(samples)}
    return out


# ------------------------------------------------------------------------------------------------
# the oracle on the host cores (cpu_baseline and --impl reference)
# ------------------------------------------------------------------------------------------------
def oracle_sample(seconds_budget: float = 15.0):
    """Time the oracle's fp64 linear on one 3B-shaped layer (7 linears, M = 1) and express it as
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
    return gbs, threads, (f"{reps} pass(es) over one 3B-shaped layer (7 linears, {packed / 1e6:.1f} MB packed), "
                          f"M=1, fp64 oracle, {threads} threads")


def run_reference(args, rank, world):
    if rank != 0:
        return None
    budget = max(5.0, min(60.0, 0.05 * args.steps + 5.0))
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


def profile_linear(m: int, n: int, k: int) -> None:
    """Quantize one random n x k linear on the device and run nf4_linear four times (M = m), for
    profiler captures of a single kernel; prints nothing to time."""
    import nf4_weight_only_gb300 as nf4
    from nf4_weight_only_gb300 import build, synth
    build.build()
    nf4.load()
    dev = torch.device("cuda", 0)
    codes, scales = nf4.quantize(synth.device_weights(1, n, k, dev))
    x = synth.device_activations_bf16(2, m, k, dev)
    y = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
    for _ in range(4):
        nf4.nf4_linear(x, codes, scales, y)
    torch.cuda.synchronize()
    print(f"profile-linear M={m} N={n} K={k}: ok, device error word {nf4.nf4_check_device_error()}")


def profile_codec(n: int, k: int) -> None:
    """Quantize one random n x k matrix on the device and dequantize it, twice each, for profiler
    captures of the two codec kernels; prints nothing to time."""
    import nf4_weight_only_gb300 as nf4
    from nf4_weight_only_gb300 import build, synth
    build.build()
    nf4.load()
    dev = torch.device("cuda", 0)
    w = synth.device_weights(41, n, k, dev)
    for _ in range(2):
        codes, scales = nf4.quantize(w)
        w_hat = nf4.dequant(codes, scales)
    torch.cuda.synchronize()
    print(f"profile-codec N={n} K={k}: ok, {w_hat.shape[0]} rows")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--skip-prefill", action="store_true", help="skip the prefill, embedding, codec and overflow lines")
    ap.add_argument("--skip-cpu-baseline", action="store_true")
    ap.add_argument("--profile-codec", nargs=2, type=int, metavar=("N", "K"),
                    help="quantize and dequantize one N x K matrix (for single-kernel profiler captures)")
    ap.add_argument("--profile-linear", nargs=3, type=int, metavar=("M", "N", "K"),
                    help="run one M x N x K linear four times (for single-kernel profiler captures) and exit")
    args = ap.parse_args()
    if args.profile_linear:
        profile_linear(*args.profile_linear)
        return
    if args.profile_codec:
        profile_codec(*args.profile_codec)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":  # the oracle on host cores: rank 0 alone, no process group
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res))
        return
    if world > 1:
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        torch.distributed.init_process_group("nccl")
    if True:
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
