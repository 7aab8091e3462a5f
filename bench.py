#!/usr/bin/env python3
"""Benchmark of the NF4 weight-only linear layer on one GB300 (or N independent replicas).

Headline: NF4 GEMV (M = 1) HBM GB/s on the packed bytes over one decode pass of the 32B-shaped
weight sweep (hidden 5120, intermediate 27648, 64 layers, 16.58 GB of codes + scales resident in
HBM).  A step is one pass over every linear of every layer in dependency order -- per layer q|k|v
(one grouped launch, shared input), o, gate|up (grouped), down: 256 launches chained with
programmatic dependent launch and replayed from one CUDA graph.

Every other workload is reported beside it under "configs": the single 2048 x 2048 linear (weights
rotated over more than four L2 sizes of copies, the hot-L2 figure labelled apart), the 3B-shaped
decode pass, the 14B-shaped pass at M = 1, 4 and 8, and the 20B-shaped prefill at M = 32 and 512.
The device error word of the bounded pipeline waits is read after every timed region, and the
cpu_baseline leg checks sampled outputs of the headline's timed graph against the oracle.

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
HEADLINE = W.SWEEP_32B

# One decoder layer's linears in dependency order; names in one tuple read the same input.
LAYER_STEPS = (("q", "k", "v"), ("o",), ("gate", "up"), ("down",))


class BenchError(RuntimeError):
    pass


def traffic_per_launch(summary: str):
    """DRAM bytes per launch of the dominant kernel from a committed ncu summary (None if absent)."""
    import re
    path = os.path.join(ROOT, "profiles", summary)
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


def check_device_error(nf4, where: str) -> None:
    """The bounded pipeline waits record a code when one runs out (the launch's outputs are then
    unspecified): a timed region that saw one is not a measurement."""
    code = nf4.nf4_check_device_error()
    if code:
        raise BenchError(f"{where}: device error word {code} after the timed region")


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


def build_layers(nf4, synth, wl: W.Workload, dev, layers: int = None):
    """Quantize every linear of every layer on the device (fp32 weights drawn there, then freed)."""
    out = []
    for layer in range(wl.layers if layers is None else layers):
        mats = {}
        for li, lin in enumerate(wl.linears):
            w = synth.device_weights(wl.seed * 100003 + layer * 16 + li, lin.n, lin.k, dev,
                                     outlier_frac=wl.outlier_frac)
            codes, scales = nf4.quantize(w)
            del w
            mats[lin.name] = (lin, codes, scales)
        out.append(mats)
    torch.cuda.synchronize()
    return out


def run_pass(nf4, layers, xs, ys, stream):
    """One pass in dependency order: per layer q|k|v (grouped), o, gate|up (grouped), down."""
    for mats, yl in zip(layers, ys):
        for names in LAYER_STEPS:
            lin = mats[names[0]][0]
            if len(names) == 1:
                nf4.nf4_linear(xs[lin.k], mats[names[0]][1], mats[names[0]][2], yl[names[0]], stream)
            else:
                nf4.nf4_linear_grouped(xs[lin.k], [mats[n][1] for n in names], [mats[n][2] for n in names],
                                       [yl[n] for n in names], stream)


class DecodePass:
    """One decode pass of a layered workload at M tokens, captured in one CUDA graph.  Every y is a
    view of one flat buffer (each n is a multiple of 8, so every view stays 16-byte aligned), which
    the end-to-end step copies back in one transfer."""

    def __init__(self, nf4, synth, wl: W.Workload, m: int, dev, layers=None, x_seed: int = 77):
        self.nf4, self.wl, self.m, self.dev = nf4, wl, m, dev
        self.layers = layers if layers is not None else build_layers(nf4, synth, wl, dev)
        nl = len(self.layers)
        self.xs = {k: synth.device_activations_bf16(x_seed + k + 1000 * m, m, k, dev) for k in {l.k for l in wl.linears}}
        self.y_flat = torch.empty(nl * m * sum(lin.n for lin in wl.linears), dtype=torch.bfloat16, device=dev)
        self.ys, off = [], 0
        for mats in self.layers:
            yl = {}
            for name, (lin, _, _) in mats.items():
                yl[name] = self.y_flat[off:off + m * lin.n].view(m, lin.n)
                off += m * lin.n
            self.ys.append(yl)
        self.stream = torch.cuda.Stream(device=dev)
        torch.cuda.synchronize()  # x is drawn on the default stream
        with torch.cuda.stream(self.stream):
            run_pass(nf4, self.layers, self.xs, self.ys, self.stream)  # first call builds the table
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=self.stream):
            run_pass(nf4, self.layers, self.xs, self.ys, self.stream)
        torch.cuda.synchronize()
        self.launches = nl * len(LAYER_STEPS)
        self.packed = sum(lin.n * (lin.k // 2 + lin.k // 64 * 2) for lin in wl.linears) * nl
        self.algo = self.packed + nl * sum(2 * m * lin.k + 2 * m * lin.n for lin in wl.linears)
        self.flops = 2.0 * m * sum(lin.n * lin.k for lin in wl.linears) * nl

    def time(self, steps, warmup):
        per, total, samples = timed_replays(self.graph, self.stream, steps, warmup, self.dev.index)
        check_device_error(self.nf4, f"{self.wl.name} M={self.m}")
        return per, total, samples

    def e2e(self, steps, warmup):
        """The same graph with every x copied in from pinned host memory and all y copied back each
        step (the host side of a real decode step).  Returns (seconds per step, h2d, d2h bytes)."""
        xs_host = {k: v.cpu().pin_memory() for k, v in self.xs.items()}
        y_host = torch.empty(self.y_flat.shape, dtype=self.y_flat.dtype).pin_memory()

        def step():
            for k, h in xs_host.items():
                self.xs[k].copy_(h, non_blocking=True)
            self.graph.replay()
            y_host.copy_(self.y_flat, non_blocking=True)

        with torch.cuda.stream(self.stream):
            for _ in range(warmup):
                step()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(self.stream):
            e0.record(self.stream)
            for _ in range(steps):
                step()
            e1.record(self.stream)
        torch.cuda.synchronize()
        check_device_error(self.nf4, f"{self.wl.name} M={self.m} end to end")
        return e0.elapsed_time(e1) / 1e3 / steps, sum(2 * v.numel() for v in self.xs.values()), 2 * self.y_flat.numel()


M1_KERNEL = "gemv_kernel (CUDA-core GEMV, M <= 3) / narrow_kernel<1> (tcgen05, K past the GEMV's range)"


def decode_line(dp: DecodePass, steps, warmup, pk):
    per, total, samples = dp.time(steps, warmup)
    t = total / steps
    gbs = dp.packed / t / 1e9
    return {"workload": dp.wl.name.split(",")[0] + f", M={dp.m}", "M": dp.m, "layers": len(dp.layers),
            "launches_per_step": dp.launches, "packed_bytes_per_step": dp.packed, "ms_per_step": round(t * 1e3, 4),
            "packed_gbs": round(gbs, 1), "frac_of_hbm": round(gbs / pk["hbm_gbs"], 4),
            "tflops": round(dp.flops / t / 1e12, 3), "kernel": M1_KERNEL if dp.m <= 4 else "narrow_kernel<8> (tcgen05)",
            "clocks": clocks_summary(samples)}


def single_2048(nf4, synth, dev, pk, steps, warmup):
    """The single 2048 x 2048 linear at M = 1.  Its 2.2 MB of weights fit in L2, so the timed graph
    runs it over distinct copies rotating through more than four L2 sizes of memory (cold, the
    figure reported); the same graph over one copy gives the hot-L2 figure, labelled apart."""
    wl = W.SINGLE_2048
    lin = wl.linears[0]
    w = synth.device_weights(wl.seed * 100003, lin.n, lin.k, dev)
    codes, scales = nf4.quantize(w)
    del w
    packed = lin.n * (lin.k // 2 + lin.k // 64 * 2)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    copies = max(4, -(-4 * l2 // packed))
    cs = [(codes.clone(), scales.clone()) for _ in range(copies)]
    x = synth.device_activations_bf16(1000, 1, lin.k, dev)
    y = torch.empty((1, lin.n), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()
    out = {}
    for label, seq in (("rotated", cs), ("hot_l2", [cs[0]] * copies)):
        with torch.cuda.stream(stream):
            for c, s in seq[:2]:
                nf4.nf4_linear(x, c, s, y, stream)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for c, s in seq:
                nf4.nf4_linear(x, c, s, y, stream)
        per, total, samples = timed_replays(g, stream, max(3, steps // 20), warmup, dev.index)
        check_device_error(nf4, f"single 2048 {label}")
        t = total / max(3, steps // 20) / copies
        gbs = packed / t / 1e9
        out[label] = {"us_per_linear": round(t * 1e6, 3), "packed_gbs": round(gbs, 1),
                      "frac_of_hbm": round(gbs / pk["hbm_gbs"], 4), "clocks": clocks_summary(samples)}
    del cs
    return {"workload": wl.name, "copies": copies, "bytes_rotated": copies * packed, "l2_bytes": l2,
            "kernel": "gemv_kernel<1,1,2> (CUDA-core GEMV)", "packed_bytes": packed,
            "figure": "rotated (cold: distinct copies over > 4 x L2); hot_l2 is one copy replayed", **out}


def prefill_lines(nf4, synth, dev, pk, steps, warmup):
    """TFLOP/s of the four 20B-shaped prefill linears (gate|up grouped) at M = 32 and M = 512."""
    wl = W.PREFILL_20B
    layers = build_layers(nf4, synth, wl, dev)
    mats = layers[0]
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
        n = max(10, steps // 4)
        times, total, samples = timed_replays(graph, stream, n, warmup, dev.index)
        check_device_error(nf4, f"prefill M={m}")
        t = total / n
        flops = sum(2.0 * m * lin.n * lin.k for lin, _, _ in mats.values())
        tf = flops / t / 1e12
        packed = sum(lin.n * (lin.k // 2 + lin.k // 64 * 2) for lin, _, _ in mats.values())
        out[f"M{m}"] = {"workload": f"20B-shaped prefill, 4 linears, M={m}", "tflops": round(tf, 2),
                        "frac_of_bf16_peak": round(tf / pk["bf16_tflops"], 4),
                        "frac_of_bf16_sustained": round(tf / pk["bf16_tflops_sustained"], 4),
                        "peak_note": "burst peak: a sub-millisecond graph replayed; sustained beside it",
                        "kernel": "narrow_kernel<32> (tcgen05, small M)" if m <= 32 else
                                  "stream_kernel<256> (tcgen05 GEMM, dequant into tensor memory)",
                        "packed_gbs": round(packed / t / 1e9, 1), "frac_of_hbm": round(packed / t / 1e9 / pk["hbm_gbs"], 4),
                        "ms": round(t * 1e3, 4), "clocks": clocks_summary(samples)}
    return out


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
        check_device_error(nf4, "overflow ring")
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
    check_device_error(nf4, "embed")
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


# ------------------------------------------------------------------------------------------------
# the oracle on the host cores (cpu_baseline and --impl reference)
# ------------------------------------------------------------------------------------------------
def oracle_layer_sample(o, seed: int = 5):
    """One 32B-shaped layer (7 linears, M = 1) of random packed weights drawn on the host (the
    oracle's speed does not depend on the values), with x from the seeded generator."""
    from nf4_weight_only_gb300 import synth
    rng = np.random.default_rng(seed)
    out = []
    for lin in HEADLINE.linears:
        codes = rng.integers(0, 256, size=(lin.n, lin.k // 2), dtype=np.uint8)
        scales = (rng.random((lin.n, lin.k // 64), dtype=np.float32) * 0.09 + 0.01).astype(np.float16).view(np.uint16)
        out.append((lin, codes, scales, synth.activations_bf16(seed + lin.k, 1, lin.k)))
    return out


def time_oracle(o, sample, threads: int, budget_s: float, max_reps: int = 50):
    """Repeat the oracle's fp64 linear over `sample` until `budget_s` seconds have passed.
    Returns (packed GB/s, seconds, repetitions)."""
    packed = sum(lin.n * (lin.k // 2 + lin.k // 64 * 2) for lin, *_ in sample)
    reps, total = 0, 0.0
    while (total < budget_s or reps == 0) and reps < max_reps:
        t0 = time.perf_counter()
        for lin, codes, scales, x in sample:
            o.linear(x, codes, scales, nthreads=threads)
        total += time.perf_counter() - t0
        reps += 1
    return packed * reps / total / 1e9, total, reps


def cpu_baseline(o):
    """The oracle on this host's cores: all threads on a whole 32B-shaped layer, one thread on its q
    projection (a rate in the metric's unit; nothing is extrapolated)."""
    threads = os.cpu_count() or 1
    sample = oracle_layer_sample(o)
    gbs, secs, reps = time_oracle(o, sample, threads, 8.0)
    gbs1, secs1, reps1 = time_oracle(o, sample[:1], 1, 4.0)
    lin = sample[0][0]
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": (f"{reps} pass(es) over one 32B-shaped layer (7 linears, 259 MB packed, random codes), "
                       f"M=1, fp64 oracle, {threads} threads, {secs:.2f} s measured"),
            "extrapolated": False,
            "single_thread": {"value": round(gbs1, 4), "unit": "GB/s", "cores": 1,
                              "sample": f"{reps1} pass(es) over the {lin.k}->{lin.n} q projection, {secs1:.2f} s measured"}}


def check_sampled_outputs(nf4, o, dp: DecodePass, checks=((0, "q"), (0, "gate"), (-1, "down")), rows_per: int = 64,
                          seed: int = 7):
    """Sampled outputs of the timed graph against the oracle: for the listed (layer, linear) pairs,
    the same fp32 weights are drawn again on the device, the sampled rows copied to the host and
    quantized by the oracle (which must give the GPU's codes and scales bit for bit), and the oracle's
    linear on those codes and the generator's x must bound the GPU's outputs."""
    from nf4_weight_only_gb300 import synth
    wl = dp.wl
    rng = np.random.default_rng(seed)
    names = [lin.name for lin in wl.linears]
    worst, checked = 0.0, 0
    for layer, name in checks:
        layer = layer % len(dp.layers)
        li = names.index(name)
        lin, codes_d, scales_d = dp.layers[layer][name]
        rows = np.unique(np.concatenate([[0, lin.n - 1], rng.choice(lin.n, rows_per - 2, replace=False)]))
        w = synth.device_weights(wl.seed * 100003 + layer * 16 + li, lin.n, lin.k, dp.dev, outlier_frac=wl.outlier_frac)
        sel = torch.from_numpy(rows.astype(np.int64)).to(dp.dev)
        w_rows = w[sel].cpu().numpy()
        del w
        c_ref, s_ref = o.quantize(w_rows)
        if not (np.array_equal(codes_d[sel].cpu().numpy(), c_ref) and
                np.array_equal(scales_d[sel].cpu().view(torch.int16).numpy().view(np.uint16), s_ref)):
            raise BenchError(f"layer {layer} {name}: packed weights differ from the oracle's")
        x = dp.xs[lin.k].cpu().view(torch.int16).numpy().view(np.uint16)
        y64, mag = o.linear(x, c_ref, s_ref, nthreads=os.cpu_count() or 1)
        got = dp.ys[layer][name].cpu().view(torch.int16).numpy().view(np.uint16)[:, rows]
        import oracle as oracle_mod
        ok, ratio, mask = oracle_mod.within_tolerance(got, y64, mag)
        if not ok:
            raise BenchError(f"layer {layer} {name}: {np.count_nonzero(~mask)} sampled outputs outside the bound")
        worst = max(worst, float(ratio))
        checked += got.size
    return {"outputs_checked": int(checked), "worst_error_over_bound": round(worst, 4), "ok": True,
            "linears": [f"layer {l % len(dp.layers)} {n}" for l, n in checks]}


def run_reference(args, rank, world):
    """The oracle, as it stands, on this host's cores; a step is one 32B-shaped layer (7 linears) of
    the headline pass, timed in full."""
    if rank != 0:
        return None
    import oracle
    o = oracle.default()
    threads = os.cpu_count() or 1
    sample = oracle_layer_sample(o)
    packed = sum(lin.n * (lin.k // 2 + lin.k // 64 * 2) for lin, *_ in sample)
    for _ in range(args.warmup):
        time_oracle(o, sample, threads, 0.0, max_reps=1)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        time_oracle(o, sample, threads, 0.0, max_reps=1)
        times.append(time.perf_counter() - t0)
    total = sum(times)
    gbs = packed * args.steps / total / 1e9
    return {
        "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(total / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
        "config": {"workload": HEADLINE.name, "step": "one layer (7 linears, 259 MB packed) of the 64-layer pass, timed in full"},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": f"{args.steps} steps of one 32B-shaped layer, fp64 oracle, {threads} threads, "
                                   f"{total:.2f} s measured", "extrapolated": False},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_ours(args, rank, world):
    import nf4_weight_only_gb300 as nf4
    from nf4_weight_only_gb300 import build, synth

    build.build()
    nf4.load()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    pk = peaks()
    only = set(args.only.split(",")) if args.only else None

    def want(name):
        return only is None or name in only

    result = {}
    if want("headline"):
        dp = DecodePass(nf4, synth, HEADLINE, 1, dev,
                        layers=build_layers(nf4, synth, HEADLINE, dev, layers=args.layers), x_seed=377)
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        per, total_s, samples = dp.time(args.steps, args.warmup)
        if world > 1:
            torch.distributed.barrier()
            total_s = max_over_ranks(total_s, dev)
        step_s = statistics.median(per)
        gbs = job_throughput(dp.packed, args.steps, world, total_s) / 1e9
        per_launch_s = total_s / args.steps / dp.launches
        achieved = (dp.algo / dp.launches) / per_launch_s / 1e9
        e2e_s, h2d, d2h = dp.e2e(max(3, min(args.steps, 50)), max(3, args.warmup))
        result = {
            "metric": METRIC, "value": round(gbs, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(step_s * 1e3, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": HEADLINE.name if args.layers is None else f"{HEADLINE.name} (first {args.layers} layers)",
                       "M": 1, "launches_per_step": dp.launches,
                       "launch_structure": "per layer: q|k|v grouped, o, gate|up grouped, down (PDL-chained)",
                       "packed_bytes_per_step": dp.packed,
                       "l2": f"inputs larger than L2 ({dp.packed / 1e9:.2f} GB of packed weights per step)",
                       "graph": "one CUDA graph per step", "peak_source": pk["source"]},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": round(achieved / pk["hbm_gbs"], 4),
                         "traffic": traffic_per_launch("gemv_decode_32b_launch_list.md"),
                         "algorithmic_bytes_per_launch": int(dp.algo / dp.launches), "kernel": M1_KERNEL,
                         "note": "algorithmic bytes (codes+scales+x+y) per launch / average launch time over the "
                                 "timed steps, inter-launch gaps included; peak of measured"},
            "packed_frac_of_hbm": round(gbs / world / pk["hbm_gbs"], 4),
            "e2e": {"value": round(dp.packed / e2e_s / 1e9, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "gpu_launches": dp.launches * args.steps,
            "clocks": clocks_summary(samples),
        }
        if rank == 0 and not args.skip_cpu_baseline:
            import oracle
            o = oracle.default()
            result["cpu_baseline"] = cpu_baseline(o)
            result["output_check"] = check_sampled_outputs(nf4, o, dp)
        del dp
        torch.cuda.empty_cache()
    configs = {}
    steps_sub, warm_sub = max(5, args.steps // 2), max(3, args.warmup)
    if want("c1"):
        configs["single_2048"] = single_2048(nf4, synth, dev, pk, args.steps, warm_sub)
    if want("c2"):
        dp = DecodePass(nf4, synth, W.DECODE_3B, 1, dev)
        configs["decode_3b_M1"] = decode_line(dp, steps_sub, warm_sub, pk)
        del dp
        torch.cuda.empty_cache()
    if want("c3"):
        layers = build_layers(nf4, synth, W.DECODE_14B, dev)
        for m in W.DECODE_14B.tokens:
            dp = DecodePass(nf4, synth, W.DECODE_14B, m, dev, layers=layers, x_seed=177)
            configs[f"decode_14b_M{m}"] = decode_line(dp, steps_sub, warm_sub, pk)
            del dp
        del layers
        torch.cuda.empty_cache()
    if want("c5"):
        for k, v in prefill_lines(nf4, synth, dev, pk, steps_sub, warm_sub).items():
            configs[f"prefill_20b_{k}"] = v
        torch.cuda.empty_cache()
    if configs:
        result["configs"] = configs
    if want("codec"):
        result.update(codec_bench(nf4, synth, dev, pk))
    if want("embed"):
        result["embed"] = embed_bench(nf4, synth, dev, pk)
    if want("overflow"):
        result["overflow"] = overflow_bench(nf4, synth, dev)
    return result


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
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--only", default=None,
                    help="comma-separated subset of headline,c1,c2,c3,c5,codec,embed,overflow (default: all)")
    ap.add_argument("--layers", type=int, default=None,
                    help="run only the first N layers of the headline workload (for profiler captures)")
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
    try:
        res = run_ours(args, rank, world)
    except BenchError as e:
        if rank == 0:
            print(json.dumps({"metric": METRIC, "value": None, "error": str(e)}))
        sys.exit(1)
    if rank == 0 and res:
        print(json.dumps(res))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
