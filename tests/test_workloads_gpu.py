"""Full-size workloads in the launch structure the bench times, checked against the oracle.

Every workload is built as the bench builds it: weights from the seeded device generator
(`synth.device_weights`, keyed by workload seed, layer and linear), quantized by `nf4_quantize`, and
each layer run as q|k|v (grouped), o, gate|up (grouped), down.  The 3B-shaped decode pass is
captured in one CUDA graph and replayed, as in the bench.  The checks never take an input from the
CUDA path.  For a checked linear the test draws the same fp32 weights again, copies the sampled rows
to the host, and quantizes them with the oracle.  The GPU codes and scales of those rows must equal
the oracle's bit for bit (quantize parity).  The oracle's linear then runs on the oracle's own codes
and on x from the seeded generator, and every sampled output must lie within the bound
|y - y64| <= 2^-8 |y64| + 2^-12 sum_k |x_k w_k|.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import bench
import oracle
from gpu_util import DEV, dev_to_bits, f16_dev_to_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nf4():
    import nf4_weight_only_gb300 as m
    from nf4_weight_only_gb300 import build
    build.build()
    m.load()
    return m


@pytest.fixture(scope="module")
def o():
    return oracle.default()


def _device_error(nf4) -> int:
    """Reads and clears the device error word of the bounded pipeline waits (0 = none)."""
    import ctypes
    lib = nf4.load()
    lib.nf4_check_device_error.argtypes = [ctypes.POINTER(ctypes.c_int)]
    lib.nf4_check_device_error.restype = ctypes.c_int
    code = ctypes.c_int(-1)
    assert lib.nf4_check_device_error(ctypes.byref(code)) == 0
    return code.value


def _check_rows(nf4, o, wl, layer, li, lin, codes_d, scales_d, x_d, y_d, rows):
    """Quantize parity and linear parity of one linear of one layer on the listed output rows."""
    from nf4_weight_only_gb300 import synth
    w = synth.device_weights(wl.seed * 100003 + layer * 16 + li, lin.n, lin.k, DEV, outlier_frac=wl.outlier_frac)
    sel = torch.from_numpy(rows.astype(np.int64)).to(DEV)
    w_rows = w[sel].cpu().numpy()
    del w
    c_ref, s_ref = o.quantize(w_rows)
    where = f"{wl.name}: layer {layer} {lin.name}"
    assert np.array_equal(codes_d[sel].cpu().numpy(), c_ref), f"{where}: codes differ from the oracle"
    assert np.array_equal(f16_dev_to_bits(scales_d[sel]), s_ref), f"{where}: scales differ from the oracle"
    y64, mag = o.linear(dev_to_bits(x_d), c_ref, s_ref, nthreads=16)
    got = dev_to_bits(y_d)[:, rows]
    ok, ratio, mask = oracle.within_tolerance(got, y64, mag)
    assert ok, f"{where}: {np.count_nonzero(~mask)} of {mask.size} outputs outside tolerance (worst {ratio:.3f})"
    return ratio


def _rows(rng, n, count):
    """`count` distinct rows of n, always with the first and the last."""
    if count >= n:
        return np.arange(n)
    pick = rng.choice(np.arange(1, n - 1), size=max(count - 2, 0), replace=False)
    return np.unique(np.concatenate([[0, n - 1], pick]))


def _run_pass(nf4, layers, xs, ys, stream):
    for mats, yl in zip(layers, ys):
        for names in bench.LAYER_STEPS:
            lin = mats[names[0]][0]
            if len(names) == 1:
                nf4.nf4_linear(xs[lin.k], mats[names[0]][1], mats[names[0]][2], yl[names[0]], stream)
            else:
                nf4.nf4_linear_grouped(xs[lin.k], [mats[n][1] for n in names], [mats[n][2] for n in names],
                                       [yl[n] for n in names], stream)


def _check_pass(nf4, o, wl, layers, xs, ys, full_layers, rows_full, rows_other, seed):
    rng = np.random.default_rng(seed)
    worst = 0.0
    for layer in range(wl.layers):
        count = rows_full if layer in full_layers else rows_other
        for li, lin in enumerate(wl.linears):
            _, codes_d, scales_d = layers[layer][lin.name]
            rows = _rows(rng, lin.n, count)
            worst = max(worst, _check_rows(nf4, o, wl, layer, li, lin, codes_d, scales_d, xs[lin.k],
                                           ys[layer][lin.name], rows))
    return worst


def _empty_outputs(layers, m):
    """y buffers filled with a NaN pattern, so that an output the pass never writes fails the check."""
    return [{name: torch.full((m, lin.n), float("nan"), dtype=torch.bfloat16, device=DEV)
             for name, (lin, _, _) in mats.items()} for mats in layers]


def test_decode_3b_pass_graph(nf4, o):
    """3B-shaped decode (36 layers, M = 1): the bench's 144 PDL-chained launches captured in one CUDA
    graph and replayed.  Layers 0 and 35 are checked on every output row, every other layer on 24
    rows of each linear (with the first and the last)."""
    from nf4_weight_only_gb300 import synth, workloads as W
    wl = W.DECODE_3B
    layers = bench.build_layers(nf4, synth, wl, DEV)
    xs = {k: synth.device_activations_bf16(77 + k, 1, k, DEV) for k in {l.k for l in wl.linears}}
    ys = _empty_outputs(layers, 1)
    stream = torch.cuda.Stream(device=DEV)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        _run_pass(nf4, layers, xs, ys, stream)  # warm-up (kernel attributes, tensor maps) before the capture
    torch.cuda.synchronize()
    ys = _empty_outputs(layers, 1)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        _run_pass(nf4, layers, xs, ys, stream)
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()
    assert _device_error(nf4) == 0
    _check_pass(nf4, o, wl, layers, xs, ys, {0, wl.layers - 1}, 1 << 30, 24, seed=36)


@pytest.mark.parametrize("m", [1, 4, 8])
def test_decode_14b_pass(nf4, o, m):
    """14B-shaped decode (48 layers) at M = 1, 4 and 8 in the bench's launch structure on one stream:
    layers 0 and 47 checked on 256 rows of each linear, every other layer on 8."""
    from nf4_weight_only_gb300 import synth, workloads as W
    wl = W.DECODE_14B
    layers = _layers_14b(nf4)
    xs = {k: synth.device_activations_bf16(177 + k + 1000 * m, m, k, DEV) for k in {l.k for l in wl.linears}}
    ys = _empty_outputs(layers, m)
    stream = torch.cuda.Stream(device=DEV)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        _run_pass(nf4, layers, xs, ys, stream)
    torch.cuda.synchronize()
    assert _device_error(nf4) == 0
    _check_pass(nf4, o, wl, layers, xs, ys, {0, wl.layers - 1}, 256, 8, seed=48 + m)


_cache = {}


def _layers_14b(nf4):
    """The 14B-shaped layers (7 GB packed), quantized once for the three token counts."""
    from nf4_weight_only_gb300 import synth, workloads as W
    if "14b" not in _cache:
        _cache.clear()
        torch.cuda.empty_cache()
        _cache["14b"] = bench.build_layers(nf4, synth, W.DECODE_14B, DEV)
    return _cache["14b"]


def test_sweep_32b_pass(nf4, o):
    """32B-shaped sweep (64 layers, 16.6 GB packed, M = 1), the bench's headline: its 256 PDL-chained
    launches captured in one CUDA graph and replayed; layers 0 and 63 checked on 256 rows of each
    linear, every other layer on 4."""
    from nf4_weight_only_gb300 import synth, workloads as W
    _cache.clear()
    torch.cuda.empty_cache()
    wl = W.SWEEP_32B
    layers = bench.build_layers(nf4, synth, wl, DEV)
    xs = {k: synth.device_activations_bf16(377 + k + 1000, 1, k, DEV) for k in {l.k for l in wl.linears}}
    stream = torch.cuda.Stream(device=DEV)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        _run_pass(nf4, layers, xs, _empty_outputs(layers, 1), stream)
    torch.cuda.synchronize()
    ys = _empty_outputs(layers, 1)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        _run_pass(nf4, layers, xs, ys, stream)
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()
    assert _device_error(nf4) == 0
    _check_pass(nf4, o, wl, layers, xs, ys, {0, wl.layers - 1}, 256, 4, seed=64)
    del layers, graph
    torch.cuda.empty_cache()


@pytest.mark.parametrize("m", [32, 512])
def test_prefill_20b_graph(nf4, o, m):
    """20B-shaped prefill (1% outlier weights) at M = 32 and 512: gate|up grouped, down, qkv, captured
    in one CUDA graph and replayed as the bench does; 96 rows of each linear checked for all M tokens."""
    from nf4_weight_only_gb300 import synth, workloads as W
    wl = W.PREFILL_20B
    layers = bench.build_layers(nf4, synth, wl, DEV)
    xs = {k: synth.device_activations_bf16(99 + k, m, k, DEV) for k in {l.k for l in wl.linears}}
    groups = (("gate", "up"), ("down",), ("qkv",))
    stream = torch.cuda.Stream(device=DEV)

    def step(ys):
        for names in groups:
            lin = layers[0][names[0]][0]
            nf4.nf4_linear_grouped(xs[lin.k], [layers[0][n][1] for n in names], [layers[0][n][2] for n in names],
                                   [ys[0][n] for n in names], stream)

    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        step(_empty_outputs(layers, m))
    torch.cuda.synchronize()
    ys = _empty_outputs(layers, m)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step(ys)
    graph.replay()
    torch.cuda.synchronize()
    assert _device_error(nf4) == 0
    _check_pass(nf4, o, wl, layers, xs, ys, {0}, 96, 96, seed=20 + m)
