"""CUDA path (through the C ABI) against the CPU oracle, element by element.

quantize and dequant must be bit-exact; the linear must meet the per-element bound
|y - y64| <= 2^-8 |y64| + 2^-12 sum_k |x_k w_k|.
"""
import multiprocessing as mp
import os

import numpy as np
import pytest
import torch

import oracle
import oracle_pins as P
from gpu_util import DEV, Guarded, bf16_to_dev, dev_to_bits, f16_dev_to_bits

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


def gpu_quantize(nf4, w: np.ndarray):
    codes, scales = nf4.quantize(torch.from_numpy(w).to(DEV))
    return codes, scales


# ------------------------------------------------------------------------------------------------
# quantize
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("n,k,seed,outliers", [
    (2048, 2048, 0, 0.0),      # the single 2048x2048 linear
    (1, 64, 1, 0.0), (7, 128, 2, 0.0), (257, 320, 3, 0.0), (33, 2112, 4, 0.0),
    (300, 6144, 5, 0.01),      # 20B-prefill-style outliers
])
def test_quantize_bit_exact(nf4, o, n, k, seed, outliers):
    from nf4_weight_only_gb300 import synth
    w = synth.weights(seed, n, k, outlier_frac=outliers)
    w[0, :64] = 0.0                # an all-zero group
    if k >= 128:
        w[0, 64:128] = -0.0        # an all-zero group of negative zeros (code 7 as well)
    if n > 1:
        w[1, 64:128] *= 1e-6       # tiny scale (fp16 subnormal range)
    if n > 2 and k >= 128:
        # absmax below 2^-120 (fp32 subnormal weights): the kernel's fast path steps aside for the
        # exact division on every weight of such a group; the fp16 scale rounds to zero
        w[2, 64:128] = (w[2, 64:128] * 1e-37).astype(np.float32)
    codes, scales = gpu_quantize(nf4, w)
    c_ref, s_ref = o.quantize(w)
    assert np.array_equal(f16_dev_to_bits(scales), s_ref)
    assert np.array_equal(codes.cpu().numpy(), c_ref)


def _oracle_codes(args):
    lo, hi = args
    keys = np.arange(lo, hi, dtype=np.int64)
    bits = np.where(keys >= 0, keys, 0x80000000 | (-keys)).astype(np.uint32)
    return lo, oracle.default().nf4_code(bits.view(np.float32))


def test_quantize_every_r_in_unit_interval(nf4):
    """Every binary32 r in [-1, 1]: groups whose first weight is 1.0 have s = 1 exactly, so the
    other 63 weights are their own normalised values r and the kernel's code must equal the
    oracle's nearest code of r."""
    lo, hi = P.ordered_key(np.float32(-1.0)), P.ordered_key(np.float32(1.0)) + 1
    per_group = 63
    chunk = per_group * (1 << 18)  # 16.5M values per chunk
    starts = list(range(lo, hi, chunk))
    ctx = mp.get_context("spawn")
    with ctx.Pool(min(16, os.cpu_count() or 1)) as pool:
        jobs = pool.imap(_oracle_codes, [(a, min(a + chunk, hi)) for a in starts])
        for a in starts:
            b = min(a + chunk, hi)
            keys = np.arange(a, b, dtype=np.int64)
            bits = np.where(keys >= 0, keys, 0x80000000 | (-keys)).astype(np.uint32)
            groups = (bits.size + per_group - 1) // per_group
            w = np.zeros((groups, 64), np.float32)
            w[:, 0] = 1.0
            flat = w[:, 1:].reshape(-1)
            flat[:bits.size] = bits.view(np.float32)
            w[:, 1:] = flat.reshape(groups, per_group)
            codes, scales = gpu_quantize(nf4, w)
            got = P.unpack_low_nibble_first(codes.cpu().numpy())[:, 1:].reshape(-1)[:bits.size]
            a2, want = next(jobs)
            assert a2 == a
            bad = np.flatnonzero(got != want)
            assert bad.size == 0, f"code differs at r={bits.view(np.float32)[bad[0]]!r}: gpu {got[bad[0]]} oracle {want[bad[0]]}"
            assert np.all(f16_dev_to_bits(scales) == 0x3C00)


def test_quantize_near_thresholds_any_scale(nf4, o):
    """Normalised values w / s within a few ulps of every decision threshold, for 4096 random
    scales s (log-uniform in [1e-3, 1e3], none a power of two): the kernel divides by an approximate
    reciprocal first and must hand each of these weights to the exact division, so its codes equal
    the oracle's for all of them."""
    rng = np.random.default_rng(77)
    mids = P.decision_thresholds(P.qlora_published_table()).astype(np.float64)  # the 15 fp32 thresholds
    groups = 4096
    s = np.exp(rng.uniform(np.log(1e-3), np.log(1e3), groups)).astype(np.float32)
    s = np.where(np.frexp(s)[0] == 0.5, np.nextafter(s, np.float32(2.0)), s).astype(np.float32)
    idx = rng.integers(0, 15, (groups, 63))
    ulp = rng.integers(-40, 41, (groups, 63)).astype(np.float64)
    r = mids[idx] * (1.0 + ulp * 2.0 ** -23)
    w = np.empty((groups, 64), np.float32)
    w[:, 0] = s
    w[:, 1:] = (r * s[:, None].astype(np.float64)).astype(np.float32)
    w = w.reshape(512, 8 * 64)
    codes, scales = gpu_quantize(nf4, w)
    c_ref, s_ref = o.quantize(w)
    assert np.array_equal(f16_dev_to_bits(scales), s_ref)
    assert np.array_equal(codes.cpu().numpy(), c_ref)


def test_quantize_large_sampled_rows(nf4, o):
    """A 5120 x 27648 matrix (the 32B-shaped down projection) generated on the device: sampled rows
    copied back as fp32 are re-quantized by the oracle."""
    from nf4_weight_only_gb300 import synth
    w = synth.device_weights(123, 5120, 27648, DEV)
    codes, scales = nf4.quantize(w)
    rows = np.array([0, 1, 2047, 4095, 5119])
    w_rows = w[rows].cpu().numpy()
    c_ref, s_ref = o.quantize(w_rows)
    assert np.array_equal(codes[rows].cpu().numpy(), c_ref)
    assert np.array_equal(f16_dev_to_bits(scales[rows]), s_ref)


# ------------------------------------------------------------------------------------------------
# dequant
# ------------------------------------------------------------------------------------------------
def test_dequant_every_code_and_scale(nf4, o):
    """All 16 codes against all 65536 fp16 scale patterns (non-finite ones included: both sides
    compute the same IEEE product; NaN payloads are compared as NaN only)."""
    scale_bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    row = np.array([c | ((15 - c) << 4) for c in range(16)] * 2, np.uint8)
    codes = np.tile(row, (scale_bits.size, 1))
    w_hat = nf4.dequant(torch.from_numpy(codes).to(DEV),
                        torch.from_numpy(scale_bits.view(np.int16)).view(torch.float16).to(DEV)[:, None].contiguous())
    got = dev_to_bits(w_hat)
    want = o.dequant(codes, scale_bits[:, None])
    gnan = (got & 0x7F80 == 0x7F80) & (got & 0x7F != 0)
    wnan = (want & 0x7F80 == 0x7F80) & (want & 0x7F != 0)
    assert np.array_equal(gnan, wnan)
    assert np.array_equal(got[~gnan], want[~wnan])


@pytest.mark.parametrize("n,k,seed", [(2048, 2048, 0), (1, 64, 1), (257, 320, 2), (64, 11008, 3)])
def test_dequant_bit_exact(nf4, o, n, k, seed):
    from nf4_weight_only_gb300 import synth
    w = synth.weights(seed, n, k, outlier_frac=0.01)
    c_ref, s_ref = o.quantize(w)
    out = Guarded((n, k), torch.bfloat16)
    nf4.nf4_dequant(torch.from_numpy(c_ref).to(DEV),
                    torch.from_numpy(s_ref.view(np.int16)).view(torch.float16).to(DEV), out.t)
    assert np.array_equal(dev_to_bits(out.t), o.dequant(c_ref, s_ref))
    assert out.canaries_intact()


# ------------------------------------------------------------------------------------------------
# linear
# ------------------------------------------------------------------------------------------------
def run_linear(nf4, x_bits, codes, scales):
    m, n = x_bits.shape[0], codes.shape[0]
    out = Guarded((m, n), torch.bfloat16)
    nf4.nf4_linear(bf16_to_dev(x_bits), torch.from_numpy(codes).to(DEV),
                   torch.from_numpy(scales.view(np.int16)).view(torch.float16).to(DEV), out.t)
    torch.cuda.synchronize()
    assert out.canaries_intact(), "nf4_linear wrote outside y"
    return dev_to_bits(out.t)


def check_linear(nf4, o, m, n, k, seed, outliers=0.0, nthreads=16):
    from nf4_weight_only_gb300 import synth
    w = synth.weights(seed, n, k, outlier_frac=outliers)
    x = synth.activations_bf16(seed + 1000, m, k)
    codes, scales = o.quantize(w)
    y = run_linear(nf4, x, codes, scales)
    y64, mag = o.linear(x, codes, scales, nthreads=nthreads)
    ok, ratio, mask = oracle.within_tolerance(y, y64, mag)
    assert ok, f"M={m} N={n} K={k}: {np.count_nonzero(~mask)} outside tolerance, worst ratio {ratio:.3f}"
    return ratio


@pytest.mark.parametrize("m", [1, 2, 3, 4, 5, 8])
@pytest.mark.parametrize("n,k", [(1, 64), (7, 128), (257, 2048), (96, 5120), (40, 11008), (24, 13824)])
def test_linear_small_shapes(nf4, o, m, n, k):
    check_linear(nf4, o, m, n, k, seed=n * 31 + k)


def test_linear_single_2048(nf4, o):
    """The single 2048 x 2048 linear, M = 1, seed 0."""
    from nf4_weight_only_gb300 import synth
    w = synth.weights(0, 2048, 2048)
    x = synth.activations_bf16(1000, 1, 2048)
    codes, scales = o.quantize(w)
    y = run_linear(nf4, x, codes, scales)
    y64, mag = o.linear(x, codes, scales, nthreads=16)
    ok, ratio, _ = oracle.within_tolerance(y, y64, mag)
    assert ok, ratio


def test_linear_k27648_m1(nf4, o):
    check_linear(nf4, o, 1, 160, 27648, seed=5)


@pytest.mark.parametrize("n,k", [(1000, 2112), (4099, 5120), (513, 3072), (700, 11008), (3000, 15360)])
def test_linear_m1_two_lanes_per_group(nf4, o, n, k):
    """M = 1 where two lanes per group leave fewer lanes idle than one (33, 80, 48, 172 and 240
    groups; 240 is 15 slices of 16, one short of the most a CTA holds): whole slices, a slice with
    a single group, several row blocks per CTA."""
    check_linear(nf4, o, 1, n, k, seed=n + 3 * k)


def test_linear_m33_outliers(nf4, o):
    check_linear(nf4, o, 33, 130, 6144, seed=6, outliers=0.01)


def test_linear_zero_input_and_zero_rows(nf4, o):
    from nf4_weight_only_gb300 import synth
    w = synth.weights(9, 64, 512)
    w[3] = 0.0
    codes, scales = o.quantize(w)
    x = np.zeros((2, 512), np.uint16)
    y = run_linear(nf4, x, codes, scales)
    assert np.all((y & 0x7FFF) == 0)
    x = synth.activations_bf16(10, 1, 512)
    y = run_linear(nf4, x, codes, scales)
    assert (y[0, 3] & 0x7FFF) == 0


def test_linear_deterministic(nf4, o):
    from nf4_weight_only_gb300 import synth
    w = synth.weights(11, 300, 5120)
    x = synth.activations_bf16(12, 3, 5120)
    codes, scales = o.quantize(w)
    y1 = run_linear(nf4, x, codes, scales)
    y2 = run_linear(nf4, x, codes, scales)
    assert np.array_equal(y1, y2)


def _entry_point_calls(nf4):
    """One call of every compute entry point (GEMV, both streaming kernels, grouped, quantize,
    dequant, embed), inputs and outputs allocated up front; returns a function(stream)."""
    from nf4_weight_only_gb300 import synth
    w = synth.device_weights(800, 512, 2048, DEV)
    codes = torch.empty((512, 1024), dtype=torch.uint8, device=DEV)
    scales = torch.empty((512, 32), dtype=torch.float16, device=DEV)
    nf4.nf4_quantize(w, codes, scales)
    w_hat = torch.empty((512, 2048), dtype=torch.bfloat16, device=DEV)
    xs = {m: synth.device_activations_bf16(801 + m, m, 2048, DEV) for m in (1, 8, 300)}
    ys = {m: torch.empty((m, 512), dtype=torch.bfloat16, device=DEV) for m in (1, 8, 300)}
    g_ys = [torch.empty((8, 512), dtype=torch.bfloat16, device=DEV) for _ in range(2)]
    ids = torch.arange(0, 512, 7, dtype=torch.int32, device=DEV)
    rows = torch.empty((ids.numel(), 2048), dtype=torch.bfloat16, device=DEV)
    torch.cuda.synchronize()

    def calls(stream):
        nf4.nf4_quantize(w, codes, scales, stream)
        nf4.nf4_dequant(codes, scales, w_hat, stream)
        for m in (1, 8, 300):
            nf4.nf4_linear(xs[m], codes, scales, ys[m], stream)
        nf4.nf4_linear_grouped(xs[8], [codes, codes], [scales, scales], g_ys, stream)
        nf4.nf4_embed(ids, codes, scales, rows, stream)
    return calls


def test_calls_neither_sync_nor_allocate(nf4):
    """After the first call on a device, no entry point waits for the device or allocates device
    memory: queued behind a ~100 ms device sleep, every call returns to the host at once, and the
    device's free memory is the same after 20 rounds of all of them."""
    import time
    calls = _entry_point_calls(nf4)
    stream = torch.cuda.Stream(device=DEV)
    calls(stream)  # first use per device: builds the constant table (one host wait, documented)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info(DEV)
    with torch.cuda.stream(stream):
        torch.cuda._sleep(200_000_000)  # ~100 ms of device time ahead of the calls
        t0 = time.perf_counter()
        for _ in range(20):
            calls(stream)
        host_s = time.perf_counter() - t0
    assert not stream.query(), "the sleep ended before the calls returned: the host waited"
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info(DEV)
    assert host_s < 0.05, f"140 calls took {host_s * 1e3:.1f} ms on the host (a synchronising call?)"
    assert free1 == free0, f"device free memory changed by {free0 - free1} bytes"
    assert device_error(nf4) == 0


_DETERMINISM_SCRIPT = r"""
import hashlib, torch
import nf4_weight_only_gb300 as nf4
from nf4_weight_only_gb300 import synth
nf4.load()
dev = torch.device("cuda", 0)
h = hashlib.sha256()
for m, n, k, seed in [(1, 1000, 5120, 0), (3, 300, 11008, 1), (8, 2048, 6144, 2), (300, 777, 2048, 3)]:
    codes, scales = nf4.quantize(synth.device_weights(810 + seed, n, k, dev))
    x = synth.device_activations_bf16(820 + seed, m, k, dev)
    y = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
    nf4.nf4_linear(x, codes, scales, y)
    g = [torch.empty((m, n), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    nf4.nf4_linear_grouped(x, [codes, codes], [scales, scales], g)
    torch.cuda.synchronize()
    for t in (codes, scales, y, g[0], g[1]):
        h.update(t.cpu().view(torch.uint8).numpy().tobytes() if t.dtype == torch.uint8
                 else t.cpu().view(torch.int16).numpy().tobytes())
print("HASH", h.hexdigest())
"""


def test_outputs_identical_across_fresh_processes(nf4):
    """The same inputs give the same output bytes in three fresh processes (GEMV, both streaming
    kernels, grouped launches, quantize)."""
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    hashes = []
    for _ in range(3):
        r = subprocess.run([sys.executable, "-c", _DETERMINISM_SCRIPT], cwd=root, capture_output=True, text=True,
                           timeout=300)
        assert r.returncode == 0, r.stderr[-2000:]
        hashes.append([l for l in r.stdout.splitlines() if l.startswith("HASH ")][-1])
    assert len(set(hashes)) == 1, hashes


_FIRST_CALL_CAPTURED_SCRIPT = r"""
import torch
import nf4_weight_only_gb300 as nf4
from nf4_weight_only_gb300 import synth
nf4.load()
dev = torch.device("cuda", 0)
cases = []
for m, n, k, seed in [(1, 1000, 5120, 0), (8, 640, 2048, 1), (300, 384, 1024, 2)]:
    codes, scales = synth.device_packed(830 + seed, n, k, dev)  # torch only: no library call yet
    x = synth.device_activations_bf16(840 + seed, m, k, dev)
    cases.append((x, codes, scales, torch.empty((m, n), dtype=torch.bfloat16, device=dev)))
torch.cuda.synchronize()
s = torch.cuda.Stream()
g = torch.cuda.CUDAGraph()
with torch.cuda.graph(g, stream=s):  # the process's first library calls, captured
    for x, codes, scales, y in cases:
        nf4.nf4_linear(x, codes, scales, y, stream=s)
g.replay()
torch.cuda.synchronize()
for x, codes, scales, y in cases:
    ref = torch.empty_like(y)
    nf4.nf4_linear(x, codes, scales, ref)
    torch.cuda.synchronize()
    assert torch.equal(ref.view(torch.int16), y.view(torch.int16))
print("OK", nf4.nf4_check_device_error())
"""


def test_first_calls_may_be_captured(nf4):
    """In a fresh process the first library calls (GEMV, small-M and GEMM-form kernels) are made
    inside a CUDA graph capture: the replayed graph gives the same bytes as eager calls afterwards
    (no call needs one-time device work outside a capture)."""
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _FIRST_CALL_CAPTURED_SCRIPT], cwd=root, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert "OK 0" in r.stdout, r.stdout[-500:]


def test_first_call_of_a_fresh_host_thread(nf4, o):
    """A host thread whose first CUDA work is a library call on the tensor-core paths (M = 8 and
    M = 300; their launch encodes tensor maps through the driver, which needs a current context)
    gets the same bytes as the main thread."""
    import threading
    from nf4_weight_only_gb300 import synth
    cases = []
    for m, n, k, seed in [(8, 640, 2048, 0), (300, 384, 1024, 1)]:
        codes, scales = nf4.quantize(synth.device_weights(960 + seed, n, k, DEV))
        x = synth.device_activations_bf16(961 + seed, m, k, DEV)
        ref = torch.empty((m, n), dtype=torch.bfloat16, device=DEV)
        nf4.nf4_linear(x, codes, scales, ref)
        cases.append((x, codes, scales, ref, torch.empty_like(ref)))
    torch.cuda.synchronize()
    for x, codes, scales, ref, out in cases:
        errors = []

        def worker():
            try:
                nf4.nf4_linear(x, codes, scales, out)  # the thread's first CUDA call
            except Exception as e:  # reported below
                errors.append(repr(e))

        th = threading.Thread(target=worker)
        th.start()
        th.join()
        assert not errors, errors
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


def test_concurrent_host_threads_and_streams(nf4, o):
    """Four host threads, each with its own stream, run the GEMV (M = 1, 3), the T <= 32 streaming
    kernel (M = 8), the wide one (M = 300) and a grouped launch ten times each, all at once: every
    result equals the single-threaded one bit for bit (ctypes releases the GIL around the calls)."""
    import threading
    from nf4_weight_only_gb300 import synth
    cases = [(1, 4096, 2048, 0), (3, 1536, 11008, 1), (8, 6144, 5120, 2), (300, 1024, 2048, 3)]
    prepared = []
    for m, n, k, seed in cases:
        codes, scales = nf4.quantize(synth.device_weights(900 + seed, n, k, DEV))
        x = synth.device_activations_bf16(950 + seed, m, k, DEV)
        ref = torch.empty((m, n), dtype=torch.bfloat16, device=DEV)
        nf4.nf4_linear(x, codes, scales, ref)
        prepared.append((x, codes, scales, ref))
    gx = prepared[1][0]
    g_ref = [torch.empty((3, n), dtype=torch.bfloat16, device=DEV) for n in (1536, 512)]
    g_mats = [(prepared[1][1], prepared[1][2]), nf4.quantize(synth.device_weights(990, 512, 11008, DEV))]
    nf4.nf4_linear_grouped(gx, [c for c, _ in g_mats], [s for _, s in g_mats], g_ref)
    torch.cuda.synchronize()
    errors = []

    def worker(i):
        try:
            stream = torch.cuda.Stream(device=DEV)
            x, codes, scales, ref = prepared[i]
            outs = [torch.empty_like(ref) for _ in range(10)]
            g_outs = [[torch.empty_like(r) for r in g_ref] for _ in range(10)]
            for j in range(10):
                nf4.nf4_linear(x, codes, scales, outs[j], stream)
                nf4.nf4_linear_grouped(gx, [c for c, _ in g_mats], [s for _, s in g_mats], g_outs[j], stream)
            stream.synchronize()
            for j in range(10):
                if not torch.equal(outs[j].view(torch.int16), ref.view(torch.int16)):
                    errors.append(f"thread {i} call {j}: linear differs")
                for a, b in zip(g_outs[j], g_ref):
                    if not torch.equal(a.view(torch.int16), b.view(torch.int16)):
                        errors.append(f"thread {i} call {j}: grouped differs")
        except Exception as e:  # reported below
            errors.append(f"thread {i}: {e!r}")

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(cases))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors[:5]
    assert device_error(nf4) == 0


@pytest.mark.parametrize("m,n,k", [(1, 3, (1 << 26) + 192), (3, 2, (1 << 24) + 64)])
def test_linear_huge_k(nf4, o, m, n, k):
    """K of 16.8 M and 67.1 M (ragged past a power of two): the streaming kernel's group, box and
    scale-window arithmetic at sizes where a 32-bit byte offset of a row's scales would overflow."""
    from nf4_weight_only_gb300 import synth
    w = synth.device_weights(700 + n, n, k, DEV)
    codes, scales = nf4.quantize(w)
    x = synth.device_activations_bf16(701 + n, m, k, DEV)
    y = torch.empty((m, n), dtype=torch.bfloat16, device=DEV)
    nf4.nf4_linear(x, codes, scales, y)
    torch.cuda.synchronize()
    assert device_error(nf4) == 0
    c_ref, s_ref = o.quantize(w.cpu().numpy())
    del w
    assert np.array_equal(codes.cpu().numpy(), c_ref)
    assert np.array_equal(f16_dev_to_bits(scales), s_ref)
    y64, mag = o.linear(dev_to_bits(x), c_ref, s_ref, nthreads=16)
    ok, ratio, mask = oracle.within_tolerance(dev_to_bits(y), y64, mag)
    assert ok, f"M={m} N={n} K={k}: worst ratio {ratio:.3f}"


def test_linear_more_tokens_than_one_grid(nf4, o):
    """M = 65535 * 256 + 40 tokens (more token tiles than the grid's y dimension holds), K = 64,
    N = 24: the call runs in two chunks; 4096 sampled tokens, those around the chunk boundary and
    the first and last included, checked against the oracle."""
    from nf4_weight_only_gb300 import synth
    chunk = 65535 * 256
    m, n, k = chunk + 40, 24, 64
    w = synth.device_weights(730, n, k, DEV)
    codes, scales = nf4.quantize(w)
    x = synth.device_activations_bf16(731, m, k, DEV)
    y = torch.empty((m, n), dtype=torch.bfloat16, device=DEV)
    nf4.nf4_linear(x, codes, scales, y)
    torch.cuda.synchronize()
    assert device_error(nf4) == 0
    c_ref, s_ref = o.quantize(w.cpu().numpy())
    assert np.array_equal(codes.cpu().numpy(), c_ref)
    rng = np.random.default_rng(732)
    toks = np.unique(np.concatenate([[0, m - 1, chunk - 2, chunk - 1, chunk, chunk + 1, chunk + 39],
                                     rng.integers(0, m, 4089)]))
    sel = torch.from_numpy(toks.astype(np.int64)).to(DEV)
    y64, mag = o.linear(dev_to_bits(x[sel]), c_ref, s_ref, nthreads=16)
    ok, ratio, mask = oracle.within_tolerance(dev_to_bits(y[sel]), y64, mag)
    assert ok, f"{np.count_nonzero(~mask)} sampled outputs outside tolerance (worst {ratio:.3f})"


def test_linear_five_million_rows(nf4, o):
    """N = 5,000,000 rows of K = 64 at M = 1 (the GEMV's row-range split over the whole grid);
    4096 sampled rows, the first and the last included, checked against the oracle."""
    from nf4_weight_only_gb300 import synth
    n, k = 5_000_000, 64
    w = synth.device_weights(720, n, k, DEV)
    codes, scales = nf4.quantize(w)
    x = synth.device_activations_bf16(721, 1, k, DEV)
    y = torch.empty((1, n), dtype=torch.bfloat16, device=DEV)
    nf4.nf4_linear(x, codes, scales, y)
    torch.cuda.synchronize()
    assert device_error(nf4) == 0
    rng = np.random.default_rng(722)
    rows = np.unique(np.concatenate([[0, n - 1], rng.integers(0, n, 4094)]))
    sel = torch.from_numpy(rows.astype(np.int64)).to(DEV)
    c_ref, s_ref = o.quantize(w[sel].cpu().numpy())
    assert np.array_equal(codes[sel].cpu().numpy(), c_ref)
    y64, mag = o.linear(dev_to_bits(x), c_ref, s_ref, nthreads=16)
    ok, ratio, mask = oracle.within_tolerance(dev_to_bits(y)[:, rows], y64, mag)
    assert ok, f"{np.count_nonzero(~mask)} sampled rows outside tolerance (worst {ratio:.3f})"


def test_timed_out_wait_reports_and_device_stays_usable(nf4, o):
    """A bounded wait that runs out (one thread on a barrier nothing arrives on, 1 ms) records
    code 39 instead of hanging; the next linear on the same device is still correct."""
    nf4.nf4_diag_bounded_wait(1_000_000)
    torch.cuda.synchronize()
    assert device_error(nf4) == 39
    assert device_error(nf4) == 0  # reading clears the word
    check_linear(nf4, o, 1, 257, 2048, seed=5)
    check_linear(nf4, o, 8, 130, 192, seed=6)
    assert device_error(nf4) == 0


@pytest.mark.parametrize("m,n,k", [(1, 16384, 786432), (1, 393216, 32768), (512, 16384, 131072)])
def test_wait_limit_restarts_at_each_wait(nf4, o, m, n, k):
    """Every pipeline wait limited to 100 us: a healthy linear that runs for more than ten times as
    long (the streaming kernel at M = 1 with K = 786432, the GEMV over 393216 rows, the M = 512
    GEMM; 6.8 GB or 2.2 TFLOP each) finishes with the device error word at 0 and correct sampled
    rows, because the limit restarts at each wait.  Under the same limit the diagnostic wait still
    reports code 39."""
    from nf4_weight_only_gb300 import synth
    codes, scales = synth.device_packed(740 + m, n, k, DEV)
    x = synth.device_activations_bf16(741 + m, m, k, DEV)
    y = torch.empty((m, n), dtype=torch.bfloat16, device=DEV)
    torch.cuda.synchronize()
    nf4.nf4_linear(x, codes, scales, y)  # first launch of the kernel (module load) outside the timing
    torch.cuda.synchronize()
    assert device_error(nf4) == 0
    nf4.nf4_diag_set_wait_limit(100_000)
    try:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        nf4.nf4_linear(x, codes, scales, y)
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        assert device_error(nf4) == 0
        assert ms > 1.0, f"the linear took {ms:.3f} ms, not long enough against the 0.1 ms limit"
        nf4.nf4_diag_bounded_wait(1_000_000)
        torch.cuda.synchronize()
        assert device_error(nf4) == 39
    finally:
        nf4.nf4_diag_set_wait_limit(0)
        torch.cuda.synchronize()
    rng = np.random.default_rng(742)
    rows = np.unique(np.concatenate([[0, 1, n // 2, n - 1], rng.integers(0, n, 4)]))
    sel = torch.from_numpy(rows.astype(np.int64)).to(DEV)
    y64, mag = o.linear(dev_to_bits(x), codes[sel].cpu().numpy(), f16_dev_to_bits(scales[sel]), nthreads=16)
    ok, ratio, mask = oracle.within_tolerance(dev_to_bits(y)[:, rows], y64, mag)
    assert ok, f"{np.count_nonzero(~mask)} sampled outputs outside tolerance (worst {ratio:.3f})"
    del codes, scales, x, y
    torch.cuda.empty_cache()


def test_empty_is_noop(nf4):
    y = torch.full((4,), 7.0, dtype=torch.bfloat16, device=DEV)
    x = torch.zeros((1, 64), dtype=torch.bfloat16, device=DEV)
    codes = torch.zeros((1, 32), dtype=torch.uint8, device=DEV)
    scales = torch.zeros((1, 1), dtype=torch.float16, device=DEV)
    lib = nf4.load()
    import ctypes
    st = lib.nf4_linear(ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(codes.data_ptr()),
                        ctypes.c_void_p(scales.data_ptr()), ctypes.c_void_p(y.data_ptr()), 0, 1, 64, None)
    assert st == 0
    torch.cuda.synchronize()
    assert torch.all(y == 7.0)


def test_bad_alignment_rejected_on_device_pointers(nf4):
    import ctypes
    lib = nf4.load()
    x = torch.zeros((1, 128 + 8), dtype=torch.bfloat16, device=DEV)
    codes = torch.zeros((4, 64), dtype=torch.uint8, device=DEV)
    scales = torch.zeros((4, 2), dtype=torch.float16, device=DEV)
    y = torch.zeros((1, 4), dtype=torch.bfloat16, device=DEV)
    st = lib.nf4_linear(ctypes.c_void_p(x.data_ptr() + 2), ctypes.c_void_p(codes.data_ptr()),
                        ctypes.c_void_p(scales.data_ptr()), ctypes.c_void_p(y.data_ptr()), 1, 4, 128, None)
    assert st == 3  # NF4_ERR_ALIGN


# ------------------------------------------------------------------------------------------------
# tensor-core path (M >= 5)
# ------------------------------------------------------------------------------------------------
def device_error(nf4):
    import ctypes
    lib = nf4.load()
    lib.nf4_check_device_error.argtypes = [ctypes.POINTER(ctypes.c_int)]
    lib.nf4_check_device_error.restype = ctypes.c_int
    code = ctypes.c_int(-1)
    assert lib.nf4_check_device_error(ctypes.byref(code)) == 0
    return code.value


@pytest.mark.parametrize("m", [5, 16, 17, 32, 33, 64, 100, 128, 129, 256, 300, 512, 513])
def test_linear_tensor_core_tokens(nf4, o, m):
    check_linear(nf4, o, m, 257, 1024, seed=m)
    assert device_error(nf4) == 0


@pytest.mark.parametrize("n,k", [(1, 64), (7, 128), (128, 64), (130, 192), (383, 2048), (256, 6144), (64, 16384)])
def test_linear_tensor_core_shapes(nf4, o, n, k):
    check_linear(nf4, o, 40, n, k, seed=n + k, outliers=0.01)
    assert device_error(nf4) == 0


@pytest.mark.parametrize("m,n,k", [(260, 9761, 512), (512, 19583, 256)])
def test_linear_wide_tile_runs(nf4, o, m, n, k):
    """More 128-row tiles than a token tile's share of the SMs (77 and 153 tiles against 76 CTAs
    per token tile): persistent CTAs walk runs of one to three tiles, the last tile ragged."""
    check_linear(nf4, o, m, n, k, seed=m + n)
    assert device_error(nf4) == 0


def test_linear_grouped_wide_tile_runs(nf4, o):
    """A grouped call at M = 300 whose problems (5000, 9000 and 130 rows: 40, 71 and 2 tiles) share
    76 CTAs per token tile in proportion to their tiles; every output meets the oracle bound."""
    from nf4_weight_only_gb300 import synth
    k, m = 512, 300
    ns = [5000, 9000, 130]
    x = synth.activations_bf16(902, m, k)
    xd = bf16_to_dev(x)
    packs, ys = [], []
    for i, n in enumerate(ns):
        c, sc = o.quantize(synth.weights(910 + i, n, k))
        packs.append((c, sc))
        ys.append(torch.empty((m, n), dtype=torch.bfloat16, device=DEV))
    nf4.nf4_linear_grouped(xd, [torch.from_numpy(c).to(DEV) for c, _ in packs],
                           [torch.from_numpy(sc.view(np.int16)).to(DEV).view(torch.float16) for _, sc in packs], ys)
    torch.cuda.synchronize()
    for (c, sc), y in zip(packs, ys):
        y64, mag = o.linear(x, c, sc, nthreads=16)
        ok, ratio, _ = oracle.within_tolerance(dev_to_bits(y), y64, mag)
        assert ok, ratio
    assert device_error(nf4) == 0


def test_linear_tensor_core_prefill_sampled(nf4, o):
    """20B-shaped prefill gate projection (6144 -> 16384) at M = 512, checked on sampled outputs."""
    from nf4_weight_only_gb300 import synth
    n, k, m = 16384, 6144, 512
    w = synth.device_weights(4 * 100003, n, k, DEV, outlier_frac=0.01)
    codes, scales = nf4.quantize(w)
    x = synth.device_activations_bf16(99 + k, m, k, DEV)
    y = torch.empty((m, n), dtype=torch.bfloat16, device=DEV)
    nf4.nf4_linear(x, codes, scales, y)
    torch.cuda.synchronize()
    assert device_error(nf4) == 0
    rng = np.random.default_rng(0)
    mi = rng.integers(0, m, 3000)
    ni = rng.integers(0, n, 3000)
    mi[:8] = [0, m - 1, 0, m - 1, 255, 256, 511, 7]
    ni[:8] = [0, 0, n - 1, n - 1, 127, 128, 16383, 8191]
    # the oracle quantizes the generator's fp32 rows itself; the GPU codes of those rows must match
    rows, ni_local = np.unique(ni, return_inverse=True)
    sel = torch.from_numpy(rows.astype(np.int64)).to(DEV)
    c_ref, s_ref = o.quantize(w[sel].cpu().numpy())
    assert np.array_equal(codes[sel].cpu().numpy(), c_ref)
    assert np.array_equal(f16_dev_to_bits(scales[sel]), s_ref)
    x_h = dev_to_bits(x)
    y64, mag = o.linear_entries(x_h, c_ref, s_ref, mi, ni_local)
    ok, ratio, mask = oracle.within_tolerance(dev_to_bits(y)[mi, ni], y64, mag)
    assert ok, f"{np.count_nonzero(~mask)} sampled outputs outside tolerance (worst {ratio:.3f})"


def test_linear_negative_and_zero_scales(nf4, o):
    """Scales outside what quantize writes (negative, zero, tiny subnormal) follow the same rule."""
    from nf4_weight_only_gb300 import synth
    rng = np.random.default_rng(5)
    n, k = 200, 512
    codes = rng.integers(0, 256, (n, k // 2), dtype=np.uint8)
    scales = (rng.standard_normal((n, k // 64)) * 0.05).astype(np.float16)
    scales[0, :] = 0
    scales[1, :] = np.float16(-0.0)
    scales[2, :] = np.float16(2.0 ** -24)
    scales[3, :] = np.float16(65504.0)
    sbits = scales.view(np.uint16)
    for m in (1, 3, 9, 40):
        x = synth.activations_bf16(m, m, k)
        y = run_linear(nf4, x, codes, sbits)
        y64, mag = o.linear(x, codes, sbits)
        ok, ratio, _ = oracle.within_tolerance(y, y64, mag)
        assert ok, (m, ratio)
    assert device_error(nf4) == 0


# ------------------------------------------------------------------------------------------------
# grouped linears sharing x
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("m", [1, 3, 4, 7, 32])
def test_linear_grouped(nf4, o, m):
    """q, k and v of a 2048-wide layer (plus a ragged fourth) in one call: every output meets the
    oracle bound and a second call gives the same bytes.  (Separate calls may split K differently,
    so their low-order bits are not required to match.)"""
    from nf4_weight_only_gb300 import synth
    k = 2048
    ns = [2048, 256, 256, 37]
    x = synth.activations_bf16(50 + m, m, k)
    xd = bf16_to_dev(x)
    mats = []
    for i, n in enumerate(ns):
        w = synth.weights(60 + i, n, k)
        c, s = o.quantize(w)
        mats.append((c, s, torch.from_numpy(c).to(DEV),
                     torch.from_numpy(s.view(np.int16)).view(torch.float16).to(DEV)))
    ys = [torch.empty((m, n), dtype=torch.bfloat16, device=DEV) for n in ns]
    ys2 = [torch.empty((m, n), dtype=torch.bfloat16, device=DEV) for n in ns]
    nf4.nf4_linear_grouped(xd, [t[2] for t in mats], [t[3] for t in mats], ys)
    nf4.nf4_linear_grouped(xd, [t[2] for t in mats], [t[3] for t in mats], ys2)
    torch.cuda.synchronize()
    assert device_error(nf4) == 0
    for (c, s, cd, sd), y, y2 in zip(mats, ys, ys2):
        assert torch.equal(y.view(torch.int16), y2.view(torch.int16))
        y64, mag = o.linear(x, c, s, nthreads=16)
        ok, ratio, _ = oracle.within_tolerance(dev_to_bits(y), y64, mag)
        assert ok, ratio


@pytest.mark.parametrize("m", [1, 3, 8, 100])
def test_linear_grouped_eight(nf4, o, m):
    """The most linears one grouped call takes (8), ragged row counts with an empty one, K = 640
    (ten groups, a ragged K-slice): GEMV (M = 1, 3), narrow (M = 8) and wide (M = 100) streaming;
    every output meets the oracle bound."""
    from nf4_weight_only_gb300 import synth
    k = 640
    ns = [1, 130, 0, 257, 64, 7, 1000, 3]
    x = synth.activations_bf16(70 + m, m, k)
    xd = bf16_to_dev(x)
    mats = []
    for i, n in enumerate(ns):
        c, s = o.quantize(synth.weights(80 + i, n, k)) if n else (np.zeros((0, k // 2), np.uint8),
                                                                  np.zeros((0, k // 64), np.uint16))
        mats.append((c, s, torch.from_numpy(c).to(DEV), torch.from_numpy(s.view(np.int16)).view(torch.float16).to(DEV)))
    ys = [torch.empty((m, n), dtype=torch.bfloat16, device=DEV) for n in ns]
    nf4.nf4_linear_grouped(xd, [t[2] for t in mats], [t[3] for t in mats], ys)
    torch.cuda.synchronize()
    assert device_error(nf4) == 0
    for (c, s, _, _), y, n in zip(mats, ys, ns):
        if n == 0:
            continue
        y64, mag = o.linear(x, c, s, nthreads=16)
        ok, ratio, _ = oracle.within_tolerance(dev_to_bits(y), y64, mag)
        assert ok, f"N={n}: worst ratio {ratio:.3f}"


# ------------------------------------------------------------------------------------------------
# small-M tensor-core streaming (M <= 32): tiles of 128 rows plus a partial tile split into
# K-slices, ragged last stages, every token-tile size
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("m", [5, 8, 16, 32])
@pytest.mark.parametrize("n,k", [(2048, 11008), (22016, 2048), (19457, 640), (3, 27648), (19500, 320)])
def test_linear_stream_tiles(nf4, o, m, n, k):
    check_linear(nf4, o, m, n, k, seed=7 * n + k + m)
    assert device_error(nf4) == 0


@pytest.mark.parametrize("m,n,k", [
    (8, 5168, 1024),   # 34 rows a CTA on 152 SMs: three K-slices (10 rows a tensor-memory quarter)
    (16, 5168, 1024),  # the same at 16 tokens (48 pseudo-token columns)
    (4, 3496, 1024),   # 23 rows: five slices
    (8, 2736, 1024),   # 18 rows: six slices
    (4, 1824, 448),    # 12 rows, seven groups: seven slices
    (8, 5120, 13824),  # the 14B-shaped down projection at M = 8
])
def test_linear_stream_slices_not_power_of_two(nf4, o, m, n, k):
    """Partial tiles whose K-slice count is not a power of two: a row's slices sit in consecutive lanes
    of one tensor-memory quarter, and a token's columns can straddle two 16-column loads."""
    check_linear(nf4, o, m, n, k, seed=13 * n + k + m)
    assert device_error(nf4) == 0


@pytest.mark.parametrize("m,n,k", [(1, 300, 36864), (1, 19457, 36864), (2, 150, 17408), (3, 2048, 20480),
                                   (4, 129, 17408)])
def test_linear_stream_long_k(nf4, o, m, n, k):
    """M <= 4 with K past the GEMV's register-resident range runs the streaming kernel."""
    check_linear(nf4, o, m, n, k, seed=11 * n + k + m)
    assert device_error(nf4) == 0


# ------------------------------------------------------------------------------------------------
# packed embedding rows
# ------------------------------------------------------------------------------------------------
def run_embed(nf4, ids, codes_d, scales_d, k):
    out = Guarded((len(ids), k), torch.bfloat16)
    nf4.nf4_embed(torch.from_numpy(np.asarray(ids, np.int32)).to(DEV), codes_d, scales_d, out.t)
    torch.cuda.synchronize()
    assert out.canaries_intact(), "nf4_embed wrote outside out"
    return dev_to_bits(out.t)


def test_embed_bit_exact(nf4, o):
    from nf4_weight_only_gb300 import synth
    v, k = 1000, 2048
    codes, scales = o.quantize(synth.weights(21, v, k))
    cd = torch.from_numpy(codes).to(DEV)
    sd = torch.from_numpy(scales.view(np.int16)).view(torch.float16).to(DEV)
    rng = np.random.default_rng(22)
    ids = np.concatenate([[0, v - 1, 7, 7], rng.integers(0, v, 300)]).astype(np.int32)
    got = run_embed(nf4, ids, cd, sd, k)
    want, bad = o.embed(ids, codes, scales)
    assert bad == 0 and np.array_equal(got, want)
    assert device_error(nf4) == 0


def test_embed_vocabulary_sampled(nf4, o):
    """A 3B-shaped vocabulary (151936 x 2048) quantized on the device; 512 sampled ids (with the first
    and last rows) checked bit for bit against the oracle on those rows."""
    from nf4_weight_only_gb300 import synth
    v, k = 151936, 2048
    w = synth.device_weights(23, v, k, DEV)
    codes_d, scales_d = nf4.quantize(w)
    rng = np.random.default_rng(24)
    ids = np.concatenate([[0, v - 1], rng.integers(0, v, 510)]).astype(np.int32)
    got = run_embed(nf4, ids, codes_d, scales_d, k)
    uniq, inv = np.unique(ids, return_inverse=True)
    sel = torch.from_numpy(uniq.astype(np.int64)).to(DEV)
    # the oracle quantizes the generator's rows itself; the GPU's packed rows must match them
    c_h, s_h = o.quantize(w[sel].cpu().numpy())
    del w
    assert np.array_equal(codes_d[sel].cpu().numpy(), c_h)
    assert np.array_equal(f16_dev_to_bits(scales_d[sel]), s_h)
    want, bad = o.embed(inv.astype(np.int32), c_h, s_h)
    assert bad == 0 and np.array_equal(got, want)


def test_embed_out_of_range_ids(nf4, o):
    from nf4_weight_only_gb300 import synth
    v, k = 50, 128
    codes, scales = o.quantize(synth.weights(25, v, k))
    cd = torch.from_numpy(codes).to(DEV)
    sd = torch.from_numpy(scales.view(np.int16)).view(torch.float16).to(DEV)
    assert device_error(nf4) == 0
    ids = np.array([3, -1, v, 2 ** 31 - 1, v - 1], np.int32)
    got = run_embed(nf4, ids, cd, sd, k)
    want, bad = o.embed(ids, codes, scales)
    assert bad == 3 and np.array_equal(got, want)
    assert not got[1:4].any()
    assert device_error(nf4) == 41
    assert device_error(nf4) == 0  # read and cleared


def test_embed_empty_is_noop(nf4):
    out = torch.full((1, 64), 3.0, dtype=torch.bfloat16, device=DEV)
    ids = torch.zeros((0,), dtype=torch.int32, device=DEV)
    codes = torch.zeros((2, 32), dtype=torch.uint8, device=DEV)
    scales = torch.zeros((2, 1), dtype=torch.float16, device=DEV)
    nf4.nf4_embed(ids, codes, scales, out)
    torch.cuda.synchronize()
    assert torch.all(out == 3.0)


# ------------------------------------------------------------------------------------------------
# overflow streaming through the two-slot ring
# ------------------------------------------------------------------------------------------------
def _host_weights(nf4, seed, n, k):
    """Packed weights quantized on the device; returns (device codes, scales, pinned host copies)."""
    from nf4_weight_only_gb300 import synth
    codes, scales = nf4.quantize(synth.device_weights(seed, n, k, DEV))
    return codes, scales, codes.cpu().pin_memory(), scales.cpu().pin_memory()


def _bits_to_f64(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _f64_to_bf16_bits(v):
    return torch.from_numpy(np.asarray(v, np.float64)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_ring_chain_matches_resident(nf4, o):
    """Five chained M = 1 linears (y of one is x of the next) of different sizes streamed from
    pinned host memory: every y is bit for bit the resident nf4_linear result, and every y meets
    the oracle's bound for a chain the oracle runs itself.

    The oracle's chain feeds its own bf16-rounded y64 forward, never the GPU's y.  Link i + 1 then
    sees inputs that may differ from the GPU's by delta_k <= tol_i,k + 2^-9 |y64_i,k| (the GPU's
    error bound plus the oracle's own rounding), which moves the exact sum by at most
    D = sum_k delta_k |w_hat_k|; the accepted error of link i + 1 is the per-linear bound plus
    D (1 + 2^-8 + 2^-12), all computed from the oracle's values."""
    from nf4_weight_only_gb300 import synth
    dims = [2048, 2560, 1024, 2048, 11008, 2048]
    mats = [_host_weights(nf4, 300 + i, dims[i + 1], dims[i]) for i in range(len(dims) - 1)]
    x0 = synth.device_activations_bf16(310, 1, dims[0], DEV)
    ys = [torch.empty((1, n), dtype=torch.bfloat16, device=DEV) for n in dims[1:]]
    xs = [x0] + ys[:-1]
    slot = max(nf4.Ring.bytes_needed(dims[i + 1], dims[i]) for i in range(len(mats)))
    with nf4.Ring(slot) as ring:
        ring.run([(xs[i], mats[i][2], mats[i][3], ys[i]) for i in range(len(mats))])
        torch.cuda.synchronize()
    for i, (cd, sd, _, _) in enumerate(mats):
        want = torch.empty_like(ys[i])
        nf4.nf4_linear(xs[i], cd, sd, want)
        torch.cuda.synchronize()
        assert torch.equal(want.view(torch.int16), ys[i].view(torch.int16)), f"linear {i}"
    # The oracle checks the first linear, whose x comes from the generator (the later ones read the
    # GPU's y): it quantizes the same fp32 weights itself, which the GPU's packed copy must match.
    c_ref, s_ref = o.quantize(synth.device_weights(300, dims[1], dims[0], DEV).cpu().numpy())
    assert np.array_equal(mats[0][2].numpy(), c_ref)
    assert np.array_equal(mats[0][3].view(torch.int16).numpy().view(np.uint16), s_ref)
    y64, absum = o.linear(dev_to_bits(x0), c_ref, s_ref, nthreads=16)
    ok, ratio, _ = oracle.within_tolerance(dev_to_bits(ys[0]), y64, absum)
    assert ok, f"oracle bound, linear 0: worst ratio {ratio:.3f}"
    # the whole chain against the oracle's own chain (see the docstring for the bound)
    x_o = dev_to_bits(x0)
    delta = np.zeros(dims[0])
    for i in range(len(mats)):
        c_ref, s_ref = o.quantize(synth.device_weights(300 + i, dims[i + 1], dims[i], DEV).cpu().numpy())
        assert np.array_equal(mats[i][2].numpy(), c_ref), f"packed codes, linear {i}"
        y64, absum = o.linear(x_o, c_ref, s_ref, nthreads=16)
        w_abs = np.abs(_bits_to_f64(o.dequant(c_ref, s_ref)))
        d = w_abs @ delta
        tol = 2.0 ** -8 * np.abs(y64[0]) + 2.0 ** -12 * absum[0] + d * (1 + 2.0 ** -8 + 2.0 ** -12)
        err = np.abs(_bits_to_f64(dev_to_bits(ys[i]))[0] - y64[0])
        assert np.all(err <= tol), f"linear {i}: worst error / bound {np.max(err / tol):.3f}"
        delta = tol + 2.0 ** -9 * np.abs(y64[0])
        x_o = _f64_to_bf16_bits(y64)
    assert device_error(nf4) == 0


@pytest.mark.parametrize("m", [4, 32])
def test_ring_small_batch(nf4, o, m):
    """M = 4 and M = 32 (tensor-core small-M kernel) through the ring, twelve distinct matrices
    over two slots, compared with the resident results; the first and the last also against the
    oracle (its own quantization of the same weights, the generator's x)."""
    from nf4_weight_only_gb300 import synth
    n, k = 3072, 2048
    mats = [_host_weights(nf4, 400 + i, n, k) for i in range(12)]
    x = synth.device_activations_bf16(401, m, k, DEV)
    ys = [torch.empty((m, n), dtype=torch.bfloat16, device=DEV) for _ in mats]
    with nf4.Ring(nf4.Ring.bytes_needed(n, k)) as ring:
        ring.run([(x, c[2], c[3], y) for c, y in zip(mats, ys)])
        torch.cuda.synchronize()
    for (cd, sd, _, _), y in zip(mats, ys):
        want = torch.empty_like(y)
        nf4.nf4_linear(x, cd, sd, want)
        torch.cuda.synchronize()
        assert torch.equal(want.view(torch.int16), y.view(torch.int16))
    for i in (0, len(mats) - 1):
        c_ref, s_ref = o.quantize(synth.device_weights(400 + i, n, k, DEV).cpu().numpy())
        assert np.array_equal(mats[i][2].numpy(), c_ref)
        y64, absum = o.linear(dev_to_bits(x), c_ref, s_ref, nthreads=16)
        ok, ratio, _ = oracle.within_tolerance(dev_to_bits(ys[i]), y64, absum)
        assert ok, f"matrix {i}: worst ratio {ratio:.3f}"


def test_ring_runs_back_to_back_and_in_a_graph(nf4):
    """Two runs enqueued without a host sync reuse the slots safely; a captured run replays to the
    same bytes, and an eager run after the capture still agrees."""
    from nf4_weight_only_gb300 import synth
    n, k = 4096, 4096
    a = [_host_weights(nf4, 500 + i, n, k) for i in range(3)]
    b = [_host_weights(nf4, 510 + i, n, k) for i in range(3)]
    x = synth.device_activations_bf16(520, 1, k, DEV)
    ya = [torch.empty((1, n), dtype=torch.bfloat16, device=DEV) for _ in a]
    yb = [torch.empty((1, n), dtype=torch.bfloat16, device=DEV) for _ in b]
    want = []
    for cd, sd, _, _ in a + b:
        w = torch.empty((1, n), dtype=torch.bfloat16, device=DEV)
        nf4.nf4_linear(x, cd, sd, w)
        want.append(w)
    torch.cuda.synchronize()
    stream = torch.cuda.Stream(device=DEV)
    with nf4.Ring(nf4.Ring.bytes_needed(n, k)) as ring:
        ring.run([(x, m[2], m[3], y) for m, y in zip(a, ya)], stream)
        ring.run([(x, m[2], m[3], y) for m, y in zip(b, yb)], stream)
        torch.cuda.synchronize()
        for w, y in zip(want, ya + yb):
            assert torch.equal(w.view(torch.int16), y.view(torch.int16))
        for y in ya + yb:
            y.zero_()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            ring.run([(x, m[2], m[3], y) for m, y in zip(a + b, ya + yb)], stream)
        for _ in range(2):
            graph.replay()
        torch.cuda.synchronize()
        for w, y in zip(want, ya + yb):
            assert torch.equal(w.view(torch.int16), y.view(torch.int16))
        for y in yb:
            y.zero_()
        ring.run([(x, m[2], m[3], y) for m, y in zip(b, yb)], stream)
        torch.cuda.synchronize()
        for w, y in zip(want[3:], yb):
            assert torch.equal(w.view(torch.int16), y.view(torch.int16))


def test_ring_errors(nf4):
    """A matrix larger than a slot and pageable host memory are refused before anything is
    enqueued; the ring keeps working afterwards."""
    from nf4_weight_only_gb300 import synth
    n, k = 1024, 2048
    cd, sd, ch, sh = _host_weights(nf4, 600, n, k)
    x = synth.device_activations_bf16(601, 1, k, DEV)
    y = torch.full((1, n), 7.0, dtype=torch.bfloat16, device=DEV)
    with nf4.Ring(nf4.Ring.bytes_needed(n, k) - 16) as small:
        with pytest.raises(nf4.NF4Error) as e:
            small.run([(x, ch, sh, y)])
        assert e.value.status == 2
    with nf4.Ring(nf4.Ring.bytes_needed(n, k)) as ring:
        with pytest.raises(nf4.NF4Error) as e:
            ring.run([(x, ch.clone(), sh, y)])  # clone(): pageable host memory
        assert e.value.status == 7
        torch.cuda.synchronize()
        assert torch.all(y == 7.0)
        ring.run([(x, ch, sh, y)])
        want = torch.empty_like(y)
        nf4.nf4_linear(x, cd, sd, want)
        torch.cuda.synchronize()
        assert torch.equal(want.view(torch.int16), y.view(torch.int16))
