"""GPU test of nf4_linear_host_noalloc, the streamed linear that allocates nothing.

Some callers cannot allocate device memory when they run a layer: their own pool allocator already
holds the GPU's memory, or their loop cannot pay for cudaMalloc / cudaFree, which may synchronise
the device.  For them the library stages host-resident packed weights through a fixed device array
of its own (16 MiB) instead of the cudaMalloc'ed slots of a ring.  This file checks, through the C
ABI, that two calls in a row give what the existing nf4_linear gives on device-resident copies of
the same weights (bit for bit, hence within the oracle's bound, which is checked too), and that a
linear too large for the array or held in pageable memory is refused before anything runs.

The file name makes pytest collect it last, so a run that stops at the first failure has already
run every other test; it also passes on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import DEV, dev_to_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nf4():
    import nf4_weight_only_gb300 as m
    from nf4_weight_only_gb300 import build
    build.build()
    m.load()
    return m


def _weights(nf4, seed, n, k):
    """Packed weights quantized on the device, with page-locked host copies."""
    from nf4_weight_only_gb300 import synth
    codes, scales = nf4.quantize(synth.device_weights(seed, n, k, DEV))
    return codes, scales, codes.cpu().pin_memory(), scales.cpu().pin_memory()


def _resident(nf4, x, codes, scales):
    y = torch.empty((x.shape[0], codes.shape[0]), dtype=torch.bfloat16, device=DEV)
    nf4.nf4_linear(x, codes, scales, y)
    return y


def test_two_calls_in_a_row_match_nf4_linear(nf4):
    from nf4_weight_only_gb300 import synth
    # A: M = 1 on the CUDA-core GEMV, 11.97 MB of packed weights (near the 16 MiB limit);
    # B: M = 8 on the tensor-core streaming kernel.  B overwrites the array A used.
    cases = [(1, 11008, 2048, 700), (8, 3072, 4096, 710)]
    mats = [_weights(nf4, seed, n, k) for _, n, k, seed in cases]
    xs = [synth.device_activations_bf16(seed + 1, m, k, DEV) for m, _, k, seed in cases]
    for (_, n, k, _) in cases:
        assert nf4.Ring.bytes_needed(n, k) <= nf4.noalloc_slot_bytes()
    want = [_resident(nf4, x, cd, sd) for x, (cd, sd, _, _) in zip(xs, mats)]
    got = [torch.full_like(w, 3.0) for w in want]
    stream = torch.cuda.Stream(device=DEV)
    stream.wait_stream(torch.cuda.current_stream())
    for rnd in range(2):  # two calls in a row (no host sync between them), then the same again
        for x, (_, _, ch, sh), y in zip(xs, mats, got):
            nf4.nf4_linear_host_noalloc(x, ch, sh, y, stream)
        stream.synchronize()
        for i, (w, y) in enumerate(zip(want, got)):
            assert torch.equal(w.view(torch.int16), y.view(torch.int16)), f"round {rnd}, call {i}"
            y.fill_(3.0)
        torch.cuda.synchronize()
    # the bound the parity tests use, on the last call of the last round
    for x, (_, _, ch, sh), y in zip(xs, mats, got):
        nf4.nf4_linear_host_noalloc(x, ch, sh, y)
    torch.cuda.synchronize()
    # The oracle quantizes the generator's fp32 weights itself (the packed copies must match them)
    # and bounds the outputs with its own codes and the generator's x.
    o = oracle.default()
    for i, (x, (_, _, ch, sh), y, (_, n, k, seed)) in enumerate(zip(xs, mats, got, cases)):
        c_ref, s_ref = o.quantize(synth.device_weights(seed, n, k, DEV).cpu().numpy())
        assert np.array_equal(ch.numpy(), c_ref) and np.array_equal(sh.view(torch.int16).numpy().view(np.uint16), s_ref)
        y64, mag = o.linear(dev_to_bits(x), c_ref, s_ref, nthreads=16)
        ok, ratio, _ = oracle.within_tolerance(dev_to_bits(y), y64, mag)
        assert ok, f"call {i}: outside the oracle bound, worst ratio {ratio:.3f}"


def test_refusals_leave_y_untouched(nf4):
    from nf4_weight_only_gb300 import synth
    # 16384 x 2048: 17.8 MB of packed weights, more than the 16 MiB array
    n, k = 16384, 2048
    assert nf4.Ring.bytes_needed(n, k) > nf4.noalloc_slot_bytes()
    _, _, ch, sh = _weights(nf4, 720, n, k)
    x = synth.device_activations_bf16(721, 1, k, DEV)
    y = torch.full((1, n), 5.0, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(nf4.NF4Error) as e:
        nf4.nf4_linear_host_noalloc(x, ch, sh, y)
    assert e.value.status == 2  # NF4_ERR_SHAPE
    n2 = 1024
    cd, sd, ch2, sh2 = _weights(nf4, 722, n2, k)
    y2 = torch.full((1, n2), 5.0, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(nf4.NF4Error) as e:
        nf4.nf4_linear_host_noalloc(x, ch2.clone(), sh2, y2)  # clone(): pageable host memory
    assert e.value.status == 7  # NF4_ERR_MEMORY
    torch.cuda.synchronize()
    assert torch.all(y == 5.0) and torch.all(y2 == 5.0)
    # and the entry point still works afterwards
    nf4.nf4_linear_host_noalloc(x, ch2, sh2, y2)
    want = _resident(nf4, x, cd, sd)
    torch.cuda.synchronize()
    assert torch.equal(want.view(torch.int16), y2.view(torch.int16))
