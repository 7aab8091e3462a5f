"""Repeated launches of the pipelined linear kernels write bit-identical outputs (GPU).

Every kernel accumulates in a fixed order, so each launch on the same inputs must write the same bits.
A synchronization fault (a slot rewritten before its readers are done, a stage read before it lands)
shows up as a launch whose output differs, or as a pipeline wait that runs out (the device error
word).  Each case runs many launches on one stream; every other launch follows a write of a buffer
larger than L2, so that copy latencies, and with them the warp roles' relative timing, change from
launch to launch.  The first launch of each case is also checked against the oracle on a few rows.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from gpu_util import DEV, dev_to_bits, f16_dev_to_bits

pytestmark = pytest.mark.gpu

LAUNCHES = int(os.environ.get("NF4_STRESS_LAUNCHES", "120"))  # per case; raise it for a longer soak


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


@pytest.fixture(scope="module")
def flush():
    return torch.empty(256 << 20, dtype=torch.uint8, device=DEV)


CASES = [
    # (what, M, rows of each linear, K)
    ("GEMV, M = 1", 1, [5120], 5120),
    ("GEMV, M = 3", 3, [7168], 5120),
    ("GEMV, M = 1, 27648-wide rows (half-size table)", 1, [5120], 27648),
    ("small-M, one 34-row tile per CTA, three K-slices (14B-shaped q)", 8, [5120], 5120),
    ("small-M grouped 2 x 13824 x 5120", 32, [13824, 13824], 5120),
    ("small-M, K = 16384", 4, [6144], 16384),
    ("small-M, two full tiles and a partial one per CTA", 16, [40000], 1024),
    ("small-M, six single-stage full tiles per CTA (K = 128)", 8, [131072], 128),
    ("GEMM-form, persistent runs of tiles", 260, [9761], 512),
    ("GEMM-form grouped, runs shared in proportion", 300, [5000, 9000, 130], 512),
    ("GEMM-form, M = 512", 512, [8192], 6144),
]


@pytest.mark.parametrize("what,m,ns,k", CASES, ids=[c[0] for c in CASES])
def test_repeated_launches_identical(nf4, o, flush, what, m, ns, k):
    from nf4_weight_only_gb300 import synth
    packs = [synth.device_packed(300 + i, n, k, DEV) for i, n in enumerate(ns)]
    x = synth.device_activations_bf16(77 + m, m, k, DEV)
    ys = [torch.empty((m, n), dtype=torch.bfloat16, device=DEV) for n in ns]

    def launch():
        if len(ns) == 1:
            nf4.nf4_linear(x, packs[0][0], packs[0][1], ys[0])
        else:
            nf4.nf4_linear_grouped(x, [c for c, _ in packs], [s for _, s in packs], ys)

    nf4.nf4_check_device_error()  # clear
    launch()
    first = [y.clone() for y in ys]
    assert nf4.nf4_check_device_error() == 0, f"{what}: a pipeline wait ran out"
    # the first launch against the oracle on a few rows of each linear
    rng = np.random.default_rng(m + k)
    xb = dev_to_bits(x)
    for (codes, scales), y in zip(packs, first):
        n = codes.shape[0]
        rows = np.unique(np.concatenate([[0, n - 1], rng.integers(0, n, 6)]))
        sel = torch.from_numpy(rows.astype(np.int64)).to(DEV)
        y64, mag = o.linear(xb, codes[sel].cpu().numpy(), f16_dev_to_bits(scales[sel]), nthreads=16)
        ok, ratio, _ = oracle.within_tolerance(dev_to_bits(y)[:, rows], y64, mag)
        assert ok, f"{what}: first launch outside the oracle bound (worst {ratio:.3f})"
    differing = []
    for i in range(LAUNCHES):
        if i % 2 == 0:
            flush.fill_(i & 0xFF)
        for y in ys:
            y.fill_(0)
        launch()
        if not all(torch.equal(y, f) for y, f in zip(ys, first)):
            differing.append(i)
    err = nf4.nf4_check_device_error()
    assert not differing and err == 0, (f"{what}: {len(differing)} of {LAUNCHES} launches differ from the first "
                                        f"(first at {differing[:1]}), device error word {err}")
    print(f"{what}: {LAUNCHES} launches bit-identical, error word 0")
