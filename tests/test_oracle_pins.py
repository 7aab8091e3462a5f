"""The oracle against its pins (CPU only).  See ``oracle_pins.py`` for what pins each function."""
import multiprocessing as mp
import os

import numpy as np
import pytest

import oracle
import oracle_pins as P


@pytest.fixture(scope="module")
def o():
    return oracle.default()


@pytest.mark.parametrize("pin", P.FAST_PINS, ids=lambda f: f.__name__)
def test_pin(o, pin):
    pin(o)


def _pool_map(fn, chunks):
    ctx = mp.get_context("spawn")
    with ctx.Pool(min(8, os.cpu_count() or 1)) as pool:
        yield from pool.imap_unordered(fn, chunks)


def test_f16_exhaustive(o):
    """Every binary32 value whose exponent field lies in [100, 145] (every value that neither
    flushes to zero nor overflows in fp16), both signs."""
    for res in _pool_map(P.f16_sweep_chunk, [(o.path, e) for e in range(100, 146)]):
        assert res is None, f"fp16 rounding differs at {res}"


def test_bf16_exhaustive_binades(o):
    """Every mantissa in the subnormal, smallest, middle and largest binades, both signs."""
    P.pin_bf16(o, exhaustive=True)


def test_code_exhaustive_unit_interval(o):
    """Every binary32 r in [-1, 1] (about 2.1e9 values) against the threshold formulation."""
    lo, hi = P.ordered_key(np.float32(-1.0)), P.ordered_key(np.float32(1.0)) + 1
    step = 1 << 24
    chunks = [(o.path, a, min(a + step, hi)) for a in range(lo, hi, step)]
    for res in _pool_map(P.code_sweep_chunk, chunks):
        assert res is None, f"nearest code differs at r={res[0]!r}: oracle {res[1]}, thresholds {res[2]}"


def test_thresholds_are_monotone_flips(o):
    """The bisection's premise: between neighbours the fp32 predicate flips exactly once."""
    t = P.qlora_published_table()
    thr = P.decision_thresholds(t)
    assert np.all(np.diff(thr) > 0)
    for i in range(15):
        assert t[i] < thr[i] <= t[i + 1]
        mid = (np.float64(t[i]) + np.float64(t[i + 1])) / 2
        assert abs(np.float64(thr[i]) - mid) < 2.0 ** -22


def test_tolerance_rule():
    """The acceptance bound accepts the correctly rounded result and rejects a clear miss."""
    y64 = np.array([1.0, -3.0e-3, 0.0, 250.0])
    mag = np.array([5.0, 0.1, 1.0, 300.0])
    y_round = P.bf16_bits_torch(y64.astype(np.float32))
    ok, ratio, _ = oracle.within_tolerance(y_round, y64, mag)
    assert ok and ratio <= 0.5 + 1e-9 + 2.0 ** -12 * 5.0 / (2.0 ** -8)
    bad = P.bf16_bits_torch((y64 + 4 * oracle.tolerance_bound(y64, mag)).astype(np.float32))
    ok, ratio, mask = oracle.within_tolerance(bad, y64, mag)
    assert not ok and ratio > 1.0 and not mask.any()
