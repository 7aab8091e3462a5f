"""Pins for the CPU oracle: checks against values the mathematics or independent routines fix.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises ``AssertionError`` when the oracle
disagrees with something that is not the oracle itself:

* the NF4 table against the QLoRA quantile construction (scipy's normal quantile);
* the fp16 / bf16 roundings against numpy's float16 cast and torch's bfloat16 cast;
* the nearest-code rule against an independent formulation: 15 decision thresholds found by
  bisection over binary32 bit patterns with the fp32 neighbour-distance rule;
* quantize against a float64 midpoint search (exact away from midpoints) and numpy's fp16 cast;
* dequant over every (code, finite fp16 scale) pair against a float64 product rounded by numpy
  (to binary32) and torch (to bfloat16);
* the linear against numpy's float64 matmul, unit-vector closed forms and exact rationals;
* a hand-derived packing example (``tests/golden/``) and the payload ratio printed by the
  deep-fold README (format paragraph: about 3.76x smaller than BF16).

The same functions run against deliberately broken builds of the oracle in
``test_oracle_mutants.py``; each planted mistake must trip at least one of them.
"""
from __future__ import annotations

import os
from fractions import Fraction

import numpy as np
import torch

import oracle as oracle_mod

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ------------------------------------------------------------------------------------------------
# helpers that hold no oracle arithmetic
# ------------------------------------------------------------------------------------------------
def f32_from_bits(bits: np.ndarray) -> np.ndarray:
    return np.asarray(bits, np.uint32).view(np.float32)


def bf16_bits_torch(a: np.ndarray) -> np.ndarray:
    """torch's float32 -> bfloat16 cast (round to nearest even), as uint16 bits."""
    t = torch.from_numpy(np.ascontiguousarray(a, np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def f16_bits_numpy(a: np.ndarray) -> np.ndarray:
    return np.asarray(a, np.float32).astype(np.float16).view(np.uint16)


def ordered_key(f: np.float32) -> int:
    """Integer key that increases with the binary32 value (sign-magnitude to two's complement)."""
    b = int(np.float32(f).view(np.uint32))
    return b if b < 0x80000000 else -(b & 0x7FFFFFFF)


def from_key(key: int) -> np.float32:
    b = key if key >= 0 else (0x80000000 | (-key))
    return np.uint32(b).view(np.float32)


def qlora_table() -> np.ndarray:
    """The QLoRA NF4 construction: quantiles of N(0,1) at evenly spaced probabilities.

    8 positive values at linspace(delta, 1/2, 9) without its last point, 7 negative values at
    linspace(delta, 1/2, 8) without its last point, and 0; all divided by the largest.  delta =
    0.9677083 is the published offset (1 - (1/32 + 1/30) / 2), spaced in binary32 as published.
    """
    from scipy.stats import norm
    d = np.float32(0.9677083)
    pos = norm.ppf(np.linspace(d, np.float32(0.5), 9, dtype=np.float32)[:-1].astype(np.float64))
    neg = -norm.ppf(np.linspace(d, np.float32(0.5), 8, dtype=np.float32)[:-1].astype(np.float64))
    v = np.sort(np.concatenate([pos, neg, [0.0]]))
    return v / v.max()


def decision_thresholds(table: np.ndarray) -> np.ndarray:
    """For each neighbour pair (i, i+1): the smallest binary32 r with |r-T[i+1]| < |r-T[i]| (fp32).

    Between T[i] and T[i+1] the fp32 distance to T[i] never decreases and the distance to T[i+1]
    never increases as r grows, so the predicate flips once and bisection over the ordered bit
    patterns finds the flip.  Equality keeps the lower code, hence the strict comparison.
    """
    t = np.asarray(table, np.float32)
    thr = np.empty(15, np.float32)
    for i in range(15):
        def closer_to_upper(key):
            r = from_key(key)
            return np.abs(np.float32(r - t[i + 1])) < np.abs(np.float32(r - t[i]))
        lo, hi = ordered_key(t[i]), ordered_key(t[i + 1])
        assert not closer_to_upper(lo) and closer_to_upper(hi)
        while hi - lo > 1:
            mid = (lo + hi) // 2
            if closer_to_upper(mid):
                hi = mid
            else:
                lo = mid
        thr[i] = from_key(hi)
    return thr


def codes_from_thresholds(r: np.ndarray, thr: np.ndarray) -> np.ndarray:
    return np.searchsorted(thr, np.asarray(r, np.float32), side="right").astype(np.uint8)


def unpack_low_nibble_first(codes: np.ndarray) -> np.ndarray:
    """[N, K/2] bytes -> [N, K] codes; weight 2j is the low nibble of byte j."""
    out = np.empty((codes.shape[0], codes.shape[1] * 2), np.uint8)
    out[:, 0::2] = codes & 0x0F
    out[:, 1::2] = codes >> 4
    return out


# ------------------------------------------------------------------------------------------------
# pins
# ------------------------------------------------------------------------------------------------
def pin_table(o):
    assert np.array_equal(o.table(), qlora_published_table()), "table must equal the published literals"
    t = o.table().astype(np.float64)
    assert np.all(np.diff(t) > 0), "table must be strictly increasing"
    assert t[0] == -1.0 and t[7] == 0.0 and t[15] == 1.0
    # The published literals are the construction rounded to binary32 (|error| <= 1 ulp at 1.0).
    assert np.max(np.abs(t - qlora_table())) <= 1.2e-7


def _f16_sample_patterns(rng) -> np.ndarray:
    """Every binary32 exponent with edge mantissas plus random ones; both signs."""
    parts = []
    edge = np.array([0, 1, 2, 0xFFF, 0x1000, 0x1001, 0x1FFF, 0x2000, 0x2001, 0x3FFF, 0x7FFFFF,
                     0x7FFFFE, 0x7FE000, 0x7FF000, 0x7FDFFF], np.uint32)
    for e in range(0, 255):
        mant = np.concatenate([edge, rng.integers(0, 1 << 23, 2048, dtype=np.uint32)])
        parts.append((np.uint32(e) << 23) | mant)
    p = np.concatenate(parts)
    return np.concatenate([p, p | np.uint32(0x80000000)])


def pin_f16(o):
    """fp32 -> fp16 RNE against numpy's cast on every exponent (edge and random mantissas)."""
    rng = np.random.default_rng(11)
    for bits in [_f16_sample_patterns(rng)]:
        f = f32_from_bits(bits)
        with np.errstate(over="ignore"):
            got, want = o.f32_to_f16(f), f16_bits_numpy(f)
        bad = np.flatnonzero(got != want)
        assert bad.size == 0, f"fp16 rounding differs at {hex(int(bits[bad[0]]))}: {got[bad[0]]:#x} vs {want[bad[0]]:#x}"


def pin_bf16(o, exhaustive: bool = False):
    """fp32 -> bf16 RNE against torch's cast (finite values)."""
    rng = np.random.default_rng(12)
    chunks = [_f16_sample_patterns(rng)]
    chunks[0] = chunks[0][(chunks[0] & np.uint32(0x7F800000)) != np.uint32(0x7F800000)]
    if exhaustive:
        for e in (0, 1, 2, 100, 126, 127, 200, 253, 254):
            base = np.arange(1 << 23, dtype=np.uint32) | (np.uint32(e) << 23)
            chunks += [base, base | np.uint32(0x80000000)]
    for bits in chunks:
        f = f32_from_bits(bits)
        got, want = o.f32_to_bf16(f), bf16_bits_torch(f)
        bad = np.flatnonzero(got != want)
        assert bad.size == 0, f"bf16 rounding differs at {hex(int(bits[bad[0]]))}"


def pin_code_windows(o, half_width: int = 1 << 15):
    """Nearest code near every decision threshold and at the special points."""
    t = o.table()
    thr = decision_thresholds(qlora_published_table())
    for i in range(15):
        k0 = ordered_key(thr[i])
        keys = np.arange(k0 - half_width, k0 + half_width, dtype=np.int64)
        bits = np.where(keys >= 0, keys, 0x80000000 | (-keys)).astype(np.uint32)
        r = f32_from_bits(bits)
        got = o.nf4_code(r)
        want = codes_from_thresholds(r, thr)
        bad = np.flatnonzero(got != want)
        assert bad.size == 0, f"code differs near threshold {i} at r={r[bad[0]]!r}: {got[bad[0]]} vs {want[bad[0]]}"
        # fp32 ties in the window go to the lower index
        d_lo = np.abs((r - t[i]).astype(np.float32))
        d_hi = np.abs((r - t[i + 1]).astype(np.float32))
        tie = np.flatnonzero(d_lo == d_hi)
        assert np.all(got[tie] == i)
    special = np.array([-1.0, 1.0, 0.0, -0.0], np.float32)
    assert list(o.nf4_code(special)) == [0, 15, 7, 7]
    assert list(o.nf4_code(t)) == list(range(16))


def qlora_published_table() -> np.ndarray:
    """The QLoRA NF4 literals as published (Dettmers et al., 2023, appendix), read from the
    golden fixture so that this module does not restate the oracle's table source."""
    vals = []
    with open(os.path.join(GOLDEN, "nf4_table_qlora.txt")) as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if line:
                vals.append(float(line))
    assert len(vals) == 16
    return np.array(vals, np.float32)


def code_sweep_chunk(args):
    """Worker for the exhaustive sweep: (lib_path, lo_key, hi_key) -> first mismatch or None.

    Keys are ordered binary32 patterns, so the expected code is constant between consecutive
    threshold keys; each constant run is compared as a whole."""
    lib_path, lo, hi = args
    o = oracle_mod.Oracle(lib_path)
    thr = decision_thresholds(qlora_published_table())
    thr_keys = [ordered_key(t) for t in thr]
    keys = np.arange(lo, hi, dtype=np.int64)
    bits = np.where(keys >= 0, keys, 0x80000000 | (-keys)).astype(np.uint32)
    r = f32_from_bits(bits)
    got = o.nf4_code(r)
    cuts = [lo] + [k for k in thr_keys if lo < k < hi] + [hi]
    for a, b in zip(cuts[:-1], cuts[1:]):
        want = sum(1 for k in thr_keys if k <= a)
        seg = got[a - lo:b - lo]
        bad = np.flatnonzero(seg != want)
        if bad.size:
            return (float(r[a - lo + bad[0]]), int(seg[bad[0]]), want)
    return None


def f16_sweep_chunk(args):
    """Worker for the exhaustive fp16 sweep: every mantissa of one exponent field, both signs."""
    lib_path, e = args
    o = oracle_mod.Oracle(lib_path)
    base = np.arange(1 << 23, dtype=np.uint32) | (np.uint32(e) << 23)
    for bits in (base, base | np.uint32(0x80000000)):
        f = f32_from_bits(bits)
        with np.errstate(over="ignore"):
            got, want = o.f32_to_f16(f), f16_bits_numpy(f)
        bad = np.flatnonzero(got != want)
        if bad.size:
            return hex(int(bits[bad[0]]))
    return None


def pin_quantize_exact(o, groups: int = 2048):
    """Quantize random groups and compare with a float64 midpoint search (exact except within a
    tiny band around each midpoint, which is skipped) and numpy's fp16 cast of the absmax."""
    rng = np.random.default_rng(21)
    t = qlora_published_table().astype(np.float64)
    mids = (t[:-1] + t[1:]) / 2.0
    w = (rng.standard_normal((groups, 64)) * 0.02).astype(np.float32)
    w[::7] = rng.standard_normal((w[::7].shape[0], 64)).astype(np.float32) * np.float32(3.0)  # other scales
    w[5, :] = 0.0                       # all-zero group
    w[9, 3] = -np.abs(w[9]).max() * 2   # negative maximum
    codes, scales = o.quantize(w.reshape(groups // 4, 256))
    codes = unpack_low_nibble_first(codes).reshape(groups, 64)
    scales = scales.reshape(groups)
    s = np.abs(w).max(axis=1)
    assert np.array_equal(scales, f16_bits_numpy(s)), "scale must be fp16 round-to-nearest of the fp32 absmax"
    r = w.astype(np.float64) / np.where(s > 0, s, 1.0).astype(np.float64)[:, None]
    want = np.searchsorted(mids, r, side="left").astype(np.uint8)
    want[s == 0] = 7
    near = np.min(np.abs(r[..., None] - mids), axis=-1) < 2.0 ** -20
    ok = (codes == want) | near
    bad = np.argwhere(~ok)
    assert bad.size == 0, f"code differs at group {bad[0][0]} element {bad[0][1]}"
    # the element holding the absmax maps to code 0 or 15
    amax = np.argmax(np.abs(w), axis=1)
    row = np.arange(groups)
    nz = s > 0
    assert np.all(codes[row[nz], amax[nz]] == np.where(w[row[nz], amax[nz]] > 0, 15, 0))


def pin_golden_pack(o):
    """Hand-derived example: a 64-weight group with w_k = 2 * T[k mod 16] has absmax 2 (exactly an
    fp16), w/s = T[k mod 16] exactly, so code k mod 16; bytes follow low-nibble-first packing."""
    exp_bytes, exp_scale = [], None
    with open(os.path.join(GOLDEN, "nf4_pack_example.txt")) as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, val = line.split("=")
            if key.strip() == "scale_bits":
                exp_scale = int(val, 16)
            elif key.strip() == "bytes":
                exp_bytes = [int(b, 16) for b in val.split()]
    t = qlora_published_table()
    w = (np.float32(2.0) * t[np.arange(64) % 16]).astype(np.float32)[None, :]
    codes, scales = o.quantize(w)
    assert int(scales[0, 0]) == exp_scale
    assert list(codes[0]) == exp_bytes


def pin_payload_ratio(o):
    """Codes + fp16 scales of an aligned matrix are 2 / (0.5 + 2/64) = 3.7647x smaller than bf16;
    the deep-fold README (format paragraph) prints about 3.76x."""
    w = np.zeros((8, 128), np.float32)
    codes, scales = o.quantize(w)
    ratio = (w.size * 2) / (codes.nbytes + scales.nbytes)
    assert abs(ratio - 2.0 / (0.5 + 2.0 / 64.0)) < 1e-12 and round(ratio, 2) == 3.76


def pin_dequant_exhaustive(o):
    """Every code against every finite fp16 scale: bf16(fp32(T[c] * scale)).  The exact product of a
    24-bit and an 11-bit significand fits in float64, numpy rounds it to binary32, torch to bf16."""
    t = qlora_published_table()
    scale_bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    finite = (scale_bits & 0x7C00) != 0x7C00
    scale_bits = scale_bits[finite]
    n = scale_bits.size
    # byte j (mod 16) holds code j in its low nibble and code 15 - j in its high nibble
    codes = np.tile(np.array([c | ((15 - c) << 4) for c in range(16)], np.uint8), 2)  # 64 codes
    codes = np.tile(codes, (n, 1))
    got = o.dequant(codes, scale_bits[:, None])
    sval = scale_bits.view(np.float16).astype(np.float64)
    j = np.arange(64) // 2 % 16
    kcode = np.where(np.arange(64) % 2 == 0, j, 15 - j)
    prod64 = t.astype(np.float64)[kcode][None, :] * sval[:, None]
    want = bf16_bits_torch(prod64.astype(np.float32))
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"dequant differs at scale {scale_bits[bad[0][0]]:#x} code {kcode[bad[0][1]]}"


def pin_roundtrip(o):
    """Invariants tying quantize and dequant together."""
    rng = np.random.default_rng(31)
    w = (rng.standard_normal((64, 256)) * 0.02).astype(np.float32)
    codes, scales = o.quantize(w)
    w_hat = o.dequant(codes, scales)
    c = unpack_low_nibble_first(codes)
    wf = oracle_mod.bf16_bits_to_f32(w_hat)
    assert np.all(wf[c == 7] == 0.0), "code 7 dequantizes to exactly 0"
    # the group's absmax element dequantizes to +-bf16(fp16(s))
    g = w.reshape(64, 4, 64)
    amax = np.argmax(np.abs(g), axis=2)
    sf = scales.view(np.float16).astype(np.float32)
    for n in range(64):
        for j in range(4):
            k = j * 64 + amax[n, j]
            want = np.float32(np.sign(w[n, k])) * oracle_mod.bf16_bits_to_f32(bf16_bits_torch(sf[n, j:j + 1]))[0]
            assert wf[n, k] == want
    # for a fixed positive scale the dequantized value increases with the code
    one = np.array([[c | (c << 4) for c in range(16)] * 2], np.uint8)
    for sb in (0x3C00, 0x2E66, 0x0001, 0x7BFF, 0x2A3F):
        v = oracle_mod.bf16_bits_to_f32(o.dequant(one, np.array([[sb]], np.uint16)))[0, 0:32:2]
        assert np.all(np.diff(v.astype(np.float64)) >= 0)
        assert np.all(np.diff(v[v != 0].astype(np.float64)) > 0)
    # re-quantizing w_hat / scale maps back to the same codes when the scale is fp16-exact
    g2 = (w.reshape(64, 4, 64) / np.abs(w.reshape(64, 4, 64)).max(axis=2, keepdims=True)
          * np.float32(0.04)).astype(np.float32)
    idx = np.argmax(np.abs(g2), axis=2)
    for n in range(64):
        for j in range(4):
            g2[n, j, idx[n, j]] = np.float32(np.sign(g2[n, j, idx[n, j]]) * 0.046875)  # fp16-exact absmax
    w2 = g2.reshape(64, 256)
    codes2, scales2 = o.quantize(w2)
    assert np.all(scales2 == f16_bits_numpy(np.float32(0.046875)))
    r = (oracle_mod.bf16_bits_to_f32(o.dequant(codes2, scales2)) / np.float32(0.046875)).astype(np.float32)
    assert np.array_equal(o.nf4_code(r), unpack_low_nibble_first(codes2))


def pin_linear(o):
    """fp64 linear against numpy's float64 matmul, unit vectors and exact rationals."""
    rng = np.random.default_rng(41)
    from nf4_weight_only_gb300 import synth
    m, n, k = 5, 33, 320
    w = synth.weights(7, n, k)
    x = synth.activations_bf16(8, m, k)
    codes, scales = o.quantize(w)
    w_hat = oracle_mod.bf16_bits_to_f32(o.dequant(codes, scales)).astype(np.float64)
    xf = oracle_mod.bf16_bits_to_f32(x).astype(np.float64)
    y64, mag = o.linear(x, codes, scales, nthreads=3)
    ref = xf @ w_hat.T
    refmag = np.abs(xf) @ np.abs(w_hat).T
    assert np.all(np.abs(y64 - ref) <= 1e-12 * refmag + 1e-300)
    assert np.all(np.abs(mag - refmag) <= 1e-12 * refmag + 1e-300)
    # one-hot activations pick out a column of w_hat exactly
    eye = np.zeros((4, k), np.uint16)
    cols = [0, 63, 64, k - 1]
    for i, c in enumerate(cols):
        eye[i, c] = 0x3F80  # bf16 1.0
    ye, _ = o.linear(eye, codes, scales)
    for i, c in enumerate(cols):
        assert np.array_equal(ye[i], w_hat[:, c])
    # exact rational sum on a small case
    ys, _ = o.linear(x[:1, :128], codes[:3, :64], scales[:3, :2])
    for j in range(3):
        exact = sum(Fraction(float(xf[0, kk])) * Fraction(float(w_hat[j, kk])) for kk in range(128))
        assert abs(Fraction(float(ys[0, j])) - exact) <= Fraction(128, 2 ** 52) * sum(
            abs(Fraction(float(xf[0, kk])) * Fraction(float(w_hat[j, kk]))) for kk in range(128))
    # the sampled-entry call agrees with the full call bit for bit
    mi = rng.integers(0, m, 40)
    ni = rng.integers(0, n, 40)
    ye2, me2 = o.linear_entries(x, codes, scales, mi, ni)
    assert np.array_equal(ye2, y64[mi, ni]) and np.array_equal(me2, mag[mi, ni])
    # thread count does not change a bit
    y1, _ = o.linear(x, codes, scales, nthreads=1)
    assert np.array_equal(y1, y64)


def pin_embed(o):
    """Packed embedding rows against numpy's gather of the (exhaustively pinned) dequantized table;
    ids outside the table give zero rows and are counted."""
    from nf4_weight_only_gb300 import synth
    v, k = 37, 192
    codes, scales = o.quantize(synth.weights(12, v, k))
    table = o.dequant(codes, scales)
    rng = np.random.default_rng(13)
    ids = np.concatenate([[0, v - 1, 5, 5], rng.integers(0, v, 60)]).astype(np.int32)
    rows, bad = o.embed(ids, codes, scales)
    assert bad == 0 and np.array_equal(rows, table[ids])
    assert np.array_equal(rows[2], rows[3])  # a repeated id gives the same row
    odd = np.array([3, -1, v, 2 ** 31 - 1, v - 1], np.int32)
    rows, bad = o.embed(odd, codes, scales)
    assert bad == 3
    assert np.array_equal(rows[[0, 4]], table[[3, v - 1]]) and not rows[1:4].any()
    rows, bad = o.embed(np.zeros(0, np.int32), codes, scales)
    assert rows.shape == (0, k) and bad == 0


FAST_PINS = [pin_table, pin_f16, pin_bf16, pin_code_windows, pin_quantize_exact, pin_golden_pack,
             pin_payload_ratio, pin_dequant_exhaustive, pin_roundtrip, pin_linear, pin_embed]
