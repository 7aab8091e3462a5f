"""NF4 oracle: plain CPU reference of the NF4 weight-only linear layer (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference`` legs of
``bench.py`` may import this package.  The CUDA library never does, and this package never imports
the CUDA library: the two share no code.

The arithmetic lives in ``nf4_oracle.c`` (plain C loops, IEEE binary32 where the definition says
fp32, double precision for the linear).  This module builds it with gcc, loads it with ctypes and
wraps it for numpy arrays.  The acceptance rule for the linear (``within_tolerance``) is stated
here too.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py`` against values fixed
by the mathematics or by independent library routines (numpy / torch casts, exact rational
arithmetic, float64 matmul, the QLoRA quantile construction), and the pins are themselves checked
to catch planted mistakes (``tests/test_oracle_mutants.py``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "nf4_oracle.c")
BUILD_DIR = os.path.join(_HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "liboracle.so")

# -ffp-contract=off: no fused multiply-add may merge the roundings the definitions spell out (gcc
# contracts by default on aarch64).  No -ffast-math, no -march: IEEE semantics on x86-64 and Arm.
CFLAGS = ["-std=c11", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math", "-pthread"]

GROUP = 64


def build(source: str = SOURCE, out: str = LIB_PATH, force: bool = False) -> str:
    """Compile ``source`` into the shared library ``out`` (skipped when ``out`` is newer)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(source)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, "-o", tmp, source, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def _p(a: np.ndarray) -> ctypes.c_void_p:
    return ctypes.c_void_p(a.ctypes.data)


class Oracle:
    """ctypes view of one build of the oracle library (the default build, or a test's variant)."""

    def __init__(self, lib_path: Optional[str] = None):
        path = lib_path or build()
        lib = ctypes.CDLL(path)
        i64, vp = ctypes.c_int64, ctypes.c_void_p
        lib.oracle_nf4_table.argtypes = [vp]
        lib.oracle_f32_to_f16_array.argtypes = [vp, i64, vp]
        lib.oracle_f32_to_bf16_array.argtypes = [vp, i64, vp]
        lib.oracle_nf4_code_array.argtypes = [vp, i64, vp]
        lib.oracle_quantize.argtypes = [vp, i64, i64, vp, vp]
        lib.oracle_quantize.restype = ctypes.c_int
        lib.oracle_dequant.argtypes = [vp, vp, i64, i64, vp]
        lib.oracle_dequant.restype = ctypes.c_int
        lib.oracle_embed.argtypes = [vp, i64, vp, vp, i64, i64, vp]
        lib.oracle_embed.restype = i64
        lib.oracle_linear.argtypes = [vp, vp, vp, i64, i64, i64, vp, vp, ctypes.c_int]
        lib.oracle_linear.restype = ctypes.c_int
        lib.oracle_linear_entries.argtypes = [vp, vp, vp, i64, i64, i64, vp, vp, i64, vp, vp]
        lib.oracle_linear_entries.restype = ctypes.c_int
        self.lib = lib
        self.path = path

    # -- table and roundings ---------------------------------------------------------------
    def table(self) -> np.ndarray:
        out = np.zeros(16, np.float32)
        self.lib.oracle_nf4_table(_p(out))
        return out

    def f32_to_f16(self, a: np.ndarray) -> np.ndarray:
        a = np.ascontiguousarray(a, np.float32)
        out = np.empty(a.shape, np.uint16)
        self.lib.oracle_f32_to_f16_array(_p(a), a.size, _p(out))
        return out

    def f32_to_bf16(self, a: np.ndarray) -> np.ndarray:
        a = np.ascontiguousarray(a, np.float32)
        out = np.empty(a.shape, np.uint16)
        self.lib.oracle_f32_to_bf16_array(_p(a), a.size, _p(out))
        return out

    def nf4_code(self, r: np.ndarray) -> np.ndarray:
        r = np.ascontiguousarray(r, np.float32)
        out = np.empty(r.shape, np.uint8)
        self.lib.oracle_nf4_code_array(_p(r), r.size, _p(out))
        return out

    # -- the three operations --------------------------------------------------------------
    def quantize(self, w: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
        """fp32 [N, K] -> (codes u8 [N, K/2], scales fp16 bits u16 [N, K/64])."""
        w = np.ascontiguousarray(w, np.float32)
        n, k = w.shape
        codes = np.empty((n, k // 2), np.uint8)
        scales = np.empty((n, k // GROUP), np.uint16)
        rc = self.lib.oracle_quantize(_p(w), n, k, _p(codes), _p(scales))
        if rc != 0:
            raise ValueError(f"oracle_quantize: bad shape {w.shape}")
        return codes, scales

    def dequant(self, codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
        """-> bf16 bits u16 [N, K]."""
        codes = np.ascontiguousarray(codes, np.uint8)
        scales = np.ascontiguousarray(scales, np.uint16)
        n, k = codes.shape[0], codes.shape[1] * 2
        out = np.empty((n, k), np.uint16)
        rc = self.lib.oracle_dequant(_p(codes), _p(scales), n, k, _p(out))
        if rc != 0:
            raise ValueError("oracle_dequant: bad shape")
        return out

    def embed(self, ids: np.ndarray, codes: np.ndarray, scales: np.ndarray) -> Tuple[np.ndarray, int]:
        """int32 ids [n] of a V-row table -> (bf16 bits u16 [n, K], number of ids outside [0, V))."""
        ids = np.ascontiguousarray(ids, np.int32)
        codes = np.ascontiguousarray(codes, np.uint8)
        scales = np.ascontiguousarray(scales, np.uint16)
        v, k = codes.shape[0], codes.shape[1] * 2
        out = np.empty((ids.size, k), np.uint16)
        bad = self.lib.oracle_embed(_p(ids), ids.size, _p(codes), _p(scales), v, k, _p(out))
        if bad < 0:
            raise ValueError("oracle_embed: bad shape")
        return out, int(bad)

    def linear(self, x_bf16: np.ndarray, codes: np.ndarray, scales: np.ndarray,
               nthreads: int = 1) -> Tuple[np.ndarray, np.ndarray]:
        """x bf16 bits [M, K] -> (y64 [M, N], abs_sum [M, N]) in float64."""
        x = np.ascontiguousarray(x_bf16, np.uint16)
        codes = np.ascontiguousarray(codes, np.uint8)
        scales = np.ascontiguousarray(scales, np.uint16)
        m, k = x.shape
        n = codes.shape[0]
        if codes.shape[1] * 2 != k:
            raise ValueError("oracle.linear: K mismatch")
        y64 = np.empty((m, n), np.float64)
        mag = np.empty((m, n), np.float64)
        rc = self.lib.oracle_linear(_p(x), _p(codes), _p(scales), m, n, k, _p(y64), _p(mag), nthreads)
        if rc != 0:
            raise ValueError(f"oracle_linear failed ({rc})")
        return y64, mag

    def linear_entries(self, x_bf16: np.ndarray, codes: np.ndarray, scales: np.ndarray,
                       m_idx: np.ndarray, n_idx: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
        """The same sums for the listed (m, n) entries only."""
        x = np.ascontiguousarray(x_bf16, np.uint16)
        codes = np.ascontiguousarray(codes, np.uint8)
        scales = np.ascontiguousarray(scales, np.uint16)
        mi = np.ascontiguousarray(m_idx, np.int64)
        ni = np.ascontiguousarray(n_idx, np.int64)
        m, k = x.shape
        n = codes.shape[0]
        y64 = np.empty(mi.size, np.float64)
        mag = np.empty(mi.size, np.float64)
        rc = self.lib.oracle_linear_entries(_p(x), _p(codes), _p(scales), m, n, k, _p(mi), _p(ni),
                                            mi.size, _p(y64), _p(mag))
        if rc != 0:
            raise ValueError("oracle_linear_entries failed")
        return y64, mag


_default: Optional[Oracle] = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle()
    return _default


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """bf16 bits -> float32 (exact: the bits are the top half of the binary32 pattern)."""
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


def tolerance_bound(y64: np.ndarray, abs_sum: np.ndarray) -> np.ndarray:
    """Per-element acceptance bound of the linear: 2^-8 |y64| + 2^-12 sum_k |x_k w_k|.

    2^-9 |y64| of it is the bf16 output rounding alone; the rest covers fp32 accumulation in any
    order.
    """
    return np.ldexp(np.abs(y64), -8) + np.ldexp(abs_sum, -12)


def within_tolerance(y_bf16: np.ndarray, y64: np.ndarray, abs_sum: np.ndarray):
    """(all_ok, worst ratio |y - y64| / bound, per-element ok mask) for bf16 outputs."""
    y = bf16_bits_to_f32(y_bf16).astype(np.float64)
    bound = tolerance_bound(y64, abs_sum)
    err = np.abs(y - y64)
    ok = err <= bound
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(bound > 0, err / np.where(bound > 0, bound, 1.0), np.where(err > 0, np.inf, 0.0))
    return bool(ok.all()), float(ratio.max(initial=0.0)), ok
