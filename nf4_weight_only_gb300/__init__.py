"""NF4 weight-only linear layer for NVIDIA GB300 (sm_103a): thin Python binding of libnf4.so.

The library (``csrc/``, C ABI in ``include/nf4.h``) does all the work.  This module only marshals
torch tensors (device memory and streams) into the C calls of the same names and raises
``NF4Error`` on a non-OK status.  There is no CPU fallback: if ``libnf4.so`` has not been built
(``nf4_weight_only_gb300.build.build()``), every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import build as _build

GROUP = 64
LIB_PATH = _build.LIB_PATH

STATUS_NAMES = {0: "NF4_OK", 1: "NF4_ERR_NULL", 2: "NF4_ERR_SHAPE", 3: "NF4_ERR_ALIGN",
                4: "NF4_ERR_ALIAS", 5: "NF4_ERR_UNSUPPORTED_DEVICE", 6: "NF4_ERR_CUDA", 7: "NF4_ERR_MEMORY",
                8: "NF4_ERR_CAPTURE"}

# Every symbol include/nf4.h declares.
EXPORTED = ("nf4_quantize", "nf4_dequant", "nf4_linear", "nf4_linear_grouped", "nf4_embed",
            "nf4_ring_create", "nf4_ring_run", "nf4_ring_destroy", "nf4_linear_host_noalloc",
            "nf4_check_device_error", "nf4_diag_bounded_wait", "nf4_diag_set_wait_limit", "nf4_status_str",
            "nf4_abi_version", "nf4_noalloc_slot_bytes", "nf4_last_cuda_error")


class HostLinear(ctypes.Structure):
    """nf4_host_linear: one linear of a streamed list (x, y on the device; codes, scales pinned host)."""
    _fields_ = [("x", ctypes.c_void_p), ("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("y", ctypes.c_void_p), ("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64)]


class NF4Error(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_str(status)}")


_lib: Optional[ctypes.CDLL] = None


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libnf4.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is missing: build it with nf4_weight_only_gb300.build.build() "
                           "(no CPU fallback exists)")
    lib = ctypes.CDLL(p)
    vp, i64, ci = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.nf4_quantize.argtypes = [vp, i64, i64, vp, vp, vp]
    lib.nf4_quantize.restype = ci
    lib.nf4_dequant.argtypes = [vp, vp, i64, i64, vp, vp]
    lib.nf4_dequant.restype = ci
    lib.nf4_linear.argtypes = [vp, vp, vp, vp, i64, i64, i64, vp]
    lib.nf4_linear.restype = ci
    lib.nf4_linear_grouped.argtypes = [vp, i64, i64, ci, vp, vp, vp, vp, vp]
    lib.nf4_linear_grouped.restype = ci
    lib.nf4_embed.argtypes = [vp, i64, vp, vp, i64, i64, vp, vp]
    lib.nf4_embed.restype = ci
    lib.nf4_ring_create.argtypes = [i64, ctypes.POINTER(ctypes.c_void_p)]
    lib.nf4_ring_create.restype = ci
    lib.nf4_ring_run.argtypes = [vp, vp, i64, vp]
    lib.nf4_ring_run.restype = ci
    lib.nf4_ring_destroy.argtypes = [vp]
    lib.nf4_ring_destroy.restype = ci
    lib.nf4_linear_host_noalloc.argtypes = [vp, vp, vp, vp, i64, i64, i64, vp]
    lib.nf4_linear_host_noalloc.restype = ci
    lib.nf4_status_str.argtypes = [ci]
    lib.nf4_status_str.restype = ctypes.c_char_p
    lib.nf4_check_device_error.argtypes = [ctypes.POINTER(ctypes.c_int)]
    lib.nf4_check_device_error.restype = ci
    lib.nf4_diag_bounded_wait.argtypes = [i64, vp]
    lib.nf4_diag_bounded_wait.restype = ci
    lib.nf4_diag_set_wait_limit.argtypes = [i64, vp]
    lib.nf4_diag_set_wait_limit.restype = ci
    lib.nf4_noalloc_slot_bytes.argtypes = []
    lib.nf4_noalloc_slot_bytes.restype = i64
    lib.nf4_last_cuda_error.argtypes = []
    lib.nf4_last_cuda_error.restype = ctypes.c_char_p
    lib.nf4_abi_version.argtypes = []
    lib.nf4_abi_version.restype = ci
    if path is None:
        _lib = lib
    return lib


def status_str(status: int) -> str:
    try:
        return load().nf4_status_str(status).decode()
    except RuntimeError:
        return STATUS_NAMES.get(status, f"status {status}")


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _ptr(t: Optional[torch.Tensor]) -> ctypes.c_void_p:
    if t is None:
        return ctypes.c_void_p(0)
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _check(status: int, what: str) -> None:
    if status != 0:
        if status == 6:  # NF4_ERR_CUDA: name the CUDA error behind it
            raise NF4Error(status, f"{what} [{load().nf4_last_cuda_error().decode()}]")
        raise NF4Error(status, what)


def nf4_quantize(w: torch.Tensor, codes: torch.Tensor, scales: torch.Tensor, stream=None) -> None:
    """w fp32 [N, K] -> codes uint8 [N, K/2], scales fp16 [N, K/64] (all CUDA tensors)."""
    n, k = w.shape
    _check(load().nf4_quantize(_ptr(w), n, k, _ptr(codes), _ptr(scales), _stream(stream)), "nf4_quantize")


def nf4_dequant(codes: torch.Tensor, scales: torch.Tensor, w_hat: torch.Tensor, stream=None) -> None:
    """codes [N, K/2], scales [N, K/64] -> w_hat bf16 [N, K]."""
    n, k = codes.shape[0], codes.shape[1] * 2
    _check(load().nf4_dequant(_ptr(codes), _ptr(scales), n, k, _ptr(w_hat), _stream(stream)), "nf4_dequant")


def nf4_linear(x: torch.Tensor, codes: torch.Tensor, scales: torch.Tensor, y: torch.Tensor,
               stream=None) -> None:
    """y[M, N] = x[M, K] * w_hat^T (bf16 in, bf16 out)."""
    m, k = x.shape
    n = codes.shape[0]
    _check(load().nf4_linear(_ptr(x), _ptr(codes), _ptr(scales), _ptr(y), m, n, k, _stream(stream)),
           "nf4_linear")


def nf4_linear_grouped(x: torch.Tensor, codes, scales, ys, stream=None) -> None:
    """ys[i][M, N_i] = x[M, K] * w_hat_i^T for the lists codes, scales, ys (same length, <= 8)."""
    m, k = x.shape
    n = len(codes)
    if not (len(scales) == len(ys) == n):
        raise ValueError("codes, scales and ys must have the same length")
    arr = ctypes.c_void_p * n
    c_arr = arr(*[_ptr(c).value for c in codes])
    s_arr = arr(*[_ptr(s).value for s in scales])
    y_arr = arr(*[_ptr(y).value for y in ys])
    ns = (ctypes.c_int64 * n)(*[c.shape[0] for c in codes])
    _check(load().nf4_linear_grouped(_ptr(x), m, k, n, ctypes.cast(c_arr, ctypes.c_void_p),
                                     ctypes.cast(s_arr, ctypes.c_void_p), ctypes.cast(y_arr, ctypes.c_void_p),
                                     ctypes.cast(ns, ctypes.c_void_p), _stream(stream)), "nf4_linear_grouped")


def nf4_embed(ids: torch.Tensor, codes: torch.Tensor, scales: torch.Tensor, out: torch.Tensor, stream=None) -> None:
    """out[i] = w_hat[ids[i]] for int32 ids, codes [V, K/2], scales [V, K/64] -> out bf16 [n, K]."""
    v, k = codes.shape[0], codes.shape[1] * 2
    _check(load().nf4_embed(_ptr(ids), ids.numel(), _ptr(codes), _ptr(scales), v, k, _ptr(out), _stream(stream)),
           "nf4_embed")


def nf4_ring_create(slot_bytes: int) -> int:
    """A ring of two device slots of `slot_bytes` each (returns the opaque handle)."""
    h = ctypes.c_void_p(0)
    _check(load().nf4_ring_create(slot_bytes, ctypes.byref(h)), "nf4_ring_create")
    return h.value


def nf4_ring_run(ring: int, ops, stream=None) -> None:
    """Stream a list of linears (x, codes, scales, y) through the ring: codes [N, K/2] and scales
    [N, K/64] in pinned host memory, x [M, K] and y [M, N] on the device."""
    arr = (HostLinear * max(1, len(ops)))()
    for i, (x, codes, scales, y) in enumerate(ops):
        arr[i] = HostLinear(_ptr(x).value, _ptr(codes).value, _ptr(scales).value, _ptr(y).value,
                            x.shape[0], codes.shape[0], x.shape[1])
    _check(load().nf4_ring_run(ctypes.c_void_p(ring), ctypes.cast(arr, ctypes.c_void_p), len(ops), _stream(stream)),
           "nf4_ring_run")


def nf4_ring_destroy(ring: int) -> None:
    _check(load().nf4_ring_destroy(ctypes.c_void_p(ring)), "nf4_ring_destroy")


class Ring:
    """Two reusable device slots through which packed weights in pinned host memory are streamed."""

    def __init__(self, slot_bytes: int):
        self.handle = nf4_ring_create(slot_bytes)
        self.slot_bytes = slot_bytes

    @staticmethod
    def bytes_needed(n: int, k: int) -> int:
        return (n * k // 2 + 255) // 256 * 256 + n * (k // GROUP) * 2

    def run(self, ops, stream=None) -> None:
        nf4_ring_run(self.handle, ops, stream)

    def close(self) -> None:
        if self.handle:
            nf4_ring_destroy(self.handle)
            self.handle = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()


def noalloc_slot_bytes() -> int:
    """Size of nf4_linear_host_noalloc's static device array, as the built library reports it."""
    return int(load().nf4_noalloc_slot_bytes())


def nf4_linear_host_noalloc(x: torch.Tensor, codes: torch.Tensor, scales: torch.Tensor, y: torch.Tensor,
                            stream=None) -> None:
    """y[M, N] = x[M, K] * w_hat^T with codes [N, K/2] and scales [N, K/64] in pinned host memory,
    staged through the library's static device buffer (no allocation; at most noalloc_slot_bytes())."""
    m, k = x.shape
    n = codes.shape[0]
    _check(load().nf4_linear_host_noalloc(_ptr(x), _ptr(codes), _ptr(scales), _ptr(y), m, n, k, _stream(stream)),
           "nf4_linear_host_noalloc")


def nf4_diag_bounded_wait(ns: int, stream=None) -> None:
    """Launch one thread whose bounded wait on a barrier nothing arrives on runs out after `ns`
    nanoseconds and records code 39 in the device error word (diagnostics)."""
    _check(load().nf4_diag_bounded_wait(int(ns), _stream(stream)), "nf4_diag_bounded_wait")


def nf4_diag_set_wait_limit(ns: int, stream=None) -> None:
    """Set the per-wait wall-clock limit of the kernels' pipeline waits (ns = 0 restores 1 s)."""
    _check(load().nf4_diag_set_wait_limit(int(ns), _stream(stream)), "nf4_diag_set_wait_limit")


def nf4_check_device_error() -> int:
    """Read and clear the device error word (0 = no pipeline wait timed out).  Synchronizes."""
    code = ctypes.c_int(0)
    _check(load().nf4_check_device_error(ctypes.byref(code)), "nf4_check_device_error")
    return code.value


# Convenience wrappers that allocate the outputs with torch.
def quantize(w: torch.Tensor, stream=None):
    n, k = w.shape
    codes = torch.empty((n, k // 2), dtype=torch.uint8, device=w.device)
    scales = torch.empty((n, k // GROUP), dtype=torch.float16, device=w.device)
    nf4_quantize(w, codes, scales, stream)
    return codes, scales


def dequant(codes: torch.Tensor, scales: torch.Tensor, stream=None) -> torch.Tensor:
    w_hat = torch.empty((codes.shape[0], codes.shape[1] * 2), dtype=torch.bfloat16, device=codes.device)
    nf4_dequant(codes, scales, w_hat, stream)
    return w_hat


def embed(ids: torch.Tensor, codes: torch.Tensor, scales: torch.Tensor, stream=None) -> torch.Tensor:
    out = torch.empty((ids.numel(), codes.shape[1] * 2), dtype=torch.bfloat16, device=codes.device)
    nf4_embed(ids, codes, scales, out, stream)
    return out


def linear(x: torch.Tensor, codes: torch.Tensor, scales: torch.Tensor, stream=None) -> torch.Tensor:
    y = torch.empty((x.shape[0], codes.shape[0]), dtype=torch.bfloat16, device=x.device)
    nf4_linear(x, codes, scales, y, stream)
    return y
