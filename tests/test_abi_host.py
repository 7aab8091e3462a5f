"""Host-side checks of the C ABI (no GPU needed): the library builds, loads, exports every symbol
that include/nf4.h declares, and rejects bad arguments before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from nf4_weight_only_gb300 import build
    path = build.build()
    import nf4_weight_only_gb300 as nf4
    return nf4.load(path)


def header_functions():
    text = open(os.path.join(ROOT, "include", "nf4.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(nf4_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = header_functions()
    assert {"nf4_quantize", "nf4_dequant", "nf4_linear", "nf4_linear_grouped", "nf4_check_device_error",
            "nf4_status_str", "nf4_abi_version"} <= set(names)
    for name in names:
        assert hasattr(lib, name), f"{name} declared in include/nf4.h but not exported"
    import nf4_weight_only_gb300 as nf4
    assert set(nf4.EXPORTED) == set(names)


def test_version_and_status_strings(lib):
    assert lib.nf4_abi_version() == 3
    for code in range(9):
        s = lib.nf4_status_str(code).decode()
        assert s.startswith("NF4_")
    assert b"unknown" in lib.nf4_status_str(99)


# Fake, never-dereferenced device addresses: every case below fails validation first.
A = 0x7F0000000000
B = 0x7F1000000000
C = 0x7F2000000000
D = 0x7F3000000000
vp = ctypes.c_void_p


def linear(lib, x, codes, scales, y, m, n, k):
    return lib.nf4_linear(vp(x), vp(codes), vp(scales), vp(y), m, n, k, None)


@pytest.mark.parametrize("m,n,k,want", [
    (1, 1, 0, 2), (1, 1, 63, 2), (1, 1, 96, 2), (-1, 4, 64, 2), (1, -4, 64, 2),
    (1, 1, -64, 2), (1 << 31, 1, 64, 2), (1, 1 << 31, 64, 2), (1, 1, 1 << 40, 2),
])
def test_linear_shape_errors(lib, m, n, k, want):
    assert linear(lib, A, B, C, D, m, n, k) == want


def test_linear_empty_is_ok_without_device(lib):
    assert linear(lib, 0, 0, 0, 0, 0, 5, 64) == 0
    assert linear(lib, 0, 0, 0, 0, 3, 0, 64) == 0


def test_linear_null_align_alias(lib):
    assert linear(lib, 0, B, C, D, 1, 4, 64) == 1
    assert linear(lib, A, B, 0, D, 1, 4, 64) == 1
    assert linear(lib, A + 2, B, C, D, 1, 4, 64) == 3
    assert linear(lib, A, B + 8, C, D, 1, 4, 64) == 3
    assert linear(lib, A, B, C, D + 4, 1, 4, 64) == 3
    # y overlapping x, codes or scales
    assert linear(lib, A, B, C, A + 64, 1, 4, 64) == 4
    assert linear(lib, A, B, C, B + 16, 1, 4, 64) == 4
    assert linear(lib, A, B, C, C, 1, 4, 64) == 4


def test_quantize_dequant_errors(lib):
    q = lib.nf4_quantize
    assert q(vp(A), 4, 100, vp(B), vp(C), None) == 2
    assert q(vp(A), -1, 64, vp(B), vp(C), None) == 2
    assert q(vp(0), 4, 64, vp(B), vp(C), None) == 1
    assert q(vp(A + 4), 4, 64, vp(B), vp(C), None) == 3
    assert q(vp(A), 4, 64, vp(A + 512), vp(C), None) == 4   # codes inside w
    assert q(vp(A), 4, 64, vp(B), vp(B + 16), None) == 4    # scales inside codes
    assert q(vp(0), 0, 64, vp(0), vp(0), None) == 0        # empty
    d = lib.nf4_dequant
    assert d(vp(B), vp(C), 4, 65, vp(D), None) == 2
    assert d(vp(B), vp(0), 4, 64, vp(D), None) == 1
    assert d(vp(B), vp(C), 4, 64, vp(D + 2), None) == 3
    assert d(vp(B), vp(C), 4, 64, vp(B), None) == 4


def test_valid_call_without_gpu_fails_cleanly(lib):
    """Past validation the library asks the runtime for the device; with no GPU it must return an
    error status (never crash)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert linear(lib, A, B, C, D, 1, 4, 64) in (5, 6)


def test_diag_wait_rejects_unbounded_limits(lib):
    """The diagnostic wait takes a limit in [1, 2^31] ns and the wait-limit setter one in [0, 2^36] ns;
    anything else is rejected on the host."""
    lib.nf4_diag_bounded_wait.argtypes = [ctypes.c_int64, vp]
    for ns in (0, -1, (1 << 31) + 1, 1 << 62):
        assert lib.nf4_diag_bounded_wait(ns, None) == 2  # NF4_ERR_SHAPE
    lib.nf4_diag_set_wait_limit.argtypes = [ctypes.c_int64, vp]
    for ns in (-1, (1 << 36) + 1, 1 << 62):
        assert lib.nf4_diag_set_wait_limit(ns, None) == 2


def test_noalloc_size_matches_header(lib):
    """The binding reads the no-alloc array's size from the library, which must equal the header's."""
    text = open(os.path.join(ROOT, "include", "nf4.h")).read()
    m = re.search(r"#define NF4_NOALLOC_SLOT_BYTES \((\d+) \* (\d+) \* (\d+)\)", text)
    assert m, "NF4_NOALLOC_SLOT_BYTES not found in include/nf4.h"
    want = int(m.group(1)) * int(m.group(2)) * int(m.group(3))
    import nf4_weight_only_gb300 as nf4
    assert nf4.noalloc_slot_bytes() == want


def test_binding_raises_without_library(tmp_path):
    import nf4_weight_only_gb300 as nf4
    with pytest.raises(RuntimeError, match="missing"):
        nf4.load(str(tmp_path / "nope.so"))


def test_grouped_validation(lib):
    arr = ctypes.c_void_p * 2
    ns = (ctypes.c_int64 * 2)(16, 8)
    g = lib.nf4_linear_grouped
    c2 = arr(B, B + 4096)
    s2 = arr(C, C + 4096)
    y2 = arr(D, D + 4096)
    args = lambda x, m, k, cnt, c, s, y, n: g(vp(x), m, k, cnt, ctypes.cast(c, vp), ctypes.cast(s, vp),
                                             ctypes.cast(y, vp), ctypes.cast(n, vp), None)
    assert args(A, 1, 64, 0, c2, s2, y2, ns) == 2          # count outside 1..8
    assert args(A, 1, 64, 9, c2, s2, y2, ns) == 2
    assert args(A, 1, 100, 2, c2, s2, y2, ns) == 2         # K not a multiple of 64
    assert g(vp(A), 1, 64, 2, None, ctypes.cast(s2, vp), ctypes.cast(y2, vp), ctypes.cast(ns, vp), None) == 1
    assert args(A + 2, 1, 64, 2, c2, s2, y2, ns) == 3      # misaligned x
    assert args(A, 1, 64, 2, c2, s2, arr(D, D + 16), ns) == 4  # y0 (32 bytes) and y1 overlap
    assert args(A, 1, 64, 2, c2, s2, arr(D, B + 16), ns) == 4  # y1 inside codes[0]
    assert args(A, 0, 64, 2, c2, s2, y2, ns) == 0          # empty


def test_embed_validation(lib):
    e = lib.nf4_embed
    e.argtypes = [vp, ctypes.c_int64, vp, vp, ctypes.c_int64, ctypes.c_int64, vp, vp]
    assert e(vp(0), 0, vp(0), vp(0), 0, 64, vp(0), None) == 0          # no ids: no-op
    assert e(vp(A), 4, vp(B), vp(C), 10, 100, vp(D), None) == 2        # K not a multiple of 64
    assert e(vp(A), -1, vp(B), vp(C), 10, 64, vp(D), None) == 2
    assert e(vp(A), 4, vp(B), vp(C), -1, 64, vp(D), None) == 2
    assert e(vp(0), 4, vp(B), vp(C), 10, 64, vp(D), None) == 1        # ids NULL
    assert e(vp(A), 4, vp(0), vp(C), 10, 64, vp(D), None) == 1        # codes NULL
    assert e(vp(A), 4, vp(B), vp(C), 10, 64, vp(0), None) == 1        # out NULL
    assert e(vp(A + 4), 4, vp(B), vp(C), 10, 64, vp(D), None) == 3
    assert e(vp(A), 4, vp(B), vp(C), 10, 64, vp(D + 2), None) == 3
    assert e(vp(A), 4, vp(B), vp(C), 10, 64, vp(A), None) == 4         # out over ids
    assert e(vp(A), 4, vp(B), vp(C), 10, 64, vp(B + 32), None) == 4    # out inside codes
    assert e(vp(A), 4, vp(B), vp(C), 10, 64, vp(C), None) == 4         # out over scales


def test_ring_validation(lib):
    """Ring calls reject bad arguments before any CUDA call (the ring pointer is never touched)."""
    h = ctypes.c_void_p(0)
    assert lib.nf4_ring_create(1 << 20, None) == 1
    assert lib.nf4_ring_create(0, ctypes.byref(h)) == 2 and h.value is None
    assert lib.nf4_ring_create(-5, ctypes.byref(h)) == 2
    assert lib.nf4_ring_run(None, vp(A), 1, None) == 1
    assert lib.nf4_ring_run(vp(A), vp(B), -1, None) == 2
    assert lib.nf4_ring_run(vp(A), None, 0, None) == 0   # empty list: no-op
    assert lib.nf4_ring_run(vp(A), None, 2, None) == 1
    assert lib.nf4_ring_destroy(None) == 0
