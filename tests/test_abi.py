"""The C-ABI library loads on a host without a GPU, exports every entry point
include/rxl.h declares, and rejects bad arguments before touching CUDA."""
import ctypes
import os
import re

import pytest

import long_context_lm_rel_gb300 as rxl

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "rxl.h")


@pytest.fixture(scope="module")
def lib():
    rxl.build()
    return rxl.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(rxl_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert {"rxl_attn_fwd", "rxl_attn_bwd", "rxl_attn_bwd_workspace_bytes", "rxl_mem_update",
            "rxl_status_string"} <= set(names)
    for n in names:
        assert getattr(lib, n) is not None, n


def test_status_strings(lib):
    for code, name in [(0, "RXL_OK"), (1, "RXL_ERR_INVALID_ARGUMENT"), (2, "RXL_ERR_UNSUPPORTED"),
                       (3, "RXL_ERR_MISALIGNED"), (4, "RXL_ERR_WORKSPACE_TOO_SMALL"), (5, "RXL_ERR_CUDA")]:
        assert rxl.rxl_status_string(code) == name


A = 1 << 20  # a 16-byte-aligned fake address: never dereferenced, calls fail validation first


def fwd_status(lib, desc, ptrs=None):
    p = ptrs or [A] * 8
    return lib.rxl_attn_fwd(ctypes.byref(desc), *p, None)


@pytest.mark.parametrize("field,value,status", [
    ("dh", 32, rxl.RXL_ERR_UNSUPPORTED), ("dtype", 7, rxl.RXL_ERR_UNSUPPORTED),
    ("B", 0, rxl.RXL_ERR_INVALID_ARGUMENT), ("L", 0, rxl.RXL_ERR_INVALID_ARGUMENT),
    ("mem_len", 9, rxl.RXL_ERR_INVALID_ARGUMENT), ("mem_head", 8, rxl.RXL_ERR_INVALID_ARGUMENT),
    ("mem_cap", -1, rxl.RXL_ERR_INVALID_ARGUMENT), ("scale", float("nan"), rxl.RXL_ERR_INVALID_ARGUMENT),
])
def test_fwd_rejects_bad_descriptor(lib, field, value, status):
    d = rxl.make_desc(1, 1, 4, 8, 8, 0, 0.125, rxl.RXL_DTYPE_F32)
    setattr(d, field, value)
    assert fwd_status(lib, d) == status


def test_fwd_rejects_null_and_misaligned(lib):
    d = rxl.make_desc(1, 1, 4, 8, 8, 0, 0.125, rxl.RXL_DTYPE_F32)
    ptrs = [A] * 8
    ptrs[3] = None
    assert fwd_status(lib, d, ptrs) == rxl.RXL_ERR_INVALID_ARGUMENT
    ptrs[3] = A + 8
    assert fwd_status(lib, d, ptrs) == rxl.RXL_ERR_MISALIGNED
    assert lib.rxl_attn_fwd(None, *[A] * 8, None) == rxl.RXL_ERR_INVALID_ARGUMENT


def test_bwd_workspace_and_checks(lib):
    d = rxl.make_desc(2, 3, 5, 7, 4, 6, 0.125, rxl.RXL_DTYPE_BF16)
    ws = rxl.rxl_attn_bwd_workspace_bytes(d)
    assert ws > 0 and ws % 16 == 0
    bad = rxl.make_desc(2, 3, 5, 7, 8, 0, 0.125, rxl.RXL_DTYPE_BF16)
    assert rxl.rxl_attn_bwd_workspace_bytes(bad) == 0
    args = [ctypes.byref(d)] + [A] * 16
    assert lib.rxl_attn_bwd(*args, ws - 1, None) == rxl.RXL_ERR_WORKSPACE_TOO_SMALL


def test_mem_update_validation_and_noops(lib):
    ring = rxl.rxl_ring(A, 4, 8, 64, 8 * 64 + 64, rxl.RXL_DTYPE_BF16, 3, 5)
    # L == 0 and cap == 0 are valid no-ops that launch nothing and keep the state
    assert lib.rxl_mem_update(ctypes.byref(ring), A, 64, 0, None) == rxl.RXL_OK
    assert (ring.head, ring.len) == (3, 5)
    empty = rxl.rxl_ring(A, 4, 0, 64, 0, rxl.RXL_DTYPE_BF16, 0, 0)
    assert lib.rxl_mem_update(ctypes.byref(empty), A, 64 * 4, 4, None) == rxl.RXL_OK
    assert (empty.head, empty.len) == (0, 0)
    for field, value, status in [("head", 8, rxl.RXL_ERR_INVALID_ARGUMENT),
                                 ("len", 9, rxl.RXL_ERR_INVALID_ARGUMENT),
                                 ("D", 4, rxl.RXL_ERR_MISALIGNED),
                                 ("dtype", 3, rxl.RXL_ERR_UNSUPPORTED),
                                 ("plane_stride", 10, rxl.RXL_ERR_INVALID_ARGUMENT)]:
        r = rxl.rxl_ring(A, 4, 8, 64, 8 * 64 + 64, rxl.RXL_DTYPE_BF16, 3, 5)
        setattr(r, field, value)
        assert lib.rxl_mem_update(ctypes.byref(r), A, 64 * 4, 4, None) == status, field
        assert r.len == (value if field == "len" else 5)
    r = rxl.rxl_ring(A, 4, 8, 64, 8 * 64 + 64, rxl.RXL_DTYPE_BF16, 3, 5)
    assert lib.rxl_mem_update(ctypes.byref(r), A + 2, 64 * 4, 4, None) == rxl.RXL_ERR_MISALIGNED
    assert lib.rxl_mem_update(ctypes.byref(r), A, 64 * 4, -1, None) == rxl.RXL_ERR_INVALID_ARGUMENT
    assert (r.head, r.len) == (3, 5)


def test_mem_update_rings_rejects_mismatched_rings(lib):
    mk = lambda head=0, length=0, D=64, cap=8: rxl.rxl_ring(A, 2, cap, D, cap * D, rxl.RXL_DTYPE_BF16, head, length)
    P = ctypes.POINTER(rxl.rxl_ring)

    def call(rings, n=None):
        n = len(rings) if n is None else n
        arr = (P * max(n, 1))(*[ctypes.pointer(r) for r in rings])
        srcs = (ctypes.c_void_p * max(n, 1))(*([A] * max(n, 1)))
        strides = (ctypes.c_longlong * max(n, 1))(*([4 * 64] * max(n, 1)))
        return lib.rxl_mem_update_rings(arr, srcs, strides, n, 4, None)

    a = mk()
    assert call([a, mk(head=1)]) == rxl.RXL_ERR_INVALID_ARGUMENT      # other head
    assert call([a, mk(length=3)]) == rxl.RXL_ERR_INVALID_ARGUMENT    # other len
    assert call([a, mk(D=128)]) == rxl.RXL_ERR_INVALID_ARGUMENT       # other width
    assert call([a, a]) == rxl.RXL_ERR_INVALID_ARGUMENT               # the same ring twice
    assert call([], n=0) == rxl.RXL_ERR_INVALID_ARGUMENT
    assert call([mk() for _ in range(9)]) == rxl.RXL_ERR_INVALID_ARGUMENT
    assert (a.head, a.len) == (0, 0)                                  # nothing advanced


def test_kernel_timing_ids(lib):
    """Kernels 0-3 (forward, backward main, backward prep, backward finish)
    read back empty before anything was timed; other ids are refused with
    cudaErrorInvalidValue. No device call is made on these paths."""
    ms, n = ctypes.c_double(-1.0), ctypes.c_int(-1)
    for k in range(4):
        assert lib.rxl_kernel_timing_read(k, ctypes.byref(ms), ctypes.byref(n)) == 0
        assert (ms.value, n.value) == (0.0, 0)
    for k in (-1, 4):
        assert lib.rxl_kernel_timing_read(k, ctypes.byref(ms), ctypes.byref(n)) == 1
