"""Python binding of librxl (include/rxl.h): argument marshalling only.

Every function has the name and the argument order of its C entry point.
Tensors may be torch tensors (their data_ptr() is passed) or raw integer
device addresses. Each call raises RxlError on a non-OK status. The library
must have been built (``build()``); nothing here computes anything, and
there is no fallback when the library is missing.
"""
from __future__ import annotations

import ctypes
import os
import threading

from .build import LIB, build  # noqa: F401

RXL_OK = 0
RXL_ERR_INVALID_ARGUMENT = 1
RXL_ERR_UNSUPPORTED = 2
RXL_ERR_MISALIGNED = 3
RXL_ERR_WORKSPACE_TOO_SMALL = 4
RXL_ERR_CUDA = 5
RXL_DTYPE_F32 = 0
RXL_DTYPE_BF16 = 1


class rxl_attn_desc(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("L", ctypes.c_int), ("dh", ctypes.c_int),
                ("mem_cap", ctypes.c_int), ("mem_len", ctypes.c_int), ("mem_head", ctypes.c_int),
                ("scale", ctypes.c_float), ("dtype", ctypes.c_int)]


class rxl_ring(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("planes", ctypes.c_int), ("cap", ctypes.c_int),
                ("D", ctypes.c_int), ("plane_stride", ctypes.c_longlong), ("dtype", ctypes.c_int),
                ("head", ctypes.c_int), ("len", ctypes.c_int)]


class rxl_layer_weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "w_q", "w_k", "w_v", "w_o", "r", "u", "vbias", "ln1_gamma", "ln1_beta",
        "w_1", "b_1", "w_2", "b_2", "ln2_gamma", "ln2_beta")]


def make_layer_weights(**tensors) -> rxl_layer_weights:
    """rxl_layer_weights from tensors (or addresses) named as its fields."""
    return rxl_layer_weights(**{k: _ptr(v) for k, v in tensors.items()})


class RxlError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {rxl_status_string(status)}"
                         + (f" (cuda error {lib().rxl_last_cuda_error()})" if status == RXL_ERR_CUDA else ""))


_lib = None
_lock = threading.Lock()


def lib():
    """The loaded librxl (ctypes). Raises if the library was not built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB):
                raise RuntimeError(f"librxl.so is not built ({LIB}); call long_context_lm_rel_gb300.build()")
            L = ctypes.CDLL(LIB)
            P, vp = ctypes.POINTER, ctypes.c_void_p
            L.rxl_attn_fwd.argtypes = [P(rxl_attn_desc)] + [vp] * 8 + [vp]
            L.rxl_attn_fwd.restype = ctypes.c_int
            L.rxl_attn_bwd_workspace_bytes.argtypes = [P(rxl_attn_desc)]
            L.rxl_attn_bwd_workspace_bytes.restype = ctypes.c_size_t
            L.rxl_attn_bwd.argtypes = [P(rxl_attn_desc)] + [vp] * 16 + [ctypes.c_size_t, vp]
            L.rxl_attn_bwd.restype = ctypes.c_int
            L.rxl_mem_update.argtypes = [P(rxl_ring), vp, ctypes.c_longlong, ctypes.c_int, vp]
            L.rxl_mem_update.restype = ctypes.c_int
            L.rxl_mem_update_rings.argtypes = [P(P(rxl_ring)), P(vp), P(ctypes.c_longlong), ctypes.c_int,
                                               ctypes.c_int, vp]
            L.rxl_mem_update_rings.restype = ctypes.c_int
            L.rxl_status_string.argtypes = [ctypes.c_int]
            L.rxl_status_string.restype = ctypes.c_char_p
            L.rxl_last_cuda_error.argtypes = []
            L.rxl_last_cuda_error.restype = ctypes.c_int
            L.rxl_last_launch_count.argtypes = []
            L.rxl_last_launch_count.restype = ctypes.c_int
            L.rxl_device_error_flags.argtypes = []
            L.rxl_device_error_flags.restype = ctypes.c_int
            L.rxl_attn_fwd_ex.argtypes = [P(rxl_attn_desc)] + [vp] * 9 + [vp]
            L.rxl_attn_fwd_ex.restype = ctypes.c_int
            L.rxl_attn_bwd_ex.argtypes = [P(rxl_attn_desc)] + [vp] * 17 + [ctypes.c_size_t, vp]
            L.rxl_attn_bwd_ex.restype = ctypes.c_int
            L.rxl_attn_fwd_reset.argtypes = [P(rxl_attn_desc)] + [vp] * 10 + [vp]
            L.rxl_attn_fwd_reset.restype = ctypes.c_int
            L.rxl_attn_bwd_reset.argtypes = [P(rxl_attn_desc)] + [vp] * 18 + [ctypes.c_size_t, vp]
            L.rxl_attn_bwd_reset.restype = ctypes.c_int
            L.rxl_qkv_proj.argtypes = [P(rxl_attn_desc), ctypes.c_int] + [vp] * 8 + [vp]
            L.rxl_qkv_proj.restype = ctypes.c_int
            L.rxl_layer_fwd_workspace_bytes.argtypes = [P(rxl_attn_desc), ctypes.c_int, ctypes.c_int]
            L.rxl_layer_fwd_workspace_bytes.restype = ctypes.c_size_t
            L.rxl_layer_fwd.argtypes = [P(rxl_attn_desc), ctypes.c_int, ctypes.c_int, P(rxl_layer_weights)] \
                + [vp] * 4 + [ctypes.c_size_t, vp]
            L.rxl_layer_fwd.restype = ctypes.c_int
            L.rxl_kernel_timing.argtypes = [ctypes.c_int]
            L.rxl_kernel_timing.restype = ctypes.c_int
            L.rxl_kernel_timing_read.argtypes = [ctypes.c_int, P(ctypes.c_double), P(ctypes.c_int)]
            L.rxl_kernel_timing_read.restype = ctypes.c_int
            L.rxl_test_fail_next_launch.argtypes = [ctypes.c_int]
            L.rxl_test_fail_next_launch.restype = None
            L.rxl_test_forward_wait_timeout.argtypes = [ctypes.c_longlong, ctypes.c_int]
            L.rxl_test_forward_wait_timeout.restype = ctypes.c_int
            L.rxl_attn_bwd_noalloc.argtypes = [P(rxl_attn_desc)] + [vp] * 15 + [vp]
            L.rxl_attn_bwd_noalloc.restype = ctypes.c_int
            L.rxl_attn_bwd_noalloc_max_scratch_bytes.argtypes = []
            L.rxl_attn_bwd_noalloc_max_scratch_bytes.restype = ctypes.c_size_t
            _lib = L
    return _lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, where: str):
    if status != RXL_OK:
        raise RxlError(status, where)


def make_desc(B, H, L, mem_cap, mem_len, mem_head=0, scale=0.125, dtype=RXL_DTYPE_BF16, dh=64):
    return rxl_attn_desc(B, H, L, dh, mem_cap, mem_len, mem_head, scale, dtype)


def rxl_attn_fwd(desc, q, k, v, r, u, vbias, o, lse, stream=None):
    _check(lib().rxl_attn_fwd(ctypes.byref(desc), *map(_ptr, (q, k, v, r, u, vbias, o, lse)),
                              _stream(stream)), "rxl_attn_fwd")


def rxl_attn_fwd_ex(desc, q, k, v, r, u, vbias, o, o_lo, lse, stream=None):
    _check(lib().rxl_attn_fwd_ex(ctypes.byref(desc), *map(_ptr, (q, k, v, r, u, vbias, o, o_lo, lse)),
                                 _stream(stream)), "rxl_attn_fwd_ex")


def rxl_attn_bwd_ex(desc, q, k, v, r, u, vbias, o, o_lo, lse, dout, dq, dk, dv, dr, du, dvbias,
                    workspace, workspace_bytes, stream=None):
    _check(lib().rxl_attn_bwd_ex(ctypes.byref(desc),
                                 *map(_ptr, (q, k, v, r, u, vbias, o, o_lo, lse, dout, dq, dk, dv, dr,
                                             du, dvbias, workspace)),
                                 int(workspace_bytes), _stream(stream)), "rxl_attn_bwd_ex")


def rxl_attn_fwd_reset(desc, mem_visible, q, k, v, r, u, vbias, o, o_lo, lse, stream=None):
    _check(lib().rxl_attn_fwd_reset(ctypes.byref(desc),
                                    *map(_ptr, (mem_visible, q, k, v, r, u, vbias, o, o_lo, lse)),
                                    _stream(stream)), "rxl_attn_fwd_reset")


def rxl_attn_bwd_reset(desc, mem_visible, q, k, v, r, u, vbias, o, o_lo, lse, dout, dq, dk, dv, dr,
                       du, dvbias, workspace, workspace_bytes, stream=None):
    _check(lib().rxl_attn_bwd_reset(ctypes.byref(desc),
                                    *map(_ptr, (mem_visible, q, k, v, r, u, vbias, o, o_lo, lse, dout,
                                                dq, dk, dv, dr, du, dvbias, workspace)),
                                    int(workspace_bytes), _stream(stream)), "rxl_attn_bwd_reset")


def rxl_qkv_proj(desc, d_model, h_mem, h_cur, w_q, w_k, w_v, q, k, v, stream=None):
    _check(lib().rxl_qkv_proj(ctypes.byref(desc), int(d_model),
                              *map(_ptr, (h_mem, h_cur, w_q, w_k, w_v, q, k, v)), _stream(stream)),
           "rxl_qkv_proj")


def rxl_layer_fwd_workspace_bytes(desc, d_model, d_ff) -> int:
    return int(lib().rxl_layer_fwd_workspace_bytes(ctypes.byref(desc), int(d_model), int(d_ff)))


def rxl_layer_fwd(desc, d_model, d_ff, weights, h_mem, h_in, h_out, workspace, workspace_bytes,
                  stream=None):
    _check(lib().rxl_layer_fwd(ctypes.byref(desc), int(d_model), int(d_ff), ctypes.byref(weights),
                               *map(_ptr, (h_mem, h_in, h_out, workspace)), int(workspace_bytes),
                               _stream(stream)), "rxl_layer_fwd")


def rxl_attn_bwd_workspace_bytes(desc) -> int:
    return int(lib().rxl_attn_bwd_workspace_bytes(ctypes.byref(desc)))


def rxl_attn_bwd(desc, q, k, v, r, u, vbias, o, lse, dout, dq, dk, dv, dr, du, dvbias,
                 workspace, workspace_bytes, stream=None):
    _check(lib().rxl_attn_bwd(ctypes.byref(desc),
                              *map(_ptr, (q, k, v, r, u, vbias, o, lse, dout, dq, dk, dv, dr, du,
                                          dvbias, workspace)),
                              int(workspace_bytes), _stream(stream)), "rxl_attn_bwd")


def rxl_attn_bwd_noalloc(desc, q, k, v, r, u, vbias, o, lse, dout, dq, dk, dv, dr, du, dvbias,
                         stream=None):
    """rxl_attn_bwd for callers that cannot allocate: the scratch is a fixed
    array inside the library (see include/rxl.h for its size and rules)."""
    _check(lib().rxl_attn_bwd_noalloc(ctypes.byref(desc),
                                      *map(_ptr, (q, k, v, r, u, vbias, o, lse, dout, dq, dk, dv,
                                                  dr, du, dvbias)),
                                      _stream(stream)), "rxl_attn_bwd_noalloc")


def rxl_attn_bwd_noalloc_max_scratch_bytes() -> int:
    return int(lib().rxl_attn_bwd_noalloc_max_scratch_bytes())


def rxl_mem_update(ring: rxl_ring, src, src_plane_stride: int, L: int, stream=None):
    _check(lib().rxl_mem_update(ctypes.byref(ring), _ptr(src), int(src_plane_stride), int(L),
                                _stream(stream)), "rxl_mem_update")


def rxl_mem_update_rings(rings, srcs, src_plane_strides, L: int, stream=None):
    """rxl_mem_update of several rings of one geometry in one launch; the
    rxl_ring structs in `rings` are advanced in place."""
    n = len(rings)
    ring_ptrs = (ctypes.POINTER(rxl_ring) * n)(*[ctypes.pointer(r) for r in rings])
    src_arr = (ctypes.c_void_p * n)(*[_ptr(x) for x in srcs])
    str_arr = (ctypes.c_longlong * n)(*[int(x) for x in src_plane_strides])
    _check(lib().rxl_mem_update_rings(ring_ptrs, src_arr, str_arr, n, int(L), _stream(stream)),
           "rxl_mem_update_rings")


RXL_KERNEL_FWD, RXL_KERNEL_BWD_MAIN, RXL_KERNEL_BWD_PREP, RXL_KERNEL_BWD_FINISH = 0, 1, 2, 3


def rxl_kernel_timing(enable: bool):
    rc = lib().rxl_kernel_timing(1 if enable else 0)
    if rc:
        raise RuntimeError(f"rxl_kernel_timing: cuda error {rc}")


def rxl_kernel_timing_read(kernel: int):
    """(summed device ms, timed launches) of kernel since the last read."""
    ms, n = ctypes.c_double(0.0), ctypes.c_int(0)
    rc = lib().rxl_kernel_timing_read(int(kernel), ctypes.byref(ms), ctypes.byref(n))
    if rc:
        raise RuntimeError(f"rxl_kernel_timing_read: cuda error {rc}")
    return ms.value, n.value


def rxl_status_string(status: int) -> str:
    return lib().rxl_status_string(int(status)).decode()


def rxl_last_launch_count() -> int:
    return int(lib().rxl_last_launch_count())


def rxl_device_error_flags() -> int:
    return int(lib().rxl_device_error_flags())
