"""The allocation-free backward entry point.

rxl_attn_bwd_noalloc serves callers that cannot allocate device memory when
they run the backward (hosts that hand over only their inputs and outputs,
or loops that must not pay for a cudaMalloc); its scratch is a fixed array
inside the library. Through the C ABI it must give what rxl_attn_bwd with a
caller workspace gives, call after call, and refuse shapes that do not fit.
This file is collected last so that a failure here cannot hide others.
"""
import ctypes

import numpy as np
import pytest

from tests._harness import AttnCall, assert_close, assert_no_device_error, place_kv, to_host
from tests.test_gpu_attn import make_inputs

pytestmark = pytest.mark.gpu

OUTS = ("dq", "dk", "dv", "dr", "du", "dvb")


def _noalloc_outputs(c):
    import torch
    import long_context_lm_rel_gb300 as rxl
    out = {n: torch.full_like(getattr(c, n), float("nan")) for n in OUTS}
    rxl.rxl_attn_bwd_noalloc(c.desc, c.q, c.k, c.v, c.r, c.u, c.vb, c.o, c.lse, c.do,
                             out["dq"], out["dk"], out["dv"], out["dr"], out["du"], out["dvb"])
    torch.cuda.synchronize()
    return {n: to_host(t) for n, t in out.items()}


@pytest.mark.parametrize("dtype,shape", [("bf16", (2, 4, 200, 300, 250, 7)),
                                         ("f32", (1, 2, 70, 90, 60, 50))])
def test_noalloc_backward_matches_workspace_backward(dtype, shape):
    import torch
    B, H, L, cap, m, head = shape
    x = make_inputs(B, H, L, cap, m, dtype, seed=4242, D_model=256)
    c = AttnCall(x["q"], place_kv(x["k_mem"], x["k_cur"], cap, head), place_kv(x["v_mem"], x["v_cur"], cap, head),
                 x["r"], x["u"], x["vb"], cap=cap, m=m, head=head, dtype=dtype, scale=0.125)
    c.fwd().alloc_bwd(x["do"]).bwd()
    torch.cuda.synchronize()
    ref = {n: to_host(getattr(c, n)) for n in OUTS}
    for call in range(2):  # the shared scratch keeps the previous call's contents
        got = _noalloc_outputs(c)
        for n in OUTS:
            assert_close(n, got[n], ref[n], dtype, f"noalloc call {call}")
    assert_no_device_error()


def test_noalloc_rejects_shapes_beyond_its_scratch():
    import long_context_lm_rel_gb300 as rxl
    lib = rxl.lib()
    limit = rxl.rxl_attn_bwd_noalloc_max_scratch_bytes()
    big = rxl.make_desc(16, 16, 512, 512, 512, 0, 0.125, rxl.RXL_DTYPE_BF16)
    assert rxl.rxl_attn_bwd_workspace_bytes(big) > limit
    a = 1 << 20  # never dereferenced: the call must refuse before launching
    st = lib.rxl_attn_bwd_noalloc(ctypes.byref(big), *([a] * 15), None)
    assert st == rxl.RXL_ERR_WORKSPACE_TOO_SMALL


def test_noalloc_shape_whose_scratch_ends_at_the_limit():
    """B4 H16 L128 with a full 1780-row memory: the workspace ends within
    300 KB of the fixed array's end, so the fp32 dR accumulator and its TMA
    descriptor sit at the end of the array. Every output matches the
    workspace backward."""
    import torch
    B, H, L, cap, m, head = 4, 16, 128, 1780, 1780, 1700
    limit = __import__("long_context_lm_rel_gb300").rxl_attn_bwd_noalloc_max_scratch_bytes()
    x = make_inputs(B, H, L, cap, m, "bf16", seed=99)
    c = AttnCall(x["q"], place_kv(x["k_mem"], x["k_cur"], cap, head), place_kv(x["v_mem"], x["v_cur"], cap, head),
                 x["r"], x["u"], x["vb"], cap=cap, m=m, head=head, dtype="bf16", scale=0.125)
    c.fwd().alloc_bwd(x["do"])
    assert limit - (300 << 10) < c.ws_bytes <= limit, (c.ws_bytes, limit)
    c.bwd()
    torch.cuda.synchronize()
    ref = {n: to_host(getattr(c, n)) for n in OUTS}
    got = _noalloc_outputs(c)
    for n in OUTS:
        assert_close(n, got[n], ref[n], "bf16", "near the scratch limit")
    assert_no_device_error()
