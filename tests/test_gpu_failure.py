"""Failure detection without a GPU fault.

* A launch that fails (made to fail on the host by a testing hook, before
  anything reaches the GPU) comes back as RXL_ERR_CUDA with the CUDA error
  code, and nothing is written.
* A bounded device wait that runs out: the forward kernel's wait limit is
  shortened to about a millisecond and one barrier arrival (no copy or MMA is
  pending on it) is withheld; the kernel must drain its copies, free its
  tensor memory, exit, and report through rxl_device_error_flags(), and the
  context must stay usable: the next call is correct.
No test here traps, faults or waits without a limit.
"""
import numpy as np
import pytest

import oracle
from tests._harness import assert_close, assert_no_device_error, to_host
from tests.test_gpu_attn import logical, make_inputs, run_gpu

pytestmark = pytest.mark.gpu

CUDA_ERROR_INVALID_CONFIGURATION = 9  # cudaErrorInvalidConfiguration


def test_failed_launch_returns_cuda_status_and_writes_nothing():
    import torch
    import long_context_lm_rel_gb300 as rxl
    lib = rxl.lib()
    B, H, L, cap, m = 2, 2, 100, 120, 90
    x = make_inputs(B, H, L, cap, m, "bf16", seed=5)
    c = run_gpu(x, cap, m, 7, "bf16", bwd=False)
    c.alloc_bwd(x["do"])
    torch.cuda.synchronize()
    c.o.fill_(float("nan"))
    c.dq.fill_(float("nan"))
    lib.rxl_test_fail_next_launch(CUDA_ERROR_INVALID_CONFIGURATION)
    with pytest.raises(rxl.RxlError) as e:
        c.fwd()
    assert e.value.status == rxl.RXL_ERR_CUDA
    assert lib.rxl_last_cuda_error() == CUDA_ERROR_INVALID_CONFIGURATION
    torch.cuda.synchronize()
    assert torch.isnan(c.o).all(), "a failed call wrote its output"
    # the backward's first launch fails: nothing after it is launched either
    lib.rxl_test_fail_next_launch(CUDA_ERROR_INVALID_CONFIGURATION)
    with pytest.raises(rxl.RxlError) as e:
        c.bwd()
    assert e.value.status == rxl.RXL_ERR_CUDA
    torch.cuda.synchronize()
    assert torch.isnan(c.dq).all(), "a failed call wrote its output"
    # the hook is one-shot: the same calls now succeed and are correct
    c.fwd().bwd()
    torch.cuda.synchronize()
    assert_no_device_error()
    k, v = logical(x)
    o_ref, _ = oracle.fwd(x["q"], k, v, x["r"], x["u"], x["vb"], 0.125)
    assert_close("O", to_host(c.o), o_ref, "bf16")
    g = oracle.bwd(x["q"], k, v, x["r"], x["u"], x["vb"], x["do"], 0.125)
    assert_close("dQ", to_host(c.dq), g["dq"], "bf16")


def test_forward_wait_that_runs_out_is_reported_and_the_context_survives():
    import torch
    import long_context_lm_rel_gb300 as rxl
    lib = rxl.lib()
    # 2 x 64 heads x 2 query tiles = 256 items: the persistent (non-cluster) forward
    B, H, L, cap, m = 2, 64, 256, 128, 128
    x = make_inputs(B, H, L, cap, m, "bf16", seed=6, D_model=4096)
    assert lib.rxl_device_error_flags() == 0
    try:
        assert lib.rxl_test_forward_wait_timeout(2_000_000, 1) == 0   # ~1 ms at 2 GHz
        c = run_gpu(x, cap, m, 0, "bf16", bwd=False)
        torch.cuda.synchronize()
        flags = lib.rxl_device_error_flags()
    finally:
        assert lib.rxl_test_forward_wait_timeout(0, 0) == 0
    assert flags == 1, f"expected the forward's timeout bit, got {flags}"
    # the context is intact: the same call now completes and is correct
    c.fwd()
    torch.cuda.synchronize()
    assert lib.rxl_device_error_flags() == 0
    k, v = logical(x)
    o_ref, lse_ref = oracle.fwd(x["q"], k, v, x["r"], x["u"], x["vb"], 0.125)
    assert_close("O", to_host(c.o), o_ref, "bf16")
    assert_close("LSE", to_host(c.lse), lse_ref, "bf16")


@pytest.mark.parametrize("where", ["r", "vbias"])
def test_fp16_range_of_the_position_products_is_reported(where):
    """The backward's position products take r and q + vbias in fp16: an
    element beyond 65504 in magnitude is clamped and reported (bit 4 of
    rxl_device_error_flags), never silently."""
    import torch
    import long_context_lm_rel_gb300 as rxl
    lib = rxl.lib()
    B, H, L, cap, m = 1, 2, 64, 64, 32
    x = make_inputs(B, H, L, cap, m, "bf16", seed=8)
    c = run_gpu(x, cap, m, 0, "bf16")
    torch.cuda.synchronize()
    assert lib.rxl_device_error_flags() == 0          # in range: nothing reported
    if where == "r":
        c.r[1, 5, 3] = 1.0e5                          # a distance row the call reads
    else:
        c.vb[0, 7] = -7.0e4
    c.alloc_bwd(x["do"]).bwd()
    torch.cuda.synchronize()
    assert lib.rxl_device_error_flags() == 16
