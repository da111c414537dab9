"""The opt-in kernel timing hook (rxl_kernel_timing): with timing on, one
training pair (rxl_attn_fwd_ex + rxl_attn_bwd_ex) records one launch, with a
positive device time, of each timed kernel: the forward kernel, the
backward's preparation launch, its main kernel and its finish kernel; a read
clears them, and with timing off nothing is recorded."""
import pytest

from tests.test_gpu_attn import make_inputs, run_gpu

pytestmark = pytest.mark.gpu


def test_kernel_timing_covers_the_training_pair():
    import torch
    import long_context_lm_rel_gb300 as rxl
    ids = (rxl.RXL_KERNEL_FWD, rxl.RXL_KERNEL_BWD_MAIN, rxl.RXL_KERNEL_BWD_PREP, rxl.RXL_KERNEL_BWD_FINISH)
    B, H, L, cap, m = 2, 4, 256, 256, 200
    x = make_inputs(B, H, L, cap, m, "bf16", seed=11)
    c = run_gpu(x, cap, m, 37, "bf16", ex=True)  # builds the call and runs it once untimed
    torch.cuda.synchronize()
    for k in ids:
        rxl.rxl_kernel_timing_read(k)
    try:
        rxl.rxl_kernel_timing(True)
        c.fwd_ex().bwd_ex()
        torch.cuda.synchronize()
    finally:
        rxl.rxl_kernel_timing(False)
    for k in ids:
        ms, n = rxl.rxl_kernel_timing_read(k)
        assert n == 1 and ms > 0.0, (k, ms, n)
        assert rxl.rxl_kernel_timing_read(k) == (0.0, 0)
    c.fwd_ex().bwd_ex()  # timing off: nothing recorded
    torch.cuda.synchronize()
    for k in ids:
        assert rxl.rxl_kernel_timing_read(k) == (0.0, 0)


def test_kernel_timing_skips_graph_capture():
    import torch
    import long_context_lm_rel_gb300 as rxl
    ids = (rxl.RXL_KERNEL_FWD, rxl.RXL_KERNEL_BWD_MAIN, rxl.RXL_KERNEL_BWD_PREP, rxl.RXL_KERNEL_BWD_FINISH)
    B, H, L, cap, m = 2, 4, 128, 128, 128
    x = make_inputs(B, H, L, cap, m, "bf16", seed=12)
    c = run_gpu(x, cap, m, 0, "bf16", ex=True)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    try:
        rxl.rxl_kernel_timing(True)
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph, stream=side):
                c.fwd_ex().bwd_ex()
        torch.cuda.current_stream().wait_stream(side)
        graph.replay()
        torch.cuda.synchronize()
    finally:
        rxl.rxl_kernel_timing(False)
    for k in ids:
        assert rxl.rxl_kernel_timing_read(k) == (0.0, 0)
