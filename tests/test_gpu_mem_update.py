"""rxl_mem_update is bit-exact against the oracle's Tail_M on the ring's
logical contents, for every fill/overflow pattern (eq. Tail_M, update_mems)."""
import numpy as np
import pytest

import oracle
from tests._harness import ring_rows

pytestmark = pytest.mark.gpu


def _bits(rng, shape, dtype):
    if dtype == "bf16":
        return rng.integers(0, 1 << 16, size=shape, dtype=np.uint16)
    return rng.integers(0, 1 << 32, size=shape, dtype=np.uint32)


def _dev(bits):
    import torch
    t = torch.from_numpy(bits.view(np.int16 if bits.dtype == np.uint16 else np.int32).copy())
    return t.cuda()


def _host(t, dtype):
    a = t.cpu().numpy()
    return a.view(np.uint16 if dtype == "bf16" else np.uint32)


CASES = [  # (cap, L, steps, head0)
    (8, 4, 5, 0), (5, 2, 7, 3), (4, 4, 3, 1), (3, 7, 3, 2), (1600, 128, 16, 0),
    (1600, 128, 15, 1536), (6, 1, 9, 5), (0, 3, 2, 0), (128, 128, 4, 0), (512, 512, 3, 100)]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("cap,L,steps,head0", CASES)
def test_ring_update_bit_exact(dtype, cap, L, steps, head0):
    import torch
    import long_context_lm_rel_gb300 as rxl
    rng = np.random.default_rng(cap * 131 + L * 7 + steps)
    planes, D = 6, 64
    buf = _bits(rng, (planes, cap + L, D), dtype)            # ring rows, then source rows
    dev = _dev(buf)
    dt = rxl.RXL_DTYPE_BF16 if dtype == "bf16" else rxl.RXL_DTYPE_F32
    ring = rxl.rxl_ring(dev.data_ptr(), planes, cap, D, (cap + L) * D, dt, head0 if cap else 0, 0)
    mem = np.zeros((planes, 0, D), dtype=buf.dtype)
    for step in range(steps):
        new = _bits(rng, (planes, L, D), dtype)
        dev[:, cap:] = _dev(new)
        before = _host(dev, dtype)
        elem = dev.element_size()
        rxl.rxl_mem_update(ring, dev.data_ptr() + cap * D * elem, (cap + L) * D, L)
        torch.cuda.synchronize()
        mem = oracle.tail_m(mem, new, cap)
        after = _host(dev, dtype)
        assert ring.len == mem.shape[1]
        got = after[:, ring_rows(cap, ring.head, ring.len)] if cap else after[:, :0]
        assert np.array_equal(got, mem), f"step {step}"
        # nothing outside the written rows moved; the source rows are untouched
        written = np.zeros(cap + L, dtype=bool)
        nw = min(L, cap)
        if cap:
            written[ring_rows(cap, (ring.head + ring.len - nw) % cap, nw)] = True
        assert np.array_equal(after[:, ~written], before[:, ~written])
        assert rxl.rxl_last_launch_count() == (1 if cap and L else 0)


def test_ring_checkpoint_restore_continues_identically():
    import torch
    import long_context_lm_rel_gb300 as rxl
    rng = np.random.default_rng(5)
    planes, cap, L, D = 4, 1600, 128, 64
    a = _dev(_bits(rng, (planes, cap + L, D), "bf16"))
    ring_a = rxl.rxl_ring(a.data_ptr(), planes, cap, D, (cap + L) * D, rxl.RXL_DTYPE_BF16, 0, 0)
    stream = [_bits(rng, (planes, L, D), "bf16") for _ in range(20)]
    for x in stream[:11]:
        a[:, cap:] = _dev(x)
        rxl.rxl_mem_update(ring_a, a.data_ptr() + cap * D * 2, (cap + L) * D, L)
    # checkpoint: the ring bytes plus (head, len) are the whole state
    b = a.clone()
    ring_b = rxl.rxl_ring(b.data_ptr(), planes, cap, D, (cap + L) * D, rxl.RXL_DTYPE_BF16,
                          ring_a.head, ring_a.len)
    for x in stream[11:]:
        for t, rg in ((a, ring_a), (b, ring_b)):
            t[:, cap:] = _dev(x)
            rxl.rxl_mem_update(rg, t.data_ptr() + cap * D * 2, (cap + L) * D, L)
    torch.cuda.synchronize()
    assert (ring_a.head, ring_a.len) == (ring_b.head, ring_b.len)
    assert torch.equal(a, b)
