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


@pytest.mark.parametrize("cap,L,steps,head0", [(1600, 128, 15, 1536), (5, 2, 7, 3), (3, 7, 3, 2), (512, 512, 3, 100)])
def test_rings_updated_together_bit_exact(cap, L, steps, head0):
    """rxl_mem_update_rings advances K and V rings of one geometry (different
    buffers and source strides) in one launch, each bit-exact to Tail_M."""
    import torch
    import long_context_lm_rel_gb300 as rxl
    rng = np.random.default_rng(cap + 17 * L)
    planes, D = 5, 64
    k = _dev(_bits(rng, (planes, cap + L, D), "bf16"))
    v_ring = _dev(_bits(rng, (planes, cap, D), "bf16"))      # a ring without current rows
    v_src = _dev(_bits(rng, (planes, L + 3, D), "bf16"))     # a source with another plane stride
    rk = rxl.rxl_ring(k.data_ptr(), planes, cap, D, (cap + L) * D, rxl.RXL_DTYPE_BF16, head0, 0)
    rv = rxl.rxl_ring(v_ring.data_ptr(), planes, cap, D, cap * D, rxl.RXL_DTYPE_BF16, head0, 0)
    mk = np.zeros((planes, 0, D), np.uint16)
    mv = mk.copy()
    for step in range(steps):
        nk, nv = _bits(rng, (planes, L, D), "bf16"), _bits(rng, (planes, L, D), "bf16")
        k[:, cap:] = _dev(nk)
        v_src[:, :L] = _dev(nv)
        rxl.rxl_mem_update_rings([rk, rv], [k.data_ptr() + cap * D * 2, v_src], [(cap + L) * D, (L + 3) * D], L)
        assert rxl.rxl_last_launch_count() == 1
        torch.cuda.synchronize()
        mk, mv = oracle.tail_m(mk, nk, cap), oracle.tail_m(mv, nv, cap)
        assert (rk.head, rk.len) == (rv.head, rv.len) and rk.len == mk.shape[1]
        assert np.array_equal(_host(k, "bf16")[:, ring_rows(cap, rk.head, rk.len)], mk), f"K step {step}"
        assert np.array_equal(_host(v_ring, "bf16")[:, ring_rows(cap, rv.head, rv.len)], mv), f"V step {step}"


def test_wide_plane_wrapping_copy():
    """One wide plane (D = 8192 bf16 elements, 16 KB rows; 4096 rows appended
    to a full ring of 8192 at head 6000): the copy of 4 M vectors crosses the
    ring's wrap inside one plane and lands row for row."""
    import torch
    import long_context_lm_rel_gb300 as rxl
    planes, cap, L, D = 1, 8192, 4096, 8192
    head0 = 6000
    k = torch.zeros((planes, cap + L, D), device="cuda", dtype=torch.int16)
    src = torch.arange(L, device="cuda", dtype=torch.int16).view(1, L, 1).expand(planes, L, D).contiguous()
    k[:, cap:] = src
    ring = rxl.rxl_ring(k.data_ptr(), planes, cap, D, (cap + L) * D, rxl.RXL_DTYPE_BF16, head0, cap)
    rxl.rxl_mem_update(ring, k.data_ptr() + cap * D * 2, (cap + L) * D, L)
    torch.cuda.synchronize()
    assert (ring.head, ring.len) == ((head0 + L) % cap, cap)
    dst = (head0 + np.arange(L)) % cap                # where the appended rows went
    got = k[0, torch.from_numpy(dst).cuda(), :].cpu().numpy()
    assert np.array_equal(got, np.broadcast_to(np.arange(L, dtype=np.int16)[:, None], (L, D)))
