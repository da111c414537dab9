"""Per-row document reset on the GPU against the oracle.

Batch row b attends only to its newest mem_visible[b] memory rows
(Transformer-XL page, "Causal Mask With Memory", the note after the mask
picture; "Batched Streams": the reset is per row). Full forward and backward
parity, including rows reset to 0, rows whose visible memory ends mid-tile,
rings that wrap, out-of-range counts (clamped into [0, m]), the fp32 path
and seeded random shapes and counts.
"""
import numpy as np
import pytest

import oracle
from tests._harness import AttnCall, assert_close, assert_no_device_error, logical_kv, place_kv, to_host
from tests.test_gpu_attn import _random_shapes, make_inputs, logical

pytestmark = pytest.mark.gpu

CASES = [  # B, H, L, cap, m, head, mem_visible
    (3, 2, 200, 300, 250, 123, [250, 0, 77]),      # full, reset, partial; the ring wraps
    (2, 2, 130, 256, 256, 200, [129, 1]),          # tile edges +-1, wrapping ring
    (2, 1, 64, 1600, 1600, 1550, [1600, 300]),     # long ring, the visible part crosses the wrap
    (2, 2, 1, 5, 5, 2, [3, 0]),                    # one query row
]


def _run(B, H, L, cap, m, head, mvis, dtype, keep_low, clamp_to=None, seed=None):
    import torch
    x = make_inputs(B, H, L, cap, m, dtype, seed=seed if seed is not None else B * 7 + L + m)
    c = AttnCall(x["q"], place_kv(x["k_mem"], x["k_cur"], cap, head, fill=7.0),
                 place_kv(x["v_mem"], x["v_cur"], cap, head, fill=-7.0), x["r"], x["u"], x["vb"],
                 cap=cap, m=m, head=head, dtype=dtype, scale=0.125)
    c.fwd_reset(mvis, keep_low=keep_low)
    c.alloc_bwd(x["do"])
    c.bwd_reset()
    torch.cuda.synchronize()
    assert_no_device_error()
    ref_mvis = clamp_to if clamp_to is not None else mvis
    k, v = logical(x)
    tag = str((B, H, L, cap, m, head, mvis, dtype, keep_low))
    o, lse = oracle.fwd(x["q"], k, v, x["r"], x["u"], x["vb"], 0.125, mem_visible=ref_mvis)
    assert_close("O", to_host(c.o), o, dtype, tag)
    assert_close("LSE", to_host(c.lse), lse, dtype, tag)
    g = oracle.bwd(x["q"], k, v, x["r"], x["u"], x["vb"], x["do"], 0.125, mem_visible=ref_mvis)
    assert_close("dQ", to_host(c.dq), g["dq"], dtype, tag)
    dk, dv = logical_kv(to_host(c.dk), cap, head, m), logical_kv(to_host(c.dv), cap, head, m)
    assert_close("dK", dk, g["dk"], dtype, tag)
    assert_close("dV", dv, g["dv"], dtype, tag)
    # masked memory rows get exactly zero
    for b, mb in enumerate(ref_mvis):
        assert not dk[b, :, :m - mb].any() and not dv[b, :, :m - mb].any(), tag
    assert_close("dR", to_host(c.dr)[:, :m + L], g["dr"], dtype, tag)
    assert_close("du", to_host(c.du), g["du"], dtype, tag)
    assert_close("dv", to_host(c.dvb), g["dvb"], dtype, tag)


@pytest.mark.parametrize("keep_low", [False, True], ids=["recompute_D", "training_pair"])
@pytest.mark.parametrize("B,H,L,cap,m,head,mvis", CASES)
def test_reset_bf16(B, H, L, cap, m, head, mvis, keep_low):
    _run(B, H, L, cap, m, head, mvis, "bf16", keep_low)


def _random_reset_cases(seed=31):
    """Seeded random shapes and mem_visible counts in [0, m] (partial tiles,
    resets, wrapping rings); a one-row segment keeps at least one memory row
    visible, so that no output is identically zero."""
    rng = np.random.default_rng(seed)
    out = []
    for B, H, L, cap, m, head in _random_shapes(8, 2, seed=seed):
        if m == 0:
            continue
        lo = 1 if L == 1 else 0
        out.append((B, H, L, cap, m, head, [int(rng.integers(lo, m + 1)) for _ in range(B)]))
    return out


@pytest.mark.parametrize("B,H,L,cap,m,head,mvis", _random_reset_cases())
def test_reset_random_shapes(B, H, L, cap, m, head, mvis):
    _run(B, H, L, cap, m, head, mvis, "bf16", keep_low=True)


def test_reset_f32():
    _run(2, 2, 40, 64, 50, 30, [50, 13], "f32", keep_low=False)


def test_reset_counts_are_clamped():
    _run(2, 2, 100, 128, 90, 17, [-5, 10 ** 6], "bf16", keep_low=True, clamp_to=[0, 90])


def test_reset_all_rows_full_equals_plain_call():
    import torch
    B, H, L, cap, m, head = 2, 2, 150, 200, 180, 60
    x = make_inputs(B, H, L, cap, m, "bf16", seed=99)
    mk = lambda: AttnCall(x["q"], place_kv(x["k_mem"], x["k_cur"], cap, head),
                          place_kv(x["v_mem"], x["v_cur"], cap, head), x["r"], x["u"], x["vb"],
                          cap=cap, m=m, head=head, dtype="bf16", scale=0.125)
    a = mk().fwd_ex()
    a.alloc_bwd(x["do"]).bwd_ex()
    b = mk().fwd_reset([m] * B)
    b.alloc_bwd(x["do"]).bwd_reset()
    torch.cuda.synchronize()
    # same tiles, same arithmetic: bitwise for everything that is not summed
    # by reductions in L2 (whose order varies from run to run)
    for n in ("o", "lse", "dk", "dv"):
        assert torch.equal(getattr(a, n), getattr(b, n)), n
    for n in ("dr", "du", "dvb"):
        x_, y_ = getattr(a, n), getattr(b, n)
        assert (x_ - y_).abs().max() <= 1e-5 * x_.abs().max(), n
    d = (a.dq.float() - b.dq.float()).abs().max()
    assert d <= 2.0 ** -7 * a.dq.float().abs().max(), d
