"""Projection front-end on the GPU against the oracle ("Segment-Level
Recurrence": Q = H W^Q, K/V = [SG(M); H] W^{K,V}; the memory holds hidden
states in a ring). The projected K/V land in the attention's ring layout."""
import numpy as np
import pytest

import oracle
import rxl_inputs as gen
from tests._harness import (AttnCall, assert_close, assert_no_device_error, logical_kv, place_kv,
                            ring_rows, to_dev, to_host)

pytestmark = pytest.mark.gpu


def _inputs(B, H, L, m, d, seed):
    n = lambda i, shape, std: gen.round_to(gen.normal(seed, 700000 + i, shape, std), "bf16")
    return dict(h_mem=n(1, (B, m, d), 1.0), h_cur=n(2, (B, L, d), 1.0),
                wq=n(3, (d, H * 64), d ** -0.5), wk=n(4, (d, H * 64), d ** -0.5),
                wv=n(5, (d, H * 64), d ** -0.5))


def _ring(h_mem, cap, head, fill=3.0):
    B, m, d = h_mem.shape
    out = np.full((B, max(cap, 1), d), fill, dtype=np.float32)
    if m:
        out[:, ring_rows(cap, head, m)] = h_mem
    return out


def _project(x, B, H, L, cap, m, head, d):
    import torch
    import long_context_lm_rel_gb300 as rxl
    desc = rxl.make_desc(B, H, L, cap, m, head, 0.125, rxl.RXL_DTYPE_BF16)
    ring = to_dev(_ring(x["h_mem"], cap, head), "bf16")
    hc = to_dev(x["h_cur"], "bf16")
    w = [to_dev(x[n], "bf16") for n in ("wq", "wk", "wv")]
    sentinel = 11.0
    q = torch.full((B, H, L, 64), sentinel, device="cuda", dtype=torch.bfloat16)
    k = torch.full((B, H, cap + L, 64), sentinel, device="cuda", dtype=torch.bfloat16)
    v = torch.full_like(k, sentinel)
    rxl.rxl_qkv_proj(desc, d, ring if cap else None, hc, *w, q, k, v)
    torch.cuda.synchronize()
    assert_no_device_error()
    return to_host(q), to_host(k), to_host(v), sentinel


def assert_proj(name, got, ref, absmag, d, tag=""):
    """Bound from the arithmetic (O(1) outputs; the attention's 1e-3 mean rule
    is below the output's own bf16 rounding here): bf16 x bf16 products are
    exact in fp32, the fp32 sum of d of them errs by at most d * 2^-24 *
    sum |h_k||w_k| (absmag = that sum, from |h| @ |W| in float64), and the
    final rounding to bf16 by at most 2^-8 |x|."""
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    acc = d * 2.0 ** -24 * absmag
    bound = 2.0 ** -8 * (np.abs(ref) + acc) + acc + 1e-30
    excess = np.abs(got - ref) / bound
    assert excess.max() <= 1.0, f"{name}: error {excess.max():.2f} x the bound {tag}"


def _absmag(x, H):
    a = lambda n: np.abs(np.asarray(x[n], np.float64))
    return oracle.proj(a("h_mem"), a("h_cur"), a("wq"), a("wk"), a("wv"), H)


CASES = [  # B, H, L, cap, m, head, d
    (2, 6, 200, 300, 250, 123, 192),     # ragged row tiles, a wrapping ring, a 2-head column tile
    (1, 4, 129, 0, 0, 0, 64),            # no memory at all
    (2, 16, 64, 1600, 1600, 1550, 128),  # long ring wrapping mid-tile
    (3, 3, 1, 5, 5, 2, 64),              # one current row
    (2, 2, 130, 256, 100, 200, 256),     # ring not full: empty slots stay untouched
    (1, 5, 300, 130, 130, 60, 128),      # a 1-head column tile; odd row-tile lists (a CTA pair with one block)
]


@pytest.mark.parametrize("B,H,L,cap,m,head,d", CASES)
def test_projection_parity(B, H, L, cap, m, head, d):
    x = _inputs(B, H, L, m, d, seed=B + H + L + d)
    q, k, v, sentinel = _project(x, B, H, L, cap, m, head, d)
    qr, kr, vr = oracle.proj(x["h_mem"], x["h_cur"], x["wq"], x["wk"], x["wv"], H)
    qa, ka, va = _absmag(x, H)
    tag = str((B, H, L, cap, m, head, d))
    assert_proj("Q", q, qr, qa, d, tag)
    assert_proj("K", logical_kv(k, cap, head, m), kr, ka, d, tag)
    assert_proj("V", logical_kv(v, cap, head, m), vr, va, d, tag)
    empty = np.setdiff1d(np.arange(cap), ring_rows(cap, head, m)) if cap else []
    if len(empty):
        assert (k[:, :, empty] == sentinel).all() and (v[:, :, empty] == sentinel).all()


def test_projection_mid_size_full_width():
    B, H, L, cap, m, head, d = 2, 16, 512, 512, 512, 0, 1024
    x = _inputs(B, H, L, m, d, seed=3)
    q, k, v, _ = _project(x, B, H, L, cap, m, head, d)
    qr, kr, vr = oracle.proj(x["h_mem"], x["h_cur"], x["wq"], x["wk"], x["wv"], H)
    qa, ka, va = _absmag(x, H)
    assert_proj("Q", q, qr, qa, d)
    assert_proj("K", logical_kv(k, cap, head, m), kr, ka, d)
    assert_proj("V", logical_kv(v, cap, head, m), vr, va, d)


def test_projection_feeds_the_attention():
    """hidden states -> projection -> attention forward, against the oracle's
    projection followed by the oracle's attention."""
    import torch
    import long_context_lm_rel_gb300 as rxl
    B, H, L, cap, m, head, d = 2, 4, 150, 200, 180, 70, 128
    x = _inputs(B, H, L, m, d, seed=17)
    q, k, v, _ = _project(x, B, H, L, cap, m, head, d)
    r = gen.round_to(gen.rel_table(cap + L, 256, H, 64, 5, 900009), "bf16")
    u = gen.round_to(gen.normal(5, 900006, (H, 64), 0.02), "bf16")
    vb = gen.round_to(gen.normal(5, 900007, (H, 64), 0.02), "bf16")
    c = AttnCall(q, k, v, r, u, vb, cap=cap, m=m, head=head, dtype="bf16", scale=0.125).fwd()
    torch.cuda.synchronize()
    assert_no_device_error()
    qr, kr, vr = oracle.proj(x["h_mem"], x["h_cur"], x["wq"], x["wk"], x["wv"], H)
    # the attention's inputs are the bf16-rounded projections
    rb = lambda a: gen.round_to(a, "bf16")
    o_ref, lse_ref = oracle.fwd(rb(qr), rb(kr), rb(vr), r, u, vb, 0.125)
    assert_close("O", to_host(c.o), o_ref, "bf16")
    assert_close("LSE", to_host(c.lse), lse_ref, "bf16")
