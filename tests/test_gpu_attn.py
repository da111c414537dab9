"""Parity of rxl_attn_fwd / rxl_attn_bwd (called through the C ABI) with the
float64 oracle on the same seeded inputs.

* every element at sizes the oracle finishes in seconds (several tiles,
  ragged tails, rotated and wrapping rings, empty memory);
* the five configurations of the path at full size, every element: cfg1,
  cfg2 (4-segment stream), cfg3/cfg4 (forward and backward, all (b, h)),
  cfg5 as the 32-segment stream of all 16 layers, every row at the fill,
  wrap and steady-state segments;
* skew-sensitive closed-form probes (distance labels) on tile boundaries;
* calls with at most half as many (b, h, query tile) items as SMs, which the
  forward runs as 2-CTA clusters (the small cases too, one of them with a
  single key tile per item, i.e. an empty second half);
* stop-gradient: the cache is never written by the backward;
* NaN in every backward output and junk in the workspace on entry;
* seeded random shapes (tile edges, partly filled and wrapping rings, few
  and many items).
"""
import math

import numpy as np
import pytest

import oracle
import rxl_inputs as gen
from tests._harness import AttnCall, assert_close, assert_no_device_error, logical_kv, place_kv, to_host

pytestmark = pytest.mark.gpu


def make_inputs(B, H, L, cap, m, dtype, seed=0, tid0=900000, D_model=1024):
    """Synthetic inputs with the distributions of the configurations:
    Q, K, V ~ N(0,1)/sqrt(dh), u, v ~ N(0, 0.02^2), R sinusoid x W_R, dO ~ N(0,1)."""
    dh, sd = 64, 0.125
    n = lambda i, shape, std: gen.round_to(gen.normal(seed, tid0 + i, shape, std), dtype)
    return dict(
        q=n(1, (B, H, L, dh), sd), k_mem=n(2, (B, H, m, dh), sd), k_cur=n(3, (B, H, L, dh), sd),
        v_mem=n(4, (B, H, m, dh), sd), v_cur=n(5, (B, H, L, dh), sd), u=n(6, (H, dh), 0.02),
        vb=n(7, (H, dh), 0.02), do=n(8, (B, H, L, dh), 1.0),
        r=gen.round_to(gen.rel_table(cap + L, D_model, H, dh, seed, tid0 + 9), dtype))


def run_gpu(x, cap, m, head, dtype, bwd=True, scale=0.125, ex=False, fill=(7.0, -7.0)):
    """ex=True runs the training pair (forward keeps the low part of O);
    `fill` is the junk written to the K and V ring rows that hold no memory."""
    k_phys = place_kv(x["k_mem"], x["k_cur"], cap, head, fill=fill[0])
    v_phys = place_kv(x["v_mem"], x["v_cur"], cap, head, fill=fill[1])
    c = AttnCall(x["q"], k_phys, v_phys, x["r"], x["u"], x["vb"], cap=cap, m=m, head=head,
                 dtype=dtype, scale=scale)
    c.fwd_ex() if ex else c.fwd()
    if bwd:
        c.alloc_bwd(x["do"])
        c.bwd_ex() if ex else c.bwd()
    return c


def logical(x):
    return (np.concatenate([x["k_mem"], x["k_cur"]], 2), np.concatenate([x["v_mem"], x["v_cur"]], 2))


def compare_full(x, c, cap, m, head, dtype, bwd=True, scale=0.125, tag=""):
    import torch
    torch.cuda.synchronize()
    assert_no_device_error()
    k, v = logical(x)
    o, lse = oracle.fwd(x["q"], k, v, x["r"], x["u"], x["vb"], scale)
    assert_close("O", to_host(c.o), o, dtype, tag)
    assert_close("LSE", to_host(c.lse), lse, dtype, tag)
    if not bwd:
        return
    g = oracle.bwd(x["q"], k, v, x["r"], x["u"], x["vb"], x["do"], scale)
    L = x["q"].shape[2]
    assert_close("dQ", to_host(c.dq), g["dq"], dtype, tag)
    dk, dv = to_host(c.dk), to_host(c.dv)
    assert_close("dK", logical_kv(dk, cap, head, m), g["dk"], dtype, tag)
    assert_close("dV", logical_kv(dv, cap, head, m), g["dv"], dtype, tag)
    unused = np.setdiff1d(np.arange(cap), (head + np.arange(m)) % cap if m else [])
    assert np.all(dk[:, :, unused] == 0) and np.all(dv[:, :, unused] == 0), "ring rows without memory"
    dr = to_host(c.dr)
    assert_close("dR", dr[:, :m + L], g["dr"], dtype, tag)
    assert np.all(dr[:, m + L:] == 0)
    assert_close("du", to_host(c.du), g["du"], dtype, tag)
    assert_close("dv", to_host(c.dvb), g["dvb"], dtype, tag)


# ---------------------------------------------------- small full-oracle cases

SMALL = [  # B, H, L, cap, m, head
    (2, 2, 200, 300, 250, 123),   # several tiles, ragged, rotated ring that wraps
    (1, 3, 129, 0, 0, 0),         # no memory at all: plain causal attention
    (2, 1, 64, 1600, 1600, 1550), # long full ring that wraps mid-tile
    (3, 2, 1, 5, 5, 2),           # one query row
    (1, 2, 130, 128, 127, 0),     # tile edges +-1
    (2, 2, 128, 256, 0, 0),       # memory capacity but still empty
]


@pytest.mark.parametrize("ex", [False, True], ids=["plain", "training_pair"])
@pytest.mark.parametrize("B,H,L,cap,m,head", SMALL)
def test_small_bf16_full_parity(B, H, L, cap, m, head, ex):
    x = make_inputs(B, H, L, cap, m, "bf16", seed=B * 1000 + L + m)
    c = run_gpu(x, cap, m, head, "bf16", ex=ex)
    compare_full(x, c, cap, m, head, "bf16", tag=str((B, H, L, cap, m, head, ex)))


def _random_shapes(n_small, n_wide, seed=2024):
    """Seeded random shapes: small ones (few items: the forward's 2-CTA
    clusters) and wide ones (many heads: the persistent forward), with
    query lengths near tile edges, partly filled and wrapping rings."""
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n_small + n_wide):
        wide = i >= n_small
        B = int(rng.integers(1, 4)) if not wide else int(rng.integers(2, 5))
        H = int(rng.integers(1, 4)) if not wide else int(rng.integers(12, 25))
        L = int(rng.choice([1, 63, 127, 128, 129, 200, 255, 256, 257, 300]))
        cap = int(rng.choice([0, 5, 127, 128, 200, 333, 400]))
        m = int(rng.integers(0, cap + 1)) if cap else 0
        head = int(rng.integers(0, cap)) if cap else 0
        if L == 1 and m == 0:
            continue  # one visible key per row: the degenerate case below
        out.append((B, H, L, cap, m, head))
    return out


@pytest.mark.parametrize("ex", [False, True], ids=["plain", "training_pair"])
def test_single_visible_key_gradients_vanish(ex):
    """L = 1 without memory: each row sees only its own key, so P = 1,
    O = v and D = dO.v = dP, and dA = scale P (dP - D) is identically zero
    (the chain rule of "Dimension Walkthrough"). dq, dk, dr, du and dvbias are
    then exactly zero, where a bound relative to max|ref| is zero too: the
    kernel's dP and D are two fp32 sums of the same products (tensor core and
    prep), so their difference leaves rounding residues, bounded here by
    2^-16 of |dO| |v| scale |k|. dv = dO."""
    import torch
    B, H, L, cap, m, head = 2, 3, 1, 5, 0, 0
    x = make_inputs(B, H, L, cap, m, "bf16", seed=11)
    c = run_gpu(x, cap, m, head, "bf16", ex=ex)
    torch.cuda.synchronize()
    assert_no_device_error()
    k, v = logical(x)
    assert_close("O", to_host(c.o), v[:, :, :L], "bf16")
    g = oracle.bwd(x["q"], k, v, x["r"], x["u"], x["vb"], x["do"], 0.125)
    for n in ("dq", "dk", "dr", "du", "dvb"):
        assert np.all(g[n] == 0), n  # the definition's value
    dv = logical_kv(to_host(c.dv), cap, head, m)
    assert_close("dV", dv, g["dv"], "bf16")
    scale_term = np.abs(x["do"]).max() * np.abs(v).max() * 0.125 * (np.abs(k).max() + np.abs(x["r"]).max()) * 64
    for n, t in (("dq", c.dq), ("dk", c.dk), ("dr", c.dr), ("du", c.du), ("dvb", c.dvb)):
        assert np.abs(to_host(t)).max() <= scale_term * 2.0 ** -16, n


@pytest.mark.parametrize("ex", [False, True], ids=["plain", "training_pair"])
@pytest.mark.parametrize("B,H,L,cap,m,head", _random_shapes(10, 3))
def test_random_shapes_full_parity(B, H, L, cap, m, head, ex):
    x = make_inputs(B, H, L, cap, m, "bf16", seed=7 * B + 13 * H + L + cap + m)
    c = run_gpu(x, cap, m, head, "bf16", ex=ex)
    compare_full(x, c, cap, m, head, "bf16", tag=str((B, H, L, cap, m, head, ex)))


@pytest.mark.parametrize("B,H,L,cap,m,head", _random_shapes(6, 0, seed=77))
def test_random_shapes_f32_full_parity(B, H, L, cap, m, head):
    x = make_inputs(B, H, L, cap, m, "f32", seed=5 * B + 11 * H + L + cap + m)
    c = run_gpu(x, cap, m, head, "f32")
    compare_full(x, c, cap, m, head, "f32", tag=str((B, H, L, cap, m, head)))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("ex", [False, True], ids=["plain", "training_pair"])
def test_backward_outputs_and_workspace_poisoned_on_entry(dtype, ex):
    """The fp32 sums (dq, dr, du, dvbias) accumulate from zero inside the
    call (du and dvbias by atomics from two kernels): NaN in every output and
    0xFF bytes in the workspace on entry, twice in a row, must not reach the
    results."""
    import torch
    if dtype == "f32" and ex:
        pytest.skip("the training pair is the bf16 path")
    B, H, L, cap, m, head = 2, 2, 200, 300, 250, 123
    x = make_inputs(B, H, L, cap, m, dtype, seed=4242)
    c = run_gpu(x, cap, m, head, dtype, bwd=False, ex=ex)
    c.alloc_bwd(x["do"])
    for rep in range(2):
        for t in (c.dq, c.dk, c.dv, c.dr, c.du, c.dvb):
            t.fill_(float("nan"))
        c.ws.fill_(0xFF)
        c.bwd_ex() if ex else c.bwd()
        compare_full(x, c, cap, m, head, dtype, tag=f"poisoned, call {rep}")


@pytest.mark.parametrize("ex", [False, True], ids=["plain", "training_pair"])
@pytest.mark.parametrize("B,H,L,cap,m,head", [(2, 2, 200, 300, 250, 123), (2, 2, 128, 256, 0, 0),
                                              (1, 2, 130, 200, 70, 190)])
def test_nan_in_ring_rows_without_memory_does_not_leak(B, H, L, cap, m, head, ex):
    # ring rows past the memory are never read as keys: whatever they hold
    # (here NaN) must not reach O or any gradient, even through a 0 weight
    x = make_inputs(B, H, L, cap, m, "bf16", seed=77 + m)
    c = run_gpu(x, cap, m, head, "bf16", ex=ex, fill=(float("nan"), float("nan")))
    compare_full(x, c, cap, m, head, "bf16", tag=str((B, H, L, cap, m, head, ex)))


@pytest.mark.parametrize("ex", [False, True], ids=["plain", "training_pair"])
def test_few_items_two_cta_clusters(ex):
    # 4 x 16 heads x one 128-row query tile = 64 items, at most half the SMs:
    # the forward runs as 2-CTA clusters, each CTA over half of an item's key
    # tiles (here 5 memory tiles on a wrapping ring + 1 current), merged
    # through distributed shared memory
    B, H, L, cap, m, head = 4, 16, 128, 640, 600, 500
    x = make_inputs(B, H, L, cap, m, "bf16", seed=4242)
    c = run_gpu(x, cap, m, head, "bf16", ex=ex)
    compare_full(x, c, cap, m, head, "bf16", tag=f"split {ex}")


@pytest.mark.parametrize("ex", [False, True], ids=["plain", "training_pair"])
def test_persistent_forward_ragged_rows(ex):
    # 4 x 16 heads x two query tiles = 128 items, more than half the SMs: the
    # persistent forward, whose O (and low part) leave by TMA stores that
    # must stop at each (b, h) plane's last row (L = 200: the second tile's
    # last 56 rows do not exist); a wrapping ring; every element, and the low
    # part against the unrounded output
    import torch
    B, H, L, cap, m, head = 4, 16, 200, 300, 250, 123
    x = make_inputs(B, H, L, cap, m, "bf16", seed=2002)
    c = run_gpu(x, cap, m, head, "bf16", ex=ex)
    compare_full(x, c, cap, m, head, "bf16", tag=f"persistent ragged {ex}")
    if ex:
        torch.cuda.synchronize()
        k, v = logical(x)
        o_ref, _ = oracle.fwd(x["q"], k, v, x["r"], x["u"], x["vb"], 0.125)
        hi, lo = to_host(c.o), to_host(c.o_lo)
        assert np.all(np.abs(lo) <= np.abs(hi) * 2.0 ** -8 + 1e-30)
        assert np.abs(hi + lo - o_ref).mean() < 0.75 * np.abs(hi - o_ref).mean()


def test_low_part_of_o_restores_the_unrounded_output():
    import torch
    B, H, L, cap, m = 2, 2, 150, 200, 180
    x = make_inputs(B, H, L, cap, m, "bf16", seed=31)
    c = run_gpu(x, cap, m, 11, "bf16", bwd=False, ex=True)
    torch.cuda.synchronize()
    k, v = logical(x)
    o_ref, _ = oracle.fwd(x["q"], k, v, x["r"], x["u"], x["vb"], 0.125)
    hi, lo = to_host(c.o), to_host(c.o_lo)
    # o_lo is what rounding O to bf16 dropped: at most half a bf16 ulp of o
    assert np.all(np.abs(lo) <= np.abs(hi) * 2.0 ** -8 + 1e-30)
    # and o + o_lo is the unrounded (fp32) O, closer to the exact O than o
    err_hi = np.abs(hi - o_ref).mean()
    err_sum = np.abs(hi + lo - o_ref).mean()
    assert err_sum < 0.75 * err_hi, (err_sum, err_hi)


def test_small_f32_full_parity():
    x = make_inputs(2, 2, 37, 50, 41, "f32", seed=3, D_model=64)
    c = run_gpu(x, 50, 41, 17, "f32")
    compare_full(x, c, 50, 41, 17, "f32")


# ---------------------------------------------- configuration 1 (fp32, 4x12)

def test_cfg1_f32_fwd_bwd_and_memory_update():
    import torch
    import long_context_lm_rel_gb300 as rxl
    w = gen.CFG1
    p, s, mem = gen.layer_params(w), gen.segment_inputs(w), gen.initial_memory(w)
    x = dict(q=s["q"], k_mem=mem["k_mem"], k_cur=s["k_cur"], v_mem=mem["v_mem"], v_cur=s["v_cur"],
             u=p["u"], vb=p["vb"], r=p["r"], do=s["do"])
    c = run_gpu(x, w.M, w.M, 0, "f32", scale=w.scale)
    compare_full(x, c, w.M, w.M, 0, "f32", scale=w.scale)
    # one memory update: ring <- last 8 of [8 memory rows; 4 current rows]
    ring = rxl.rxl_ring(c.k.data_ptr(), w.B * w.H, w.M, w.dh, (w.M + w.L) * w.dh, rxl.RXL_DTYPE_F32, 0, w.M)
    rxl.rxl_mem_update(ring, c.k.data_ptr() + w.M * w.dh * 4, (w.M + w.L) * w.dh, w.L)
    torch.cuda.synchronize()
    want = oracle.tail_m(x["k_mem"], x["k_cur"], w.M)
    got = c.k.cpu().numpy()[:, :, (ring.head + np.arange(ring.len)) % w.M]
    assert (ring.head, ring.len) == (4, 8)
    assert np.array_equal(got.view(np.uint32), want.astype(np.float32).view(np.uint32))


# -------------------------------- configuration 2 (4-segment stream, fwd+bwd)

def test_cfg2_stream_fwd_bwd():
    import torch
    import long_context_lm_rel_gb300 as rxl
    w = gen.CFG2
    p = gen.layer_params(w)
    cap, L = w.M, w.L
    mem_k = np.zeros((w.B, w.H, 0, w.dh), np.float32)
    mem_v = mem_k.copy()
    head = 0
    k_dev = v_dev = None
    for seg in range(w.segments):
        s = gen.segment_inputs(w, seg)
        m = mem_k.shape[2]
        assert m == min(cap, seg * L)
        x = dict(q=s["q"], k_mem=mem_k, k_cur=s["k_cur"], v_mem=mem_v, v_cur=s["v_cur"],
                 u=p["u"], vb=p["vb"], r=p["r"], do=s["do"])
        c = run_gpu(x, cap, m, head, "bf16", scale=w.scale)
        if k_dev is not None:   # device rings carried over from the previous segment
            c.k[:, :, :cap] = k_dev[:, :, :cap]
            c.v[:, :, :cap] = v_dev[:, :, :cap]
            c.fwd().bwd()
        compare_full(x, c, cap, m, head, "bf16", scale=w.scale, tag=f"segment {seg}")
        rk = rxl.rxl_ring(c.k.data_ptr(), w.B * w.H, cap, w.dh, (cap + L) * w.dh, rxl.RXL_DTYPE_BF16, head, m)
        rv = rxl.rxl_ring(c.v.data_ptr(), w.B * w.H, cap, w.dh, (cap + L) * w.dh, rxl.RXL_DTYPE_BF16, head, m)
        rxl.rxl_mem_update(rk, c.k.data_ptr() + cap * w.dh * 2, (cap + L) * w.dh, L)
        rxl.rxl_mem_update(rv, c.v.data_ptr() + cap * w.dh * 2, (cap + L) * w.dh, L)
        torch.cuda.synchronize()
        mem_k = oracle.tail_m(mem_k, s["k_cur"], cap)
        mem_v = oracle.tail_m(mem_v, s["v_cur"], cap)
        head = rk.head
        k_dev, v_dev = c.k.clone(), c.v.clone()


# ------------------------------------ configurations 3 and 4 (full size)

_FULL_SIZE_REF = {}


def _full_size_reference(cfg, x, scale):
    """The oracle's forward and backward of the whole configuration (every
    (b, h)), computed once per configuration and shared by both call modes."""
    if cfg not in _FULL_SIZE_REF:
        k, v = logical(x)
        o, lse = oracle.fwd(x["q"], k, v, x["r"], x["u"], x["vb"], scale)
        g = oracle.bwd(x["q"], k, v, x["r"], x["u"], x["vb"], x["do"], scale)
        _FULL_SIZE_REF.clear()
        _FULL_SIZE_REF[cfg] = (o, lse, g)
    return _FULL_SIZE_REF[cfg]


@pytest.mark.parametrize("ex", [False, True], ids=["plain", "training_pair"])
@pytest.mark.parametrize("cfg", [3, 4])
def test_full_size_config(cfg, ex):
    """Every element of every output (O, LSE, dQ, dK, dV, dR, du, dv) over all
    (b, h) at the full size of the configuration."""
    import torch
    w = gen.CONFIGS[cfg]
    p = gen.layer_params(w)
    s = gen.segment_inputs(w)
    mem = gen.initial_memory(w)
    x = dict(q=s["q"], k_mem=mem["k_mem"], k_cur=s["k_cur"], v_mem=mem["v_mem"], v_cur=s["v_cur"],
             u=p["u"], vb=p["vb"], r=p["r"], do=s["do"])
    cap = m = w.M
    c = run_gpu(x, cap, m, 0, "bf16", scale=w.scale, ex=ex)
    torch.cuda.synchronize()
    assert_no_device_error()
    o_ref, lse_ref, g = _full_size_reference(cfg, x, w.scale)
    tag = f"cfg{cfg} {'training pair' if ex else 'plain'}"
    assert_close("O", to_host(c.o), o_ref, "bf16", tag)
    assert_close("LSE", to_host(c.lse), lse_ref, "bf16", tag)
    assert_close("dQ", to_host(c.dq), g["dq"], "bf16", tag)
    assert_close("dK", logical_kv(to_host(c.dk), cap, 0, m), g["dk"], "bf16", tag)
    assert_close("dV", logical_kv(to_host(c.dv), cap, 0, m), g["dv"], "bf16", tag)
    assert_close("dR", to_host(c.dr), g["dr"], "bf16", tag)
    assert_close("du", to_host(c.du), g["du"], "bf16", tag)
    assert_close("dv", to_host(c.dvb), g["dvb"], "bf16", tag)


# -------------------- recompute-the-window evaluation baseline (forward)

def test_window_recompute_case():
    """The evaluation baseline without a memory: every step recomputes causal
    attention over the whole window of cfg5 (M + L = 1728 positions, m = 0),
    B4 H16; every row against the oracle."""
    import torch
    B, H, W = 4, 16, 1728
    x = make_inputs(B, H, W, 0, 0, "bf16", seed=1728)
    c = run_gpu(x, 0, 0, 0, "bf16", bwd=False)
    torch.cuda.synchronize()
    assert_no_device_error()
    k, v = logical(x)
    o_ref, lse_ref = oracle.fwd(x["q"], k, v, x["r"], x["u"], x["vb"], 0.125)
    assert_close("O", to_host(c.o), o_ref, "bf16")
    assert_close("LSE", to_host(c.lse), lse_ref, "bf16")


# ------------------------- configuration 5 (16-layer evaluation stream, fwd)

def test_cfg5_stream_all_layers():
    """The 32-segment stream of every one of the 16 layers: every row of O and
    LSE against the oracle at the segments where the memory is empty,
    partial, last partial, wraps, is full for the first time, and steady."""
    import torch
    import long_context_lm_rel_gb300 as rxl
    from tests._harness import to_dev
    w = gen.CFG5
    cap, L, dh = w.M, w.L, w.dh
    check_at = {0, 1, 11, 12, 13, 31}   # empty, partial, last partial, wrap, full, steady
    for layer in range(w.layers):
        p = gen.layer_params(w, layer)
        k = torch.zeros((w.B, w.H, cap + L, dh), device="cuda", dtype=torch.bfloat16)
        v = torch.zeros_like(k)
        r_dev = AttnCall(np.zeros((w.B, w.H, L, dh), np.float32), np.zeros((w.B, w.H, cap + L, dh), np.float32),
                         np.zeros((w.B, w.H, cap + L, dh), np.float32), p["r"], p["u"], p["vb"],
                         cap=cap, m=0, head=0, dtype="bf16", scale=w.scale)
        rk = rxl.rxl_ring(k.data_ptr(), w.B * w.H, cap, dh, (cap + L) * dh, rxl.RXL_DTYPE_BF16, 0, 0)
        rv = rxl.rxl_ring(v.data_ptr(), w.B * w.H, cap, dh, (cap + L) * dh, rxl.RXL_DTYPE_BF16, 0, 0)
        mem_k = np.zeros((w.B, w.H, 0, dh), np.float32)
        mem_v = mem_k.copy()
        for seg in range(w.segments):
            s = gen.segment_inputs(w, seg, layer)
            k[:, :, cap:] = to_dev(s["k_cur"], "bf16")
            v[:, :, cap:] = to_dev(s["v_cur"], "bf16")
            q = to_dev(s["q"], "bf16")
            desc = rxl.make_desc(w.B, w.H, L, cap, rk.len, rk.head, w.scale, rxl.RXL_DTYPE_BF16)
            rxl.rxl_attn_fwd(desc, q, k, v, r_dev.r, r_dev.u, r_dev.vb, r_dev.o, r_dev.lse)
            if seg in check_at:
                torch.cuda.synchronize()
                kl = np.concatenate([mem_k, s["k_cur"]], 2)
                vl = np.concatenate([mem_v, s["v_cur"]], 2)
                o_ref, lse_ref = oracle.fwd(s["q"], kl, vl, p["r"], p["u"], p["vb"], w.scale)
                tag = f"layer {layer} segment {seg} m={rk.len} head={rk.head}"
                assert_close("O", to_host(r_dev.o), o_ref, "bf16", tag)
                assert_close("LSE", to_host(r_dev.lse), lse_ref, "bf16", tag)
            rxl.rxl_mem_update(rk, k.data_ptr() + cap * dh * 2, (cap + L) * dh, L)
            rxl.rxl_mem_update(rv, v.data_ptr() + cap * dh * 2, (cap + L) * dh, L)
            mem_k = oracle.tail_m(mem_k, s["k_cur"], cap)
            mem_v = oracle.tail_m(mem_v, s["v_cur"], cap)
        assert (rk.len, rk.head) == (cap, (32 * L - cap) % cap)
    assert_no_device_error()


# ------------------------------------------- skew-sensitive closed-form probes

@pytest.mark.parametrize("L,cap,m,head", [(4, 8, 8, 0), (127, 129, 129, 5), (128, 128, 128, 0),
                                           (129, 127, 127, 100), (128, 1600, 1600, 1550), (257, 0, 0, 0)])
def test_distance_probe_on_gpu(L, cap, m, head):
    """Q=K=u=0, v = alpha*(64 e0 + e1), R_d = (d // 64, d % 64, 0...): the
    logits are s*alpha*(i-j), exact in bf16, so P is a truncated geometric
    law over the distance i-j. V_j carries small labels of its logical
    position p = j+m: (1, p % 8, (p // 8) % 8, p // 64). O_i is then the
    expected label under that law and LSE_i a closed form; a key or a
    distance off by one moves the expected labels by ~1."""
    B, H, dh, s, alpha = 2, 2, 64, 0.125, -16.0   # s*alpha = -2
    q = np.zeros((B, H, L, dh), np.float32)
    n = m + L
    kk = np.zeros((B, H, cap + L, dh), np.float32)
    lab = np.arange(n)
    feats = [np.ones(n), lab % 8, (lab // 8) % 8, lab // 64]
    vlog = np.zeros((B, H, n, dh), np.float32)
    for ch, f in enumerate(feats):
        vlog[..., ch] = f
    vv = place_kv(vlog[:, :, :m], vlog[:, :, m:], cap, head, fill=1000.0)
    r = np.zeros((H, cap + L, dh), np.float32)
    d = np.arange(cap + L)
    r[:, :, 0], r[:, :, 1] = d // 64, d % 64
    vb = np.zeros((H, dh), np.float32)
    vb[:, 0], vb[:, 1] = 64 * alpha, alpha
    c = AttnCall(q, kk, vv, r, np.zeros((H, dh), np.float32), vb, cap=cap, m=m, head=head,
                 dtype="bf16", scale=s).fwd()
    import torch
    torch.cuda.synchronize()
    o, lse = to_host(c.o), to_host(c.lse)
    rho = math.exp(s * alpha)
    for i in range(L):
        w = rho ** np.arange(i + m + 1)           # weight of distance d = 0..i+m
        tot = w.sum()
        pos = i + m - np.arange(i + m + 1)        # logical position of the key at distance d
        assert np.abs(lse[:, :, i] - math.log(tot)).max() < 2e-3, i
        for ch, f in enumerate(feats):
            want = (w * f[pos]).sum() / tot
            err = np.abs(o[:, :, i, ch] - want).max()
            assert err <= 0.01 + 2 ** -8 * abs(want), (i, ch, float(err), want)


def test_ring_rotation_gives_same_outputs():
    """Translation invariance on the device: the same logical memory stored
    at another ring head gives the same O and LSE."""
    B, H, L, cap, m = 2, 2, 100, 300, 260
    x = make_inputs(B, H, L, cap, m, "bf16", seed=77)
    outs = []
    for head in (0, 41, 299):
        c = run_gpu(x, cap, m, head, "bf16", bwd=False)
        outs.append((to_host(c.o), to_host(c.lse)))
    for o, l in outs[1:]:
        np.testing.assert_allclose(o, outs[0][0], rtol=0, atol=2e-3)
        np.testing.assert_allclose(l, outs[0][1], rtol=0, atol=1e-5)


def test_backward_never_writes_the_cache():
    import torch
    B, H, L, cap, m = 2, 2, 96, 160, 150
    x = make_inputs(B, H, L, cap, m, "bf16", seed=13)
    c = run_gpu(x, cap, m, 37, "bf16", bwd=False)
    k0, v0 = c.k.clone(), c.v.clone()
    c.alloc_bwd(x["do"]).bwd()
    torch.cuda.synchronize()
    assert torch.equal(c.k, k0) and torch.equal(c.v, v0)
    mem_rows = (37 + np.arange(m)) % cap
    dk = to_host(c.dk)[:, :, mem_rows]
    assert np.all(np.abs(dk).sum(-1) > 0), "memory rows must receive K gradients"


def test_backward_run_to_run_variation():
    """dK, dV and the forward are reproducible bit for bit (each row comes from
    one CTA's tensor-memory accumulator, summed in a fixed order); dQ, dR, du
    and dv are sums over tiles added by hardware reductions in an order that
    varies between runs, so they agree to fp32 rounding: dR, du, dv (fp32)
    well inside 1e-4 of their largest element, dQ (rounded to bf16 after the
    sum) within one bf16 step of each element."""
    import torch
    B, H, L, cap, m = 2, 4, 384, 512, 500
    x = make_inputs(B, H, L, cap, m, "bf16", seed=90)
    c = run_gpu(x, cap, m, 3, "bf16", ex=True)
    torch.cuda.synchronize()
    first = {n: getattr(c, n).clone() for n in ("o", "lse", "dq", "dk", "dv", "dr", "du", "dvb")}
    for _ in range(3):
        c.fwd_ex().bwd_ex()
        torch.cuda.synchronize()
        for n in ("o", "lse", "dk", "dv"):
            assert torch.equal(getattr(c, n), first[n]), n
        a, b = c.dq.float(), first["dq"].float()
        assert bool(((a - b).abs() <= 2.0 ** -7 * torch.maximum(a.abs(), b.abs())).all()), "dq"
        for n in ("dr", "du", "dvb"):
            a, b = getattr(c, n).float(), first[n].float()
            assert (a - b).abs().max().item() <= 1e-4 * b.abs().max().item(), n
    assert_no_device_error()
