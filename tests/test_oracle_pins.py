"""Pins of the float64 oracle to facts the pages and the mathematics fix.

Each test ties one part of the oracle to something other than itself: a
picture or worked example printed on the pages (tests/golden/), a library
routine (torch scaled_dot_product_attention in float64), a closed form, the
pages' own relative-shift trick, a brute-force stream, or finite differences.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from tests import _golden

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def rand(rng, *shape, std=1.0):
    return rng.standard_normal(shape) * std


def make_txl_mask(q_len, mem_len):
    """Restatement of make_txl_mask (Transformer-XL page, "Causal Mask With
    Memory"): ones for the memory block, a lower triangle for the current
    block; True = visible. Shape [q_len, mem_len + q_len]."""
    mem_visible = torch.ones(q_len, mem_len, dtype=torch.bool)
    cur_visible = torch.ones(q_len, q_len, dtype=torch.bool).tril()
    return torch.cat([mem_visible, cur_visible], dim=-1)


def reference_rel_ids(q_len, mem_len):
    """Restatement of reference_rel_ids (Transformer-XL page, "Relative Shift
    Golden Test"): query position minus key position, keys -mem_len..q_len-1."""
    key_pos = torch.arange(-mem_len, q_len)
    query_pos = torch.arange(q_len)
    return query_pos[:, None] - key_pos[None, :]


def relative_shift(x):
    """Restatement of the relative-shift trick (Transformer-XL page, "Relative
    Shift Trick"): prepend a zero column, view as [k+1, q], drop the first
    row, view back as [q, k]."""
    b, h, q_len, k_len = x.shape
    zero = x.new_zeros(b, h, q_len, 1)
    x = torch.cat([zero, x], dim=-1)
    x = x.view(b, h, k_len + 1, q_len)
    return x[:, :, 1:].reshape(b, h, q_len, k_len)


def visible_from_probe(L, m, dh=64):
    """Recover the visible set from the oracle's output alone: with Q=K=R=u=v=0
    every visible key gets equal weight, and V_j = one-hot(j+m) makes
    O_i[c] = 1/count_i on exactly the visible columns."""
    assert m + L <= dh
    q = np.zeros((1, 1, L, dh))
    k = np.zeros((1, 1, m + L, dh))
    v = np.zeros((1, 1, m + L, dh))
    for c in range(m + L):
        v[0, 0, c, c] = 1.0
    r = np.zeros((1, m + L, dh))
    z = np.zeros((1, dh))
    o, lse = oracle.fwd(q, k, v, r, z, z, 0.125, nthreads=1)
    return o[0, 0, :, :m + L] > 0, o, lse


# ------------------------------------------------------------------ P-1 mask

def test_mask_matches_page_picture():
    want = _golden.mask_picture()
    L, m = want.shape[0], want.shape[1] - want.shape[0]
    got, o, lse = visible_from_probe(L, m)
    assert got.shape == (4, 7)
    np.testing.assert_array_equal(got, want)
    np.testing.assert_array_equal(got, make_txl_mask(L, m).numpy())
    # uniform weights: O_i = 1/count on visible columns, LSE_i = log(count)
    counts = want.sum(1)
    np.testing.assert_allclose(o[0, 0, np.arange(L), m + np.arange(L)], 1.0 / counts, rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse[0, 0], np.log(counts), rtol=0, atol=1e-15)


def test_worked_example_score_shape():
    ex = _golden.worked_example()
    L, m = ex["L"], ex["M"]
    rng = np.random.default_rng(1)
    z = oracle.logits(rand(rng, 1, 1, L, 64), rand(rng, 1, 1, m + L, 64), rand(rng, 1, m + L, 64),
                      rand(rng, 1, 64), rand(rng, 1, 64), 0.125, nthreads=1)
    assert z.shape[2:] == (ex["score_rows"], ex["score_cols"])
    vis = np.isfinite(z[0, 0])
    assert vis.sum(1).tolist() == [m + i + 1 for i in range(L)] == [9, 10, 11, 12]
    assert vis.sum() == 42
    got, _, _ = visible_from_probe(L, m)
    np.testing.assert_array_equal(got, vis)
    # the cached states of one layer hold M x width numbers
    assert oracle.tail_m(np.zeros((m, ex["width"])), np.zeros((L, ex["width"])), m).size == ex["memory_numbers"]


# ------------------------------------------- P-2 reduction to plain attention

def sdpa(q, k, v, mask, scale):
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))
    return F.scaled_dot_product_attention(t(q), t(k), t(v), attn_mask=mask, scale=scale).numpy()


@pytest.mark.parametrize("B,H,L,m", [(2, 3, 5, 7), (1, 2, 9, 0), (2, 1, 16, 16)])
def test_reduces_to_masked_attention(B, H, L, m):
    rng = np.random.default_rng(2 + L + m)
    dh, s = 16, 0.25
    q, k, v = rand(rng, B, H, L, dh), rand(rng, B, H, m + L, dh), rand(rng, B, H, m + L, dh)
    zr, zh = np.zeros((H, m + L, dh)), np.zeros((H, dh))
    o, lse = oracle.fwd(q, k, v, zr, zh, zh, s, nthreads=2)
    want = sdpa(q, k, v, make_txl_mask(L, m), s)
    np.testing.assert_allclose(o, want, rtol=0, atol=1e-12)
    if m == 0:
        t = lambda a: torch.from_numpy(a)
        causal = F.scaled_dot_product_attention(t(q), t(k), t(v), is_causal=True, scale=s).numpy()
        np.testing.assert_allclose(o, causal, rtol=0, atol=1e-12)
    logit = torch.from_numpy(np.einsum("bhid,bhjd->bhij", q, k) * s)
    logit = logit.masked_fill(~make_txl_mask(L, m), -math.inf)
    np.testing.assert_allclose(lse, torch.logsumexp(logit, -1).numpy(), rtol=0, atol=1e-12)


# --------------------------------------------------- P-3 bias terms separately

def test_content_bias_u_is_a_key_bias():
    rng = np.random.default_rng(3)
    B, H, L, m, dh, s = 2, 2, 6, 5, 16, 0.25
    q, k, v = rand(rng, B, H, L, dh), rand(rng, B, H, m + L, dh), rand(rng, B, H, m + L, dh)
    u = rand(rng, H, dh)
    o, _ = oracle.fwd(q, k, v, np.zeros((H, m + L, dh)), u, rand(rng, H, dh), s, nthreads=1)
    bias = s * np.einsum("hd,bhjd->bhj", u, k)[:, :, None, :]            # s * u.k_j
    mask = torch.from_numpy(np.broadcast_to(bias, (B, H, L, m + L)).copy())
    mask = mask.masked_fill(~make_txl_mask(L, m), -math.inf)
    np.testing.assert_allclose(o, sdpa(q, k, v, mask, s), rtol=0, atol=1e-12)


def test_position_terms_are_toeplitz_biases():
    rng = np.random.default_rng(4)
    B, H, L, m, dh, s = 1, 2, 7, 6, 16, 0.25
    k, v = rand(rng, B, H, m + L, dh), rand(rng, B, H, m + L, dh)
    r = rand(rng, H, m + L, dh)
    vb = rand(rng, H, dh)
    ids = reference_rel_ids(L, m)
    vis = make_txl_mask(L, m)
    safe = ids.clamp(min=0).numpy()
    # (a) global position bias alone (q = 0, u = 0): s * v.r_{i-j}
    q0 = np.zeros((B, H, L, dh))
    o, _ = oracle.fwd(q0, k, v, r, np.zeros((H, dh)), vb, s, nthreads=1)
    bias = s * np.einsum("hd,hnd->hn", vb, r)[:, safe]                    # [H, L, m+L]
    mask = torch.from_numpy(np.broadcast_to(bias, (B, H, L, m + L)).copy()).masked_fill(~vis, -math.inf)
    np.testing.assert_allclose(o, sdpa(q0, k, v, mask, s), rtol=0, atol=1e-12)
    # (b) content-position term alone (k = 0, u = v = 0): s * q_i.r_{i-j}
    q = rand(rng, B, H, L, dh)
    k0 = np.zeros_like(k)
    z = oracle.logits(q, k0, r, np.zeros((H, dh)), np.zeros((H, dh)), s, nthreads=1)
    qr = np.einsum("bhid,hnd->bhin", q, r)                               # [B,H,L,m+L]
    want = s * np.take_along_axis(qr, np.broadcast_to(safe, qr.shape), axis=-1)
    np.testing.assert_allclose(z[..., vis.numpy()], want[..., vis.numpy()], rtol=0, atol=1e-12)
    assert np.all(np.isneginf(z[..., ~vis.numpy()]))


# -------------------------------- P-4 / P-5 closed-form skew and distance labels

def distance_probe(L, m, alpha, dh=64):
    """Q=K=u=0, v = alpha*(64 e0 + e1), R_d = (floor(d/64), d mod 64, 0...), so
    v.R_d = alpha*d exactly and the logits are s*alpha*(i-j)."""
    n = m + L
    r = np.zeros((1, n, dh))
    d = np.arange(n)
    r[0, :, 0], r[0, :, 1] = d // 64, d % 64
    vb = np.zeros((1, dh))
    vb[0, 0], vb[0, 1] = 64 * alpha, alpha
    return np.zeros((1, 1, L, dh)), np.zeros((1, 1, n, dh)), r, np.zeros((1, dh)), vb


@pytest.mark.parametrize("L,m", [(4, 8), (4, 3), (7, 0), (16, 40)])
def test_skew_closed_form(L, m):
    s, alpha = 0.125, -1.6
    q, k, r, u, vb = distance_probe(L, m, alpha)
    v = np.zeros((1, 1, m + L, 64))
    for c in range(m + L):
        v[0, 0, c, c] = 1.0
    o, lse = oracle.fwd(q, k, v, r, u, vb, s, nthreads=1)
    rho = math.exp(s * alpha)
    for i in range(L):
        tot = (rho ** (i + m + 1) - 1.0) / (rho - 1.0)
        assert abs(lse[0, 0, i] - math.log(tot)) < 1e-13
        for jj in range(m + L):
            j = jj - m
            want = rho ** (i - j) / tot if j <= i else 0.0
            assert abs(o[0, 0, i, jj] - want) < 1e-15


@pytest.mark.parametrize("L,m", [(4, 3), (4, 8), (9, 5)])
def test_distance_labels_match_reference_rel_ids(L, m):
    s, alpha = 0.125, -2.0
    q, k, r, u, vb = distance_probe(L, m, alpha)
    v = np.zeros((1, 1, m + L, 64))
    for c in range(m + L):
        v[0, 0, c, c] = 1.0
    o, _ = oracle.fwd(q, k, v, r, u, vb, s, nthreads=1)
    p = o[0, 0, :, :m + L]
    diag = p[np.arange(L), m + np.arange(L)]
    vis = make_txl_mask(L, m).numpy()
    with np.errstate(divide="ignore"):
        ids = np.log(p / diag[:, None]) / (s * alpha)
    want = reference_rel_ids(L, m).numpy()
    np.testing.assert_allclose(ids[vis], want[vis], rtol=0, atol=1e-9)
    if (L, m) == (4, 3):
        np.testing.assert_array_equal(want, _golden.rel_ids())


# --------------------------------------- P-6 the pages' shift trick == lookup

@pytest.mark.parametrize("L,m", [(4, 8), (5, 0), (6, 11)])
def test_relative_shift_trick_equals_direct_lookup(L, m):
    rng = np.random.default_rng(6 + L)
    B, H, dh, s = 2, 2, 8, 0.3
    q = rand(rng, B, H, L, dh)
    r = rand(rng, H, m + L, dh)
    zero = np.zeros((H, dh))
    z = oracle.logits(q, np.zeros((B, H, m + L, dh)), r, zero, zero, s, nthreads=1)
    r_desc = r[:, ::-1, :]                      # column c <-> distance (m+L-1) - c
    x = torch.from_numpy(np.einsum("bhid,hcd->bhic", q, r_desc).copy())
    shifted = s * relative_shift(x).numpy()
    vis = make_txl_mask(L, m).numpy()
    np.testing.assert_allclose(z[..., vis], shifted[..., vis], rtol=0, atol=1e-12)


# --------------------------- P-7 rolling memory == attention over the stream

def test_rolling_memory_sees_exactly_last_M_states():
    rng = np.random.default_rng(7)
    L, M, S, dh, s = 3, 5, 6, 4, 0.5
    T = L * S
    q, k, v = rand(rng, T, dh), rand(rng, T, dh), rand(rng, T, dh)
    r = rand(rng, M + L, dh)
    u, vb = rand(rng, dh), rand(rng, dh)
    want = oracle.fullseq_fwd(q, k, v, r, u, vb, s, L, M)
    mem_k = np.zeros((0, dh))
    mem_v = np.zeros((0, dh))
    got = []
    for seg in range(S):
        sl = slice(seg * L, (seg + 1) * L)
        kk = np.concatenate([mem_k, k[sl]])[None, None]
        vv = np.concatenate([mem_v, v[sl]])[None, None]
        m = mem_k.shape[0]
        o, _ = oracle.fwd(q[sl][None, None], kk, vv, r[None, :m + L], u[None], vb[None], s, nthreads=1)
        got.append(o[0, 0])
        mem_k = oracle.tail_m(mem_k, k[sl], M)
        mem_v = oracle.tail_m(mem_v, v[sl], M)
        assert mem_k.shape[0] == min(M, (seg + 1) * L)
    np.testing.assert_allclose(np.concatenate(got), want, rtol=0, atol=1e-12)


# ----------------------------------------------------- P-8 Tail_M bit-exact

@pytest.mark.parametrize("M,L,steps", [(0, 3, 3), (5, 2, 6), (4, 4, 4), (3, 7, 3), (1600, 128, 16), (6, 1, 9)])
def test_tail_m_keeps_last_M_labels(M, L, steps):
    mem = np.zeros((2, 0, 3))
    labels = []
    for t in range(steps):
        new = np.arange(t * L, (t + 1) * L, dtype=np.float64)
        labels += new.tolist()
        hids = np.broadcast_to(new[None, :, None], (2, L, 3)).copy()
        mem = oracle.tail_m(mem, hids, M)
        want = labels[max(0, len(labels) - M):] if M > 0 else []
        assert mem.shape == (2, len(want), 3)
        np.testing.assert_array_equal(mem[0, :, 0], np.array(want, dtype=np.float64))


# ------------------------------------------ P-9 translation invariance

def test_outputs_independent_of_absolute_offset():
    rng = np.random.default_rng(9)
    B, H, L, m, dh, s = 2, 2, 5, 6, 8, 0.35
    args = (rand(rng, B, H, L, dh), rand(rng, B, H, m + L, dh), rand(rng, B, H, m + L, dh),
            rand(rng, H, m + L, dh), rand(rng, H, dh), rand(rng, H, dh))
    do = rand(rng, B, H, L, dh)
    base_o, base_l = oracle.fwd(*args, s, pos0=0, nthreads=1)
    base_g = oracle.bwd(*args, do, s, pos0=0, nthreads=1)
    for c in (17, 10**6, 3 * 10**12):
        o, l = oracle.fwd(*args, s, pos0=c, nthreads=1)
        assert np.array_equal(o, base_o) and np.array_equal(l, base_l)
        g = oracle.bwd(*args, do, s, pos0=c, nthreads=1)
        for key in base_g:
            assert np.array_equal(g[key], base_g[key]), key


# ----------------------------------------------------------- P-10 gradients

def _cfg1_like(rng):
    L, m, dh = 4, 8, 64
    return dict(q=rand(rng, 1, 1, L, dh, std=0.125), k=rand(rng, 1, 1, m + L, dh, std=0.125),
                v=rand(rng, 1, 1, m + L, dh, std=0.125), r=rand(rng, 1, m + L, dh, std=0.7),
                u=rand(rng, 1, dh, std=0.02), vb=rand(rng, 1, dh, std=0.02))


def test_gradients_match_central_differences():
    lib = oracle.load()
    rng = np.random.default_rng(10)
    x = _cfg1_like(rng)
    do = rand(rng, 1, 1, 4, 64)
    s = 0.125
    names = ["q", "k", "v", "r", "u", "vb"]

    def loss(vals):
        o, _ = oracle.fwd(*(vals[n] for n in names), s, nthreads=1, lib=lib)
        return float(np.sum(o * do))

    g = oracle.bwd(*(x[n] for n in names), do, s, nthreads=1, lib=lib)
    grad_of = {"q": "dq", "k": "dk", "v": "dv", "r": "dr", "u": "du", "vb": "dvb"}
    h = 1e-6
    for n in names:
        an = g[grad_of[n]]
        fd = np.zeros_like(x[n])
        flat = x[n].reshape(-1)
        for e in range(flat.size):
            keep = flat[e]
            flat[e] = keep + h
            lp = loss(x)
            flat[e] = keep - h
            lm = loss(x)
            flat[e] = keep
            fd.reshape(-1)[e] = (lp - lm) / (2 * h)
        err = np.max(np.abs(fd - an)) / np.max(np.abs(an))
        assert err <= 1e-6, (n, err)


def test_gradient_identities_and_stop_gradient():
    rng = np.random.default_rng(11)
    B, H, L, m, dh, s = 3, 2, 6, 5, 8, 0.3
    q, k, v = rand(rng, B, H, L, dh), rand(rng, B, H, m + L, dh), rand(rng, B, H, m + L, dh)
    r, u, vb = rand(rng, H, m + L, dh), rand(rng, H, dh), rand(rng, H, dh)
    do = rand(rng, B, H, L, dh)
    g = oracle.bwd(q, k, v, r, u, vb, do, s, nthreads=3)
    tol = 1e-12
    # softmax rows: sum_j dA_ij = 0, hence sum_j dK_j = 0 per (b,h) and sum_d dR_d = 0 per h
    assert np.max(np.abs(g["dk"].sum(2))) < tol
    assert np.max(np.abs(g["dr"].sum(1))) < tol
    # sum_j dV_j = sum_i dO_i per (b,h)
    np.testing.assert_allclose(g["dv"].sum(2), do.sum(2), rtol=0, atol=tol)
    # sum_{b,i} dQ_i = du + dv per head
    np.testing.assert_allclose(g["dq"].sum((0, 2)), g["du"] + g["dvb"], rtol=0, atol=tol)
    # stop-gradient: memory K/V rows still receive gradients (W_K, W_V learn
    # from them); there is no gradient output for the cached states at all
    assert np.min(np.abs(g["dk"][:, :, :m]).sum(-1)) > 0
    assert np.min(np.abs(g["dv"][:, :, :m]).sum(-1)) > 0
    assert set(g) == {"dq", "dk", "dv", "dr", "du", "dvb"}


def test_row_subset_and_threads_agree_with_full_forward():
    rng = np.random.default_rng(12)
    B, H, L, m, dh, s = 2, 3, 7, 9, 16, 0.25
    args = (rand(rng, B, H, L, dh), rand(rng, B, H, m + L, dh), rand(rng, B, H, m + L, dh),
            rand(rng, H, m + L, dh), rand(rng, H, dh), rand(rng, H, dh))
    o1, l1 = oracle.fwd(*args, s, nthreads=1)
    o4, l4 = oracle.fwd(*args, s, nthreads=4)
    assert np.array_equal(o1, o4) and np.array_equal(l1, l4)
    sel = [(1, 2, 6), (0, 0, 0), (1, 0, 3)]
    o, l = oracle.fwd_rows(*args, s, sel, nthreads=2)
    for n, (b, h, i) in enumerate(sel):
        assert np.array_equal(o[n], o1[b, h, i]) and l[n] == l1[b, h, i]


# ------------------------------------------------ per-row document reset

def reset_vs_sliced(mvis, B=3, H=2, L=6, m=7, dh=16, seed=11, lib=None):
    """Per-row reset ("Causal Mask With Memory", the note after the picture;
    "Batched Streams"): batch row b that sees only its newest mvis[b] memory
    rows must give exactly what the plain oracle gives on that row alone with
    only those memory rows (masking a key = removing it). Returns the names
    of the outputs that differ."""
    rng = np.random.default_rng(seed)
    q, k, v = rand(rng, B, H, L, dh), rand(rng, B, H, m + L, dh), rand(rng, B, H, m + L, dh)
    r, u, vb = rand(rng, H, m + L, dh), rand(rng, H, dh, std=0.3), rand(rng, H, dh, std=0.3)
    do = rand(rng, B, H, L, dh)
    o, lse = oracle.fwd(q, k, v, r, u, vb, 0.4, mem_visible=mvis, nthreads=1, lib=lib)
    g = oracle.bwd(q, k, v, r, u, vb, do, 0.4, mem_visible=mvis, nthreads=1, lib=lib)
    bad = []
    dr = np.zeros((H, m + L, dh))
    du, dvb = np.zeros((H, dh)), np.zeros((H, dh))
    for b in range(B):
        mb = int(mvis[b])
        keep = np.r_[m - mb:m + L]                    # newest mb memory rows, then the segment
        ob, lb = oracle.fwd(q[b:b + 1], k[b:b + 1][:, :, keep], v[b:b + 1][:, :, keep], r, u, vb, 0.4,
                            nthreads=1, lib=lib)
        gb = oracle.bwd(q[b:b + 1], k[b:b + 1][:, :, keep], v[b:b + 1][:, :, keep], r, u, vb,
                        do[b:b + 1], 0.4, nthreads=1, lib=lib)
        if not np.array_equal(o[b], ob[0]) or not np.array_equal(lse[b], lb[0]):
            bad.append(f"fwd[{b}]")
        if not np.array_equal(g["dq"][b], gb["dq"][0]):
            bad.append(f"dq[{b}]")
        for n in ("dk", "dv"):
            if not np.array_equal(g[n][b][:, keep], gb[n][0]) or np.any(g[n][b][:, :m - mb] != 0):
                bad.append(f"{n}[{b}]")
        dr[:, :mb + L] += gb["dr"]
        du += gb["du"]
        dvb += gb["dvb"]
    for n, ref in (("dr", dr), ("du", du), ("dvb", dvb)):
        if not np.array_equal(g[n], ref):
            bad.append(n)
    return bad


@pytest.mark.parametrize("mvis", [(7, 0, 3), (0, 0, 0), (7, 7, 7), (1, 6, 2)])
def test_document_reset_equals_the_row_alone(mvis):
    assert reset_vs_sliced(mvis) == []


# ------------------------------------------------ projection front-end

def test_projection_matches_brute_force_and_head_split():
    """Q = H W^Q, K/V = [SG(M); H] W^{K,V} ("Segment-Level Recurrence"), head h
    taking columns h*dh .. h*dh+dh-1: checked element by element with loops."""
    rng = np.random.default_rng(5)
    B, m, L, d, H, dh = 2, 3, 4, 8, 2, 3
    hm, hc = rand(rng, B, m, d), rand(rng, B, L, d)
    wq, wk, wv = rand(rng, d, H * dh), rand(rng, d, H * dh), rand(rng, d, H * dh)
    q, k, v = oracle.proj(hm, hc, wq, wk, wv, H)
    assert q.shape == (B, H, L, dh) and k.shape == (B, H, m + L, dh) and v.shape == k.shape
    for b in range(B):
        for h in range(H):
            for e in range(dh):
                col = h * dh + e
                for i in range(L):
                    assert abs(q[b, h, i, e] - sum(hc[b, i, c] * wq[c, col] for c in range(d))) < 1e-12
                for j in range(m + L):
                    row = hm[b, j] if j < m else hc[b, j - m]
                    assert abs(k[b, h, j, e] - sum(row[c] * wk[c, col] for c in range(d))) < 1e-12
                    assert abs(v[b, h, j, e] - sum(row[c] * wv[c, col] for c in range(d))) < 1e-12


def test_projection_identity_weights_split_the_hidden_state():
    rng = np.random.default_rng(6)
    B, m, L, H, dh = 2, 5, 3, 4, 2
    d = H * dh
    hm, hc = rand(rng, B, m, d), rand(rng, B, L, d)
    eye = np.eye(d)
    q, k, v = oracle.proj(hm, hc, eye, eye, eye, H)
    ht = np.concatenate([hm, hc], 1)
    for h in range(H):
        assert np.array_equal(q[:, h], hc[:, :, h * dh:(h + 1) * dh])
        assert np.array_equal(k[:, h], ht[:, :, h * dh:(h + 1) * dh])
        assert np.array_equal(v[:, h], ht[:, :, h * dh:(h + 1) * dh])
    # queries come from the current segment only: the memory never changes q
    q2, _, _ = oracle.proj(hm * 0 + 7.0, hc, eye, eye, eye, H)
    assert np.array_equal(q, q2)


# ------------------------------------------------ evaluation layer

def _layer_weights(rng, H, dh, d, dff, m, L):
    return dict(w_q=rand(rng, d, H * dh, std=d ** -0.5), w_k=rand(rng, d, H * dh, std=d ** -0.5),
                w_v=rand(rng, d, H * dh, std=d ** -0.5), w_o=rand(rng, H * dh, d, std=(H * dh) ** -0.5),
                r=rand(rng, H, m + L, dh), u=rand(rng, H, dh, std=0.1), vbias=rand(rng, H, dh, std=0.1),
                ln1_gamma=1 + rand(rng, d, std=0.1), ln1_beta=rand(rng, d, std=0.1),
                w_1=rand(rng, d, dff, std=d ** -0.5), b_1=rand(rng, dff, std=0.1),
                w_2=rand(rng, dff, d, std=dff ** -0.5), b_2=rand(rng, d, std=0.1),
                ln2_gamma=1 + rand(rng, d, std=0.1), ln2_beta=rand(rng, d, std=0.1))


def test_layer_norm_matches_torch():
    rng = np.random.default_rng(8)
    x, g, b = rand(rng, 3, 5, 16), rand(rng, 16), rand(rng, 16)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(x), (16,), torch.from_numpy(g),
                                         torch.from_numpy(b), eps=1e-5).numpy()
    assert np.allclose(oracle.layer_norm(x, g, b), ref, rtol=1e-13, atol=1e-13)


def test_layer_with_silent_sublayers_is_two_norms():
    """W_O = 0 and a zero FFN leave only the residual path: LN2(LN1(h))."""
    rng = np.random.default_rng(9)
    B, H, dh, L, m = 2, 2, 4, 3, 5
    d, dff = H * dh, 12
    w = _layer_weights(rng, H, dh, d, dff, m, L)
    for n in ("w_o", "w_1", "b_1", "w_2", "b_2"):
        w[n] = np.zeros_like(w[n])
    hm, hi = rand(rng, B, m, d), rand(rng, B, L, d)
    out = oracle.layer_fwd(hm, hi, w, H, 0.5, nthreads=1)
    ref = oracle.layer_norm(oracle.layer_norm(hi, w["ln1_gamma"], w["ln1_beta"]),
                            w["ln2_gamma"], w["ln2_beta"])
    assert np.allclose(out, ref, rtol=1e-13, atol=1e-13)


def test_layer_merges_heads_in_column_order():
    """With W_O = I and the FFN silent, LN1's input is h + [o_head0 | o_head1 | ...]."""
    rng = np.random.default_rng(10)
    B, H, dh, L, m = 2, 3, 4, 5, 6
    d, dff = H * dh, 8
    w = _layer_weights(rng, H, dh, d, dff, m, L)
    w["w_o"] = np.eye(d)
    for n in ("w_1", "b_1", "w_2", "b_2"):
        w[n] = np.zeros_like(w[n])
    w["ln1_gamma"], w["ln1_beta"] = np.ones(d), np.zeros(d)
    w["ln2_gamma"], w["ln2_beta"] = np.ones(d), np.zeros(d)
    hm, hi = rand(rng, B, m, d), rand(rng, B, L, d)
    q, k, v = oracle.proj(hm, hi, w["w_q"], w["w_k"], w["w_v"], H)
    o, _ = oracle.fwd(q, k, v, w["r"], w["u"], w["vbias"], 0.5, nthreads=1)
    x1 = hi + np.concatenate([o[:, h] for h in range(H)], axis=-1)
    ref = oracle.layer_norm(oracle.layer_norm(x1, np.ones(d), np.zeros(d)), np.ones(d), np.zeros(d))
    assert np.allclose(oracle.layer_fwd(hm, hi, w, H, 0.5, nthreads=1), ref, rtol=1e-12, atol=1e-12)


# ------------------------------------------- the feed-forward sublayer
# With W_O = 0 the attention sublayer contributes nothing (x1 = h_in), so
# x1n = LN1(h_in) is known without the attention and the feed-forward
# sublayer x2 = x1n + ReLU(x1n W_1 + b_1) W_2 + b_2 can be pinned to closed
# forms; LN2 (gamma = 1, beta = 0) of x2 is what the layer returns. Each pin
# takes the oracle module, so that the mutant tests can run it on a copy.

def _ffn_layer(mod, rng, d, dff, H=2):
    dh = d // H
    m, L = 3, 4
    w = _layer_weights(rng, H, dh, d, dff, m, L)
    w["w_o"] = np.zeros_like(w["w_o"])
    w["ln2_gamma"], w["ln2_beta"] = np.ones(d), np.zeros(d)
    hm, hi = rand(rng, 2, m, d), rand(rng, 2, L, d)
    x1n = mod.layer_norm(hi, w["ln1_gamma"], w["ln1_beta"])
    return w, hm, hi, x1n, H


def _ln_plain(x):
    mu = x.mean(-1, keepdims=True)
    return (x - mu) / np.sqrt(((x - mu) ** 2).mean(-1, keepdims=True) + 1e-5)


def ffn_pin_absolute_value(mod) -> bool:
    """W_1 = [I | -I], b_1 = 0, W_2 = [I ; I], b_2 = 0: ReLU(x) + ReLU(-x) = |x|,
    so x2 = x1n + |x1n| = 2 max(x1n, 0). Without the ReLU the pair cancels
    (x2 = x1n); a ReLU after W_2 instead of after W_1 gives ReLU(x - x) = 0."""
    rng = np.random.default_rng(21)
    d = 8
    w, hm, hi, x1n, H = _ffn_layer(mod, rng, d, 2 * d)
    eye = np.eye(d)
    w["w_1"], w["b_1"] = np.concatenate([eye, -eye], 1), np.zeros(2 * d)
    w["w_2"], w["b_2"] = np.concatenate([eye, eye], 0), np.zeros(d)
    assert (x1n < 0).any() and (x1n > 0).any()  # the ReLU clips somewhere
    out = mod.layer_fwd(hm, hi, w, H, 0.5, nthreads=1)
    return bool(np.allclose(out, _ln_plain(2 * np.maximum(x1n, 0)), rtol=0, atol=1e-12))


def ffn_pin_bias_before_relu(mod) -> bool:
    """W_1 = 0, b_1 = c with both signs: the hidden units are ReLU(c) (a bias
    added after the ReLU would give c); W_2 = I, b_2 = e: x2 = x1n + ReLU(c) + e."""
    rng = np.random.default_rng(22)
    d = 8
    w, hm, hi, x1n, H = _ffn_layer(mod, rng, d, d)
    c = np.array([1.5, -2.0, 0.25, -0.5, 3.0, -1.0, 0.75, -4.0])
    e = rand(rng, d, std=0.3)
    w["w_1"], w["b_1"] = np.zeros((d, d)), c
    w["w_2"], w["b_2"] = np.eye(d), e
    out = mod.layer_fwd(hm, hi, w, H, 0.5, nthreads=1)
    return bool(np.allclose(out, _ln_plain(x1n + np.maximum(c, 0) + e), rtol=0, atol=1e-12))


def ffn_pin_w1_then_w2(mod) -> bool:
    """d = d_ff, W_1 = diag(a) with a of both signs, W_2 = a cyclic shift S
    (column k of x S is column k-1 of x): x2 = x1n + ReLU(x1n diag(a)) S.
    Swapped products (ReLU(x1n S) diag(a)) differ: S is not diagonal and a
    is not constant."""
    rng = np.random.default_rng(23)
    d = 8
    w, hm, hi, x1n, H = _ffn_layer(mod, rng, d, d)
    a = np.array([1.0, -1.0, 2.0, 0.5, -3.0, 1.5, -0.25, 4.0])
    S = np.roll(np.eye(d), 1, axis=1)
    w["w_1"], w["b_1"] = np.diag(a), np.zeros(d)
    w["w_2"], w["b_2"] = S, np.zeros(d)
    want = _ln_plain(x1n + np.roll(np.maximum(x1n * a, 0), 1, axis=-1))
    swapped = _ln_plain(x1n + np.maximum(np.roll(x1n, 1, axis=-1), 0) * a)
    assert not np.allclose(want, swapped, atol=1e-3)
    out = mod.layer_fwd(hm, hi, w, H, 0.5, nthreads=1)
    return bool(np.allclose(out, want, rtol=0, atol=1e-12))


def test_ffn_relu_pair_gives_absolute_value():
    assert ffn_pin_absolute_value(oracle)


def test_ffn_bias_enters_before_the_relu():
    assert ffn_pin_bias_before_relu(oracle)


def test_ffn_applies_w1_then_w2():
    assert ffn_pin_w1_then_w2(oracle)


def test_ffn_random_weights_against_elementwise_loops():
    """Random weights (ReLU clipping part of the hidden units): every element
    of x2 against a plain loop over the hidden units."""
    rng = np.random.default_rng(24)
    d, dff = 8, 12
    w, hm, hi, x1n, H = _ffn_layer(oracle, rng, d, dff)
    B, L = x1n.shape[:2]
    x2 = np.zeros_like(x1n)
    clipped = 0
    for b in range(B):
        for i in range(L):
            for o_ in range(d):
                acc = x1n[b, i, o_] + w["b_2"][o_]
                for f in range(dff):
                    pre = w["b_1"][f] + sum(x1n[b, i, k] * w["w_1"][k, f] for k in range(d))
                    clipped += pre < 0
                    acc += max(pre, 0.0) * w["w_2"][f, o_]
                x2[b, i, o_] = acc
    assert clipped > 0
    out = oracle.layer_fwd(hm, hi, w, H, 0.5, nthreads=1)
    assert np.allclose(out, _ln_plain(x2), rtol=0, atol=1e-11)
