"""The pins must catch plausible mistakes in the oracle.

Each case copies the oracle's C source, plants one mistake (a dropped term, a
wrong sign or index, a wrong operand, a mask off by one), builds the copy
into a temporary library and runs a compact battery of the pins against it.
The unmodified source must pass the battery; every mutant must fail it.
"""
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from tests import _golden
from tests.test_oracle_pins import make_txl_mask, reference_rel_ids, distance_probe, reset_vs_sliced

SRC = os.path.join(os.path.dirname(oracle.__file__), "rxl_oracle.c")

MUTANTS = {
    "drop_u": ("content += (qi[c] + u[c]) * kj[c];", "content += qi[c] * kj[c];"),
    "drop_v": ("position += (qi[c] + vb[c]) * rd[c];", "position += qi[c] * rd[c];"),
    "r_descending": ("const double *rd = P->r + ((size_t)h * mL + (size_t)d) * dh;",
                     "const double *rd = P->r + ((size_t)h * mL + (size_t)(mL - 1 - d)) * dh;"),
    "scale_content_only": ("return P->scale * (content + position);",
                           "return P->scale * content + position;"),
    "diagonal_masked": ("return pj <= pi;", "return pj < pi;"),
    "memory_masked": ("if (pj < pos0) return 1;", "if (pj < pos0) return 0;"),
    "dS_sign": ("P->scale * p * (dp - Di);", "P->scale * p * (Di - dp);"),
    "dv_without_P": ("dvj[c] += p * doi[c];", "dvj[c] += doi[c];"),
    "dk_wrong_bias": ("dkj[c] += dA * (qi[c] + u[c]);", "dkj[c] += dA * (qi[c] + vb[c]);"),
    "dr_wrong_bias": ("drd[c] += dA * (qi[c] + vb[c]);", "drd[c] += dA * (qi[c] + u[c]);"),
    "dq_content_only": ("dqi[c] += dA * (kj[c] + rd[c]);", "dqi[c] += dA * kj[c];"),
    "du_uses_r": ("du[c] += dA * kj[c];", "du[c] += dA * rd[c];"),
    "reset_keeps_oldest": ("if (P->mvis && j < 0 && j < -P->mvis[b]) return 0;",
                           "if (P->mvis && j < 0 && j >= P->mvis[b] - P->m) return 0;"),
    "reset_off_by_one": ("if (P->mvis && j < 0 && j < -P->mvis[b]) return 0;",
                         "if (P->mvis && j < 0 && j <= -P->mvis[b]) return 0;"),
}


def _build(tmp_path, name, edit):
    with open(SRC) as f:
        src = f.read()
    if edit is not None:
        old, new = edit
        assert src.count(old) >= 1, f"mutation anchor not found: {old}"
        src = src.replace(old, new)  # the same mistake everywhere it can occur
    path = tmp_path / f"{name}.c"
    path.write_text(src)
    lib = oracle.build(str(path), str(tmp_path / f"lib{name}.so"))
    return oracle.load(lib)


def battery(lib):
    """Returns the names of the pins that fail on this library."""
    failed = []
    rng = np.random.default_rng(123)
    R = lambda *s, std=1.0: rng.standard_normal(s) * std
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))

    # mask picture (M=3, L=4)
    want = _golden.mask_picture()
    L, m = 4, 3
    q = np.zeros((1, 1, L, 64)); k = np.zeros((1, 1, m + L, 64)); v = np.zeros((1, 1, m + L, 64))
    for c in range(m + L):
        v[0, 0, c, c] = 1.0
    o, _ = oracle.fwd(q, k, v, np.zeros((1, m + L, 64)), np.zeros((1, 64)), np.zeros((1, 64)),
                      0.125, nthreads=1, lib=lib)
    if not np.array_equal(o[0, 0, :, :m + L] > 0, want):
        failed.append("mask")

    # reduction to masked attention
    B, H, L, m, dh, s = 2, 2, 5, 6, 8, 0.3
    q, k, v = R(B, H, L, dh), R(B, H, m + L, dh), R(B, H, m + L, dh)
    o, _ = oracle.fwd(q, k, v, np.zeros((H, m + L, dh)), np.zeros((H, dh)), np.zeros((H, dh)), s,
                      nthreads=1, lib=lib)
    ref = F.scaled_dot_product_attention(t(q), t(k), t(v), attn_mask=make_txl_mask(L, m), scale=s)
    if not np.allclose(o, ref.numpy(), rtol=0, atol=1e-12):
        failed.append("sdpa")

    # u as a key bias
    u = R(H, dh)
    o, _ = oracle.fwd(q, k, v, np.zeros((H, m + L, dh)), u, np.zeros((H, dh)), s, nthreads=1, lib=lib)
    bias = s * np.einsum("hd,bhjd->bhj", u, k)[:, :, None, :]
    mask = t(np.broadcast_to(bias, (B, H, L, m + L)).copy()).masked_fill(~make_txl_mask(L, m), -math.inf)
    ref = F.scaled_dot_product_attention(t(q), t(k), t(v), attn_mask=mask, scale=s)
    if not np.allclose(o, ref.numpy(), rtol=0, atol=1e-12):
        failed.append("u_bias")

    # distance labels
    L, m, alpha, s2 = 4, 8, -2.0, 0.125
    qq, kk, r, uu, vb = distance_probe(L, m, alpha)
    vv = np.zeros((1, 1, m + L, 64))
    for c in range(m + L):
        vv[0, 0, c, c] = 1.0
    o, _ = oracle.fwd(qq, kk, vv, r, uu, vb, s2, nthreads=1, lib=lib)
    p = o[0, 0, :, :m + L]
    vis = make_txl_mask(L, m).numpy()
    with np.errstate(divide="ignore", invalid="ignore"):
        ids = np.log(p / p[np.arange(L), m + np.arange(L)][:, None]) / (s2 * alpha)
    if not np.allclose(ids[vis], reference_rel_ids(L, m).numpy()[vis], rtol=0, atol=1e-9):
        failed.append("rel_ids")

    # gradients: central differences on a sample of elements of every input
    B, H, L, m, dh, s = 1, 1, 4, 5, 8, 0.3
    x = dict(q=R(B, H, L, dh), k=R(B, H, m + L, dh), v=R(B, H, m + L, dh), r=R(H, m + L, dh),
             u=R(H, dh), vb=R(H, dh))
    do = R(B, H, L, dh)
    names = ["q", "k", "v", "r", "u", "vb"]
    g = oracle.bwd(*(x[n] for n in names), do, s, nthreads=1, lib=lib)
    gk = {"q": "dq", "k": "dk", "v": "dv", "r": "dr", "u": "du", "vb": "dvb"}

    def loss():
        o, _ = oracle.fwd(*(x[n] for n in names), s, nthreads=1, lib=lib)
        return float(np.sum(o * do))

    h = 1e-6
    for n in names:
        flat = x[n].reshape(-1)
        for e in range(0, flat.size, max(1, flat.size // 12)):
            keep = flat[e]
            flat[e] = keep + h; lp = loss()
            flat[e] = keep - h; lm = loss()
            flat[e] = keep
            fd = (lp - lm) / (2 * h)
            an = g[gk[n]].reshape(-1)[e]
            if abs(fd - an) > 1e-6 * max(1.0, np.max(np.abs(g[gk[n]]))):
                failed.append("grad_" + n)
                break

    # per-row document reset: each row equals the row alone with its newest memory
    if reset_vs_sliced((7, 0, 3), lib=lib):
        failed.append("reset")
    return failed


def test_unmodified_oracle_passes_battery(tmp_path):
    assert battery(_build(tmp_path, "control", None)) == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    failed = battery(_build(tmp_path, name, MUTANTS[name]))
    assert failed, f"mutant {name} slipped through every pin"


# ------------------------------------- the evaluation layer (Python oracle)
# The same idea for oracle.layer_fwd: a copy of the oracle package's source
# with one mistake in the feed-forward sublayer, loaded as its own module, must
# fail one of the feed-forward pins.

PY_SRC = oracle.__file__
LAYER_MUTANTS = {
    "ffn_no_relu": ("z = np.maximum(x1n @ _f64(w[\"w_1\"]) + _f64(w[\"b_1\"]), 0.0)",
                    "z = x1n @ _f64(w[\"w_1\"]) + _f64(w[\"b_1\"])"),
    "ffn_bias_after_relu": ("z = np.maximum(x1n @ _f64(w[\"w_1\"]) + _f64(w[\"b_1\"]), 0.0)",
                            "z = np.maximum(x1n @ _f64(w[\"w_1\"]), 0.0) + _f64(w[\"b_1\"])"),
    "ffn_w1_w2_swapped": ("z = np.maximum(x1n @ _f64(w[\"w_1\"]) + _f64(w[\"b_1\"]), 0.0)\n"
                          "    x2 = x1n + z @ _f64(w[\"w_2\"]) + _f64(w[\"b_2\"])",
                          "z = np.maximum(x1n @ _f64(w[\"w_2\"]) + _f64(w[\"b_1\"]), 0.0)\n"
                          "    x2 = x1n + z @ _f64(w[\"w_1\"]) + _f64(w[\"b_2\"])"),
    "ffn_relu_after_w2": ("z = np.maximum(x1n @ _f64(w[\"w_1\"]) + _f64(w[\"b_1\"]), 0.0)\n"
                          "    x2 = x1n + z @ _f64(w[\"w_2\"]) + _f64(w[\"b_2\"])",
                          "z = x1n @ _f64(w[\"w_1\"]) + _f64(w[\"b_1\"])\n"
                          "    x2 = x1n + np.maximum(z @ _f64(w[\"w_2\"]), 0.0) + _f64(w[\"b_2\"])"),
    "ffn_no_residual": ("x2 = x1n + z @ _f64(w[\"w_2\"]) + _f64(w[\"b_2\"])",
                        "x2 = z @ _f64(w[\"w_2\"]) + _f64(w[\"b_2\"])"),
}


def _py_oracle(tmp_path, name, edit):
    import importlib.util
    with open(PY_SRC) as f:
        src = f.read()
    if edit is not None:
        old, new = edit
        assert src.count(old) == 1, f"mutation anchor not found: {old}"
        src = src.replace(old, new)
    pkg = tmp_path / f"oracle_{name}"
    pkg.mkdir()
    (pkg / "__init__.py").write_text(src)
    spec = importlib.util.spec_from_file_location(f"oracle_{name}", pkg / "__init__.py")
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod._lib = oracle.load()  # the C part is unchanged: reuse the built library
    return mod


def layer_battery(mod):
    from tests.test_oracle_pins import ffn_pin_absolute_value, ffn_pin_bias_before_relu, ffn_pin_w1_then_w2
    pins = {"abs": ffn_pin_absolute_value, "bias": ffn_pin_bias_before_relu, "order": ffn_pin_w1_then_w2}
    failed = []
    for n, f in pins.items():
        try:
            ok = f(mod)
        except ValueError:  # shapes that no longer fit (d != d_ff) also expose the mistake
            ok = False
        if not ok:
            failed.append(n)
    return failed


def test_unmodified_layer_passes_ffn_pins(tmp_path):
    assert layer_battery(_py_oracle(tmp_path, "control", None)) == []


@pytest.mark.parametrize("name", sorted(LAYER_MUTANTS))
def test_layer_mutant_is_caught(tmp_path, name):
    failed = layer_battery(_py_oracle(tmp_path, name, LAYER_MUTANTS[name]))
    assert failed, f"layer mutant {name} slipped through every feed-forward pin"
