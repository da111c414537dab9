"""Float64 CPU oracle for relative-position memory attention.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU
baseline leg are the only callers. The CUDA library neither imports nor links
anything here, and nothing here imports the CUDA package.

* ``fwd`` / ``fwd_rows`` / ``logits`` / ``bwd``: the C loops of
  ``rxl_oracle.c`` (explicit (i, j) loops, direct R[i-j] lookup, allow(i,j)
  mask), called through ctypes on float64 copies of the inputs.
* ``tail_m``: the memory update of the Transformer-XL page ("Batched Tensor
  Contract", update_mems; eq. Tail_M in "Segment-Level Recurrence"):
  concatenate old memory and the new hidden states along the sequence axis and
  keep the last mem_len rows; mem_len == 0 keeps nothing.
* ``fullseq_fwd``: a second, independent forward over global stream positions
  (token t of segment s sees t' with s*L - M <= t' <= t), used to check that a
  rolling memory sees exactly the last M states.

Every function is pinned by a test in tests/test_oracle_pins.py against values
the pages print, closed forms, library routines or brute force.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rxl_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "librxl_oracle.so")
_lock = threading.Lock()
_lib = None


def build(src: str = _SRC, out: str = _LIB_PATH, extra_flags=()) -> str:
    """Compile the oracle with gcc (plain -O2, IEEE arithmetic, no fast-math)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-fno-fast-math",
           "-ffp-contract=off", *extra_flags, "-o", out, src, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def _needs_build() -> bool:
    return (not os.path.exists(_LIB_PATH)
            or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))


def load(path: str | None = None):
    """Load the oracle library (building it first if it is missing/stale)."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            if _needs_build():
                build()
            _lib = _bind(ctypes.CDLL(_LIB_PATH))
    return _lib


_D = ctypes.POINTER(ctypes.c_double)
_I = ctypes.POINTER(ctypes.c_int)


def _bind(lib):
    i, d, ll = ctypes.c_int, ctypes.c_double, ctypes.c_longlong
    lib.oracle_fwd.argtypes = [i, i, i, i, i, d, ll] + [_D] * 6 + [_D, _D, i]
    lib.oracle_fwd.restype = None
    lib.oracle_fwd_rows.argtypes = [i, i, i, i, i, d, ll] + [_D] * 6 + [i, _I, _D, _D, i]
    lib.oracle_fwd_rows.restype = None
    lib.oracle_logits.argtypes = [i, i, i, i, i, d, ll] + [_D] * 5 + [_D, i]
    lib.oracle_logits.restype = None
    lib.oracle_bwd.argtypes = [i, i, i, i, i, d, ll] + [_D] * 7 + [_D] * 6 + [i]
    lib.oracle_bwd.restype = ctypes.c_int
    lib.oracle_fwd_reset.argtypes = [i, i, i, i, i, d, ll] + [_D] * 6 + [_I, _D, _D, i]
    lib.oracle_fwd_reset.restype = None
    lib.oracle_bwd_reset.argtypes = [i, i, i, i, i, d, ll] + [_D] * 6 + [_I] + [_D] * 7 + [i]
    lib.oracle_bwd_reset.restype = ctypes.c_int
    return lib


def _f64(x):
    return np.ascontiguousarray(x, dtype=np.float64)


def _p(x):
    return x.ctypes.data_as(_D)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _shapes(q, k, r):
    B, H, L, dh = q.shape
    mL = k.shape[2]
    m = mL - L
    assert k.shape == (B, H, mL, dh) and r.shape[0] == H and r.shape[2] == dh
    assert r.shape[1] >= mL, "R needs one row per distance 0..m+L-1"
    return B, H, L, m, dh


def _r_rows(r, mL):
    return _f64(r[:, :mL, :])


def _mvis(mem_visible, B, m):
    """Per batch row: newest memory rows visible (document reset), int32 [B]."""
    a = np.ascontiguousarray(np.asarray(mem_visible, dtype=np.int32).reshape(B))
    assert ((a >= 0) & (a <= m)).all(), "mem_visible must lie in [0, m]"
    return a


def fwd(q, k, v, r, u, vb, scale, pos0=0, nthreads=None, lib=None, mem_visible=None):
    """O [B,H,L,dh] and LSE [B,H,L] (float64). k, v: [B,H,m+L,dh] in logical
    order (memory rows oldest first, then the current rows). mem_visible
    (optional, [B]): batch row b sees only its newest mem_visible[b] memory
    rows (per-row document reset)."""
    lib = lib or load()
    B, H, L, m, dh = _shapes(q, k, r)
    q, k, v, u, vb = map(_f64, (q, k, v, u, vb))
    r = _r_rows(r, m + L)
    o = np.zeros((B, H, L, dh))
    lse = np.zeros((B, H, L))
    if mem_visible is None:
        lib.oracle_fwd(B, H, L, m, dh, float(scale), int(pos0), _p(q), _p(k), _p(v), _p(r),
                       _p(u), _p(vb), _p(o), _p(lse), nthreads or default_threads())
    else:
        mv = _mvis(mem_visible, B, m)
        lib.oracle_fwd_reset(B, H, L, m, dh, float(scale), int(pos0), _p(q), _p(k), _p(v), _p(r),
                             _p(u), _p(vb), mv.ctypes.data_as(_I), _p(o), _p(lse),
                             nthreads or default_threads())
    return o, lse


def fwd_rows(q, k, v, r, u, vb, scale, sel, pos0=0, nthreads=None, lib=None):
    """Forward of selected (b, h, i) rows: returns O [n,dh], LSE [n]."""
    lib = lib or load()
    B, H, L, m, dh = _shapes(q, k, r)
    q, k, v, u, vb = map(_f64, (q, k, v, u, vb))
    r = _r_rows(r, m + L)
    sel = np.ascontiguousarray(np.asarray(sel, dtype=np.int32).reshape(-1, 3))
    n = sel.shape[0]
    o = np.zeros((n, dh))
    lse = np.zeros(n)
    lib.oracle_fwd_rows(B, H, L, m, dh, float(scale), int(pos0), _p(q), _p(k), _p(v), _p(r),
                        _p(u), _p(vb), n, sel.ctypes.data_as(_I), _p(o), _p(lse),
                        nthreads or default_threads())
    return o, lse


def logits(q, k, r, u, vb, scale, pos0=0, nthreads=None, lib=None):
    """Scaled logits s*A [B,H,L,m+L]; -inf where allow(i,j) = 0."""
    lib = lib or load()
    B, H, L, m, dh = _shapes(q, k, r)
    q, k, u, vb = map(_f64, (q, k, u, vb))
    r = _r_rows(r, m + L)
    z = np.zeros((B, H, L, m + L))
    lib.oracle_logits(B, H, L, m, dh, float(scale), int(pos0), _p(q), _p(k), _p(r), _p(u),
                      _p(vb), _p(z), nthreads or default_threads())
    return z


def bwd(q, k, v, r, u, vb, dout, scale, pos0=0, nthreads=None, lib=None, mem_visible=None):
    """Gradients of sum(O * dout): dict with dq [B,H,L,dh], dk, dv [B,H,m+L,dh]
    (logical order), dr [H,m+L,dh], du, dvb [H,dh]; all float64. mem_visible
    as in fwd."""
    lib = lib or load()
    B, H, L, m, dh = _shapes(q, k, r)
    q, k, v, u, vb, dout = map(_f64, (q, k, v, u, vb, dout))
    r = _r_rows(r, m + L)
    out = {
        "dq": np.zeros((B, H, L, dh)), "dk": np.zeros((B, H, m + L, dh)),
        "dv": np.zeros((B, H, m + L, dh)), "dr": np.zeros((H, m + L, dh)),
        "du": np.zeros((H, dh)), "dvb": np.zeros((H, dh)),
    }
    outs = (_p(out["dq"]), _p(out["dk"]), _p(out["dv"]), _p(out["dr"]), _p(out["du"]), _p(out["dvb"]))
    if mem_visible is None:
        rc = lib.oracle_bwd(B, H, L, m, dh, float(scale), int(pos0), _p(q), _p(k), _p(v), _p(r),
                            _p(u), _p(vb), _p(dout), *outs, nthreads or default_threads())
    else:
        mv = _mvis(mem_visible, B, m)
        rc = lib.oracle_bwd_reset(B, H, L, m, dh, float(scale), int(pos0), _p(q), _p(k), _p(v),
                                  _p(r), _p(u), _p(vb), mv.ctypes.data_as(_I), _p(dout), *outs,
                                  nthreads or default_threads())
    if rc != 0:
        raise MemoryError("oracle_bwd: allocation failed")
    return out


def proj(h_mem, h_cur, w_q, w_k, w_v, H):
    """The projection front-end ("Segment-Level Recurrence": Q = H W^Q,
    K = [SG(M); H] W^K, V = [SG(M); H] W^V; "Batched Tensor Contract" for
    the shapes). h_mem [B,m,d] is the layer's hidden-state memory in logical
    order (oldest first), h_cur [B,L,d]; w_* [d, H*dh]; projected column
    h*dh + e is element e of head h. Returns q [B,H,L,dh] and k, v
    [B,H,m+L,dh] (logical order), float64; a matrix product is the step."""
    h_mem, h_cur = _f64(h_mem), _f64(h_cur)
    w_q, w_k, w_v = _f64(w_q), _f64(w_k), _f64(w_v)
    B, L, d = h_cur.shape
    dh = w_q.shape[1] // H
    h_t = np.concatenate([h_mem, h_cur], axis=1)           # H~ = [SG(M); H]
    split = lambda x: x.reshape(B, x.shape[1], H, dh).transpose(0, 2, 1, 3).copy()
    return split(h_cur @ w_q), split(h_t @ w_k), split(h_t @ w_v)


def layer_norm(x, gamma, beta, eps=1e-5):
    """(x - mean) / sqrt(var + eps) * gamma + beta over the last axis, with the
    biased variance (float64)."""
    x = _f64(x)
    mu = x.mean(-1, keepdims=True)
    var = ((x - mu) ** 2).mean(-1, keepdims=True)
    return (x - mu) / np.sqrt(var + eps) * _f64(gamma) + _f64(beta)


def layer_fwd(h_mem, h_in, w, H, scale, eps=1e-5, nthreads=None):
    """One evaluation layer (float64): the attention sublayer of "Segment-Level
    Recurrence" (Q = H W^Q, K/V = [SG(M); H] W^{K,V}, the relative-position
    attention) and a feed-forward sublayer, in the post-norm arrangement
    (the pages leave the layer's remaining steps open):
        x1 = h_in + Attn . W_O,  x1n = LN1(x1),
        h_out = LN2(x1n + ReLU(x1n W_1 + b_1) W_2 + b_2).
    h_mem [B,m,d] logical order, h_in [B,L,d]; w: dict of the weights named as
    the fields of rxl_layer_weights. Returns h_out [B,L,d]."""
    q, k, v = proj(h_mem, h_in, w["w_q"], w["w_k"], w["w_v"], H)
    o, _ = fwd(q, k, v, w["r"], w["u"], w["vbias"], scale, nthreads=nthreads)
    B, _, L, dh = o.shape
    om = o.transpose(0, 2, 1, 3).reshape(B, L, H * dh)      # heads merged: column h*dh + e
    x1 = _f64(h_in) + om @ _f64(w["w_o"])
    x1n = layer_norm(x1, w["ln1_gamma"], w["ln1_beta"], eps)
    z = np.maximum(x1n @ _f64(w["w_1"]) + _f64(w["b_1"]), 0.0)
    x2 = x1n + z @ _f64(w["w_2"]) + _f64(w["b_2"])
    return layer_norm(x2, w["ln2_gamma"], w["ln2_beta"], eps)


def tail_m(mem: np.ndarray, hids: np.ndarray, mem_len: int) -> np.ndarray:
    """Memory update along axis -2 (sequence axis, d innermost):
    cat([mem, hids]) then keep the last mem_len rows; mem_len == 0 keeps an
    empty memory (Transformer-XL page, update_mems / eq. Tail_M)."""
    if mem_len == 0:
        return hids[..., :0, :].copy()
    cat = np.concatenate([mem, hids], axis=-2)
    return cat[..., -mem_len:, :].copy()


def fullseq_fwd(q, k, v, r, u, vb, scale, L, M):
    """Independent forward over one global stream (single head, float64,
    explicit Python loops; tiny sizes only).

    q, k, v: [T, dh] over global positions 0..T-1, split into segments of L.
    Token t of segment s = t // L sees key t' iff s*L - M <= t' <= t and
    t' >= 0; the score uses the distance t - t'. Returns O [T, dh]."""
    q, k, v, r, u, vb = map(_f64, (q, k, v, r, u, vb))
    T, dh = q.shape
    o = np.zeros((T, dh))
    for t in range(T):
        start = (t // L) * L
        keys = [tp for tp in range(max(0, start - M), t + 1)]
        z = []
        for tp in keys:
            a = 0.0
            for c in range(dh):
                a += (q[t, c] + u[c]) * k[tp, c] + (q[t, c] + vb[c]) * r[t - tp, c]
            z.append(scale * a)
        mx = max(z)
        w = [np.exp(x - mx) for x in z]
        s = sum(w)
        for tp, wt in zip(keys, w):
            o[t] += (wt / s) * v[tp]
    return o
