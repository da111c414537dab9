"""Test-side plumbing between the seeded inputs, the oracle and the C ABI.

Host logic only: building device tensors from generator values, placing the
logical memory into ring rows, unrotating ring-layout outputs for the
oracle's logical layout, and the parity tolerances.

Tolerances (float32 path, 1e-5; bf16 path, 1e-2 * max|ref| and mean 1e-3)
are the ones the task fixes for this path.
"""
from __future__ import annotations

import numpy as np

import rxl_inputs as gen

F32_MAX_ABS = 1e-5
BF16_REL_MAX = 1e-2
BF16_MEAN = 1e-3


def torch_dtype(dtype):
    import torch
    return torch.float32 if dtype == "f32" else torch.bfloat16


def rxl_dtype(dtype):
    import long_context_lm_rel_gb300 as rxl
    return rxl.RXL_DTYPE_F32 if dtype == "f32" else rxl.RXL_DTYPE_BF16


def to_dev(x: np.ndarray, dtype: str, device="cuda"):
    """Device tensor holding exactly the generator's storage values."""
    import torch
    bits = gen.to_storage_bits(x, dtype)
    if dtype == "f32":
        return torch.from_numpy(bits.copy()).to(device)
    return torch.from_numpy(bits.view(np.int16).copy()).to(device).view(torch.bfloat16)


def to_host(t) -> np.ndarray:
    import torch
    return t.detach().float().cpu().numpy().astype(np.float64) if t.dtype != torch.float32 \
        else t.detach().cpu().numpy().astype(np.float64)


def ring_rows(cap: int, head: int, m: int) -> np.ndarray:
    """Physical ring row of each logical memory row t = 0..m-1."""
    return (head + np.arange(m)) % cap if m else np.zeros(0, dtype=np.int64)


def place_kv(mem: np.ndarray, cur: np.ndarray, cap: int, head: int, fill=0.0) -> np.ndarray:
    """Physical [B,H,cap+L,dh] K or V: logical memory rows into the ring at
    head, current rows after the ring. Unused ring rows get `fill`."""
    B, H, m, dh = mem.shape
    L = cur.shape[2]
    out = np.full((B, H, cap + L, dh), fill, dtype=np.float32)
    if m:
        out[:, :, ring_rows(cap, head, m)] = mem
    out[:, :, cap:] = cur
    return out


def logical_kv(phys: np.ndarray, cap: int, head: int, m: int) -> np.ndarray:
    """Inverse of place_kv on an output: [.., m+L, dh] in logical order."""
    return np.concatenate([phys[:, :, ring_rows(cap, head, m)], phys[:, :, cap:]], axis=2)


def assert_no_device_error():
    """No tensor-core kernel gave up on a bounded wait since the last check."""
    import long_context_lm_rel_gb300 as rxl
    flags = rxl.lib().rxl_device_error_flags()
    assert flags == 0, f"device-side wait timeout flags: {flags}"


def assert_close(name: str, got: np.ndarray, ref: np.ndarray, dtype: str, extra=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values {extra}"
    err = np.abs(got - ref)
    if dtype == "f32":
        assert err.max() <= F32_MAX_ABS, f"{name}: max abs err {err.max():.3e} > 1e-5 {extra}"
    else:
        bound = BF16_REL_MAX * max(np.abs(ref).max(), 1e-30)
        assert err.max() <= bound, f"{name}: max abs err {err.max():.3e} > {bound:.3e} {extra}"
        assert err.mean() <= BF16_MEAN, f"{name}: mean abs err {err.mean():.3e} > 1e-3 {extra}"
    return float(err.max())


class AttnCall:
    """Device buffers and one fwd (+bwd) call through the C ABI."""

    def __init__(self, q, k_phys, v_phys, r, u, vb, *, cap, m, head, dtype, scale):
        import torch
        import long_context_lm_rel_gb300 as rxl
        self.torch = torch
        self.rxl = rxl
        B, H, L, dh = q.shape
        self.shape = (B, H, L, dh)
        self.dtype = dtype
        self.cap, self.m, self.head = cap, m, head
        self.desc = rxl.make_desc(B, H, L, cap, m, head, scale, rxl_dtype(dtype))
        self.q, self.k, self.v = to_dev(q, dtype), to_dev(k_phys, dtype), to_dev(v_phys, dtype)
        rr = np.zeros((H, cap + L, dh), dtype=np.float32)
        rr[:, :min(r.shape[1], cap + L)] = r[:, :cap + L]
        self.r, self.u, self.vb = to_dev(rr, dtype), to_dev(u, dtype), to_dev(vb, dtype)
        td = torch_dtype(dtype)
        self.o = torch.empty((B, H, L, dh), device="cuda", dtype=td)
        self.lse = torch.empty((B, H, L), device="cuda", dtype=torch.float32)

    def fwd(self, stream=None):
        self.rxl.rxl_attn_fwd(self.desc, self.q, self.k, self.v, self.r, self.u, self.vb, self.o,
                              self.lse, stream)
        return self

    def fwd_ex(self, stream=None):
        """Forward of the training pair: also keeps the low part of O."""
        if not hasattr(self, "o_lo"):
            self.o_lo = self.torch.empty_like(self.o)
        self.rxl.rxl_attn_fwd_ex(self.desc, self.q, self.k, self.v, self.r, self.u, self.vb, self.o,
                                 self.o_lo, self.lse, stream)
        return self

    def bwd_ex(self, stream=None):
        self.rxl.rxl_attn_bwd_ex(self.desc, self.q, self.k, self.v, self.r, self.u, self.vb, self.o,
                                 self.o_lo, self.lse, self.do, self.dq, self.dk, self.dv, self.dr,
                                 self.du, self.dvb, self.ws, self.ws_bytes, stream)
        return self

    def alloc_bwd(self, dout):
        torch = self.torch
        B, H, L, dh = self.shape
        td = torch_dtype(self.dtype)
        self.do = to_dev(dout, self.dtype)
        self.dq = torch.empty((B, H, L, dh), device="cuda", dtype=td)
        self.dk = torch.empty_like(self.k)
        self.dv = torch.empty_like(self.v)
        self.dr = torch.empty((H, self.cap + L, dh), device="cuda", dtype=torch.float32)
        self.du = torch.empty((H, dh), device="cuda", dtype=torch.float32)
        self.dvb = torch.empty((H, dh), device="cuda", dtype=torch.float32)
        self.ws_bytes = self.rxl.rxl_attn_bwd_workspace_bytes(self.desc)
        self.ws = torch.empty(max(self.ws_bytes, 16), device="cuda", dtype=torch.uint8)
        return self

    def bwd(self, stream=None):
        self.rxl.rxl_attn_bwd(self.desc, self.q, self.k, self.v, self.r, self.u, self.vb, self.o,
                              self.lse, self.do, self.dq, self.dk, self.dv, self.dr, self.du,
                              self.dvb, self.ws, self.ws_bytes, stream)
        return self

    # per-row document reset: mem_visible [B] int32 on the device
    def fwd_reset(self, mem_visible, keep_low=True, stream=None):
        self.mvis = self.torch.tensor(np.asarray(mem_visible, dtype=np.int32), device="cuda")
        self.o_lo = self.torch.empty_like(self.o) if keep_low else None
        self.rxl.rxl_attn_fwd_reset(self.desc, self.mvis, self.q, self.k, self.v, self.r, self.u,
                                    self.vb, self.o, self.o_lo, self.lse, stream)
        return self

    def bwd_reset(self, stream=None):
        self.rxl.rxl_attn_bwd_reset(self.desc, self.mvis, self.q, self.k, self.v, self.r, self.u,
                                    self.vb, self.o, self.o_lo, self.lse, self.do, self.dq, self.dk,
                                    self.dv, self.dr, self.du, self.dvb, self.ws, self.ws_bytes,
                                    stream)
        return self
