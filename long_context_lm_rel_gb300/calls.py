"""Device buffers for one attention call and the calls themselves.

A convenience layer over the binding for programs that start from host
arrays (the benchmark, the smoke check, the tests): it places the logical
memory into the ring rows of K/V, copies every input to the device once and
keeps the output, gradient and workspace buffers of the call. Every call
goes through the C ABI; nothing here computes anything.

Layout (include/rxl.h): K/V [B, H, cap + L, dh] with logical memory row t
at physical row (head + t) mod cap and the current rows at cap .. cap+L-1.
"""
from __future__ import annotations

import numpy as np

from . import (RXL_DTYPE_BF16, RXL_DTYPE_F32, make_desc, rxl_attn_bwd, rxl_attn_bwd_ex,
               rxl_attn_bwd_reset, rxl_attn_bwd_workspace_bytes, rxl_attn_fwd, rxl_attn_fwd_ex,
               rxl_attn_fwd_reset)


def torch_dtype(dtype: str):
    import torch
    return torch.float32 if dtype == "f32" else torch.bfloat16


def rxl_dtype(dtype: str) -> int:
    return RXL_DTYPE_F32 if dtype == "f32" else RXL_DTYPE_BF16


def to_device(x: np.ndarray, dtype: str, device="cuda"):
    """Device tensor of x in the call's dtype. For bf16 the values must already
    be bf16 numbers (the conversion is then exact); NaN stays NaN."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(device=device, dtype=torch_dtype(dtype))


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


class AttnCall:
    """Device buffers and one fwd (+bwd) call through the C ABI."""

    def __init__(self, q, k_phys, v_phys, r, u, vb, *, cap, m, head, dtype, scale, to_dev=to_device):
        import torch
        self.torch = torch
        B, H, L, dh = q.shape
        self.shape = (B, H, L, dh)
        self.dtype = dtype
        self.cap, self.m, self.head = cap, m, head
        self._to_dev = to_dev
        self.desc = make_desc(B, H, L, cap, m, head, scale, rxl_dtype(dtype))
        self.q, self.k, self.v = to_dev(q, dtype), to_dev(k_phys, dtype), to_dev(v_phys, dtype)
        rr = np.zeros((H, cap + L, dh), dtype=np.float32)
        rr[:, :min(r.shape[1], cap + L)] = r[:, :cap + L]
        self.r, self.u, self.vb = to_dev(rr, dtype), to_dev(u, dtype), to_dev(vb, dtype)
        td = torch_dtype(dtype)
        self.o = torch.empty((B, H, L, dh), device="cuda", dtype=td)
        self.lse = torch.empty((B, H, L), device="cuda", dtype=torch.float32)

    def fwd(self, stream=None):
        rxl_attn_fwd(self.desc, self.q, self.k, self.v, self.r, self.u, self.vb, self.o, self.lse, stream)
        return self

    def fwd_ex(self, stream=None):
        """Forward of the training pair: also keeps the low part of O."""
        if getattr(self, "o_lo", None) is None:
            self.o_lo = self.torch.empty_like(self.o)
        rxl_attn_fwd_ex(self.desc, self.q, self.k, self.v, self.r, self.u, self.vb, self.o, self.o_lo,
                        self.lse, stream)
        return self

    def alloc_bwd(self, dout):
        torch = self.torch
        B, H, L, dh = self.shape
        td = torch_dtype(self.dtype)
        self.do = self._to_dev(dout, self.dtype)
        self.dq = torch.empty((B, H, L, dh), device="cuda", dtype=td)
        self.dk = torch.empty_like(self.k)
        self.dv = torch.empty_like(self.v)
        self.dr = torch.empty((H, self.cap + L, dh), device="cuda", dtype=torch.float32)
        self.du = torch.empty((H, dh), device="cuda", dtype=torch.float32)
        self.dvb = torch.empty((H, dh), device="cuda", dtype=torch.float32)
        self.ws_bytes = rxl_attn_bwd_workspace_bytes(self.desc)
        self.ws = torch.empty(max(self.ws_bytes, 16), device="cuda", dtype=torch.uint8)
        return self

    def bwd(self, stream=None):
        rxl_attn_bwd(self.desc, self.q, self.k, self.v, self.r, self.u, self.vb, self.o, self.lse, self.do,
                     self.dq, self.dk, self.dv, self.dr, self.du, self.dvb, self.ws, self.ws_bytes, stream)
        return self

    def bwd_ex(self, stream=None):
        rxl_attn_bwd_ex(self.desc, self.q, self.k, self.v, self.r, self.u, self.vb, self.o, self.o_lo,
                        self.lse, self.do, self.dq, self.dk, self.dv, self.dr, self.du, self.dvb, self.ws,
                        self.ws_bytes, stream)
        return self

    # per-row document reset: mem_visible [B] int32 on the device
    def fwd_reset(self, mem_visible, keep_low=True, stream=None):
        self.mvis = self.torch.tensor(np.asarray(mem_visible, dtype=np.int32), device="cuda")
        self.o_lo = self.torch.empty_like(self.o) if keep_low else None
        rxl_attn_fwd_reset(self.desc, self.mvis, self.q, self.k, self.v, self.r, self.u, self.vb, self.o,
                           self.o_lo, self.lse, stream)
        return self

    def bwd_reset(self, stream=None):
        rxl_attn_bwd_reset(self.desc, self.mvis, self.q, self.k, self.v, self.r, self.u, self.vb, self.o,
                           self.o_lo, self.lse, self.do, self.dq, self.dk, self.dv, self.dr, self.du,
                           self.dvb, self.ws, self.ws_bytes, stream)
        return self
