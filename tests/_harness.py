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


from long_context_lm_rel_gb300.calls import place_kv, ring_rows  # noqa: E402,F401


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


def AttnCall(*args, **kw):
    """The package's AttnCall with the test side's bit-exact device copies."""
    from long_context_lm_rel_gb300.calls import AttnCall as _AttnCall
    kw.setdefault("to_dev", to_dev)
    return _AttnCall(*args, **kw)
