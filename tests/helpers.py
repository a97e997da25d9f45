"""Shared test helpers: device upload of seeded inputs, the parity metric."""
from __future__ import annotations

import numpy as np

from selective_state_space_125_b300.workloads import bf16_bits


def parity_err(got, ref) -> float:
    """max_i |g_i - r_i| / max(|r_i|, rms(r)): relative error with an rms floor,
    so that outputs gated to ~0 do not divide by ~0."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    if ref.size == 0:
        return 0.0
    rms = float(np.sqrt(np.mean(ref * ref)))
    den = np.maximum(np.abs(ref), max(rms, 1e-300))
    return float(np.max(np.abs(got - ref) / den))


# Acceptance tolerances: max relative error for fp32 and bf16 inputs.
TOL = {"f32": 1e-4, "bf16": 2e-2}


def to_torch(x: np.ndarray, dtype: str, device):
    """float32 numpy array holding dtype-exact values -> torch tensor of that dtype."""
    import torch
    if dtype == "f32":
        return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(device)
    bits = bf16_bits(x)
    return torch.from_numpy(bits.view(np.int16)).to(device).view(torch.bfloat16)


def to_numpy(t) -> np.ndarray:
    import torch
    return t.detach().to(torch.float32).cpu().numpy()


def upload_scan(inp: dict, device, with_z=True, with_D=True, with_bias=True):
    dt = inp["dtype"]
    import torch
    f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(device)
    return dict(
        u=to_torch(inp["u"], dt, device), delta=to_torch(inp["delta"], dt, device),
        A_log=f32(inp["A_log"]), B=to_torch(inp["B"], dt, device), C=to_torch(inp["C"], dt, device),
        D=f32(inp["D"]) if with_D else None, z=to_torch(inp["z"], dt, device) if with_z else None,
        delta_bias=f32(inp["delta_bias"]) if with_bias else None)
