"""Shared test helpers: device copies of the seeded inputs and the parity
metric.  Holds none of the method's arithmetic."""
from __future__ import annotations

import numpy as np

from selective_state_space_144_b300 import synth

# Tolerances (rel-L2 over a whole tensor): fp32 storage, and bf16 storage
# with an fp32 state compared against the oracle's output rounded to bf16.
TOL = {"f32": 1e-5, "bf16": 2e-3}


def rel_l2(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = float(np.linalg.norm(ref.ravel()))
    num = float(np.linalg.norm((got - ref).ravel()))
    return num / den if den > 0 else num


def as_stored(y64: np.ndarray, dtype: str) -> np.ndarray:
    """The oracle's fp64 output as the kernel must store it: bf16 outputs are
    rounded to nearest even (through fp32); fp32 outputs are kept in fp64."""
    if dtype == "bf16":
        return synth.round_bf16(np.asarray(y64, dtype=np.float32)).astype(np.float64)
    return np.asarray(y64, dtype=np.float64)


def to_device(arr, dtype: str, device="cuda"):
    """numpy float32 (exact values of `dtype`) -> torch tensor of `dtype`."""
    import torch
    if arr is None:
        return None
    if dtype == "bf16":
        bits = synth.bf16_bits(arr).view(np.int16)
        return torch.from_numpy(bits.copy()).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(arr, dtype=np.float32)).to(device)


def from_device(t) -> np.ndarray:
    import torch
    return t.detach().to(torch.float32).cpu().numpy().astype(np.float64)


def scan_device_args(x: synth.ScanInputs, device="cuda"):
    """Device tensors of a ScanInputs: the six typed arrays in x.dtype and
    A, D, dt_bias in fp32."""
    d = x.dtype
    return dict(
        u=to_device(x.u, d, device), dt=to_device(x.dt_raw, d, device),
        A=to_device(x.A, "f32", device), B=to_device(x.B, d, device),
        C=to_device(x.C, d, device), D=to_device(x.D, "f32", device),
        z=to_device(x.z, d, device), dt_bias=to_device(x.dt_bias, "f32", device))
