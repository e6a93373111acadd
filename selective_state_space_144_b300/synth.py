"""Seeded synthetic inputs for the selective scan and the decode step.

This module holds no arithmetic of the method: it only draws random numbers
and rounds them to the storage type.  Both sides of every comparison (the
CUDA path and the fp64 oracle) consume exactly the arrays made here.

Recipe (the workloads' stated distributions):
  u, z, B, C ~ N(0, 1) iid; dt_raw ~ N(0, 0.5) (standard deviation 0.5);
  dt_bias[d] = log(expm1(v_d)), v_d ~ U[1e-3, 1e-1]  (so the step size at
  dt_raw = 0 lies in [1e-3, 1e-1]); A[d, n] = -(n + 1); D = 1, or
  D ~ N(1, 0.1) for the 2.8B-like layer.  Generator: numpy PCG64.  Draw
  order: u, z, B, C, dt_raw, dt_bias, then D when it is random.  Normals are
  drawn in float32 and, for bf16 workloads, rounded to bf16
  round-to-nearest-even; the float32 arrays returned hold exactly the
  rounded values.  The decode workload draws its initial state first, from
  its own stream, and every step's inputs from a per-step stream.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

# The five workloads, by what they are.
WORKLOADS = {
    "tiny_f32": dict(batch=1, L=64, d_inner=8, d_state=4, dtype="f32",
                     D="ones", seed=0),
    "mamba130m_layer": dict(batch=8, L=2048, d_inner=1536, d_state=16,
                            dtype="bf16", D="ones", seed=1),
    "long_seq_64k": dict(batch=1, L=65536, d_inner=2048, d_state=16,
                         dtype="bf16", D="ones", seed=2),
    "mamba2p8b_layer": dict(batch=4, L=4096, d_inner=5120, d_state=16,
                            dtype="bf16", D="normal", seed=3),
    "decode_256x5120": dict(batch=256, d_inner=5120, d_state=16, steps=1000,
                            dtype="bf16", D="ones", seed=4),
}


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round-to-nearest-even."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (b >> np.uint32(16)) & np.uint32(1)
    return ((b + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def bf16_value(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> the float32 values they encode."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32)
            << np.uint32(16)).view(np.float32)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """float32 values rounded to the nearest bf16 (ties to even), as float32."""
    return bf16_value(bf16_bits(x))


def _store(x: np.ndarray, dtype: str) -> np.ndarray:
    x = np.asarray(x, dtype=np.float32)
    return round_bf16(x) if dtype == "bf16" else x


@dataclass
class ScanInputs:
    """One batch of scan inputs.  Arrays are float32 holding exact values of
    the storage type `dtype` ("f32" or "bf16"); A, D, dt_bias are fp32."""
    u: np.ndarray
    dt_raw: np.ndarray
    A: np.ndarray
    B: np.ndarray
    C: np.ndarray
    D: np.ndarray | None
    z: np.ndarray | None
    dt_bias: np.ndarray | None
    dtype: str
    shape: tuple = field(default=())


def scan_inputs(batch: int, L: int, d_inner: int, d_state: int, *,
                dtype: str = "bf16", seed: int = 0, D: str = "ones",
                dt_std: float = 0.5, A_kind: str = "range",
                with_z: bool = True, with_D: bool = True,
                with_bias: bool = True) -> ScanInputs:
    """Draw scan inputs with the workloads' distributions.

    A_kind: "range" gives A[d, n] = -(n + 1); "random" gives A drawn from
    -U[0.5, 4] independently per (d, n) (used by checks that must see a
    channel-dependent A).
    """
    rng = np.random.default_rng(seed)
    f32 = np.float32
    u = _store(rng.standard_normal((batch, L, d_inner), dtype=f32), dtype)
    z = _store(rng.standard_normal((batch, L, d_inner), dtype=f32), dtype)
    B = _store(rng.standard_normal((batch, L, d_state), dtype=f32), dtype)
    C = _store(rng.standard_normal((batch, L, d_state), dtype=f32), dtype)
    dt_raw = _store(rng.standard_normal((batch, L, d_inner), dtype=f32)
                    * f32(dt_std), dtype)
    v = rng.uniform(1e-3, 1e-1, size=d_inner)
    dt_bias = np.log(np.expm1(v)).astype(f32)
    if D == "normal":
        Dv = (1.0 + 0.1 * rng.standard_normal(d_inner)).astype(f32)
    else:
        Dv = np.ones(d_inner, dtype=f32)
    if A_kind == "random":
        A = (-rng.uniform(0.5, 4.0, size=(d_inner, d_state))).astype(f32)
    else:
        A = np.tile(-np.arange(1, d_state + 1, dtype=f32), (d_inner, 1))
    return ScanInputs(u=u, dt_raw=dt_raw, A=A, B=B, C=C,
                      D=Dv if with_D else None, z=z if with_z else None,
                      dt_bias=dt_bias if with_bias else None, dtype=dtype,
                      shape=(batch, L, d_inner, d_state))


def workload_inputs(name: str, **overrides) -> ScanInputs:
    """Scan inputs of one named workload (sizes may be overridden)."""
    w = dict(WORKLOADS[name])
    w.update(overrides)
    return scan_inputs(w["batch"], w["L"], w["d_inner"], w["d_state"],
                       dtype=w["dtype"], seed=w["seed"], D=w["D"])


@dataclass
class DecodeParams:
    state0: np.ndarray     # (batch, d_inner, d_state) fp32
    A: np.ndarray          # (d_inner, d_state) fp32
    D: np.ndarray          # (d_inner,) fp32
    dt_bias: np.ndarray    # (d_inner,) fp32
    dtype: str


@dataclass
class DecodeStep:
    u: np.ndarray          # (batch, d_inner)
    dt_raw: np.ndarray
    z: np.ndarray
    B: np.ndarray          # (batch, d_state)
    C: np.ndarray


def decode_params(batch: int, d_inner: int, d_state: int, *, seed: int = 4,
                  dtype: str = "bf16") -> DecodeParams:
    """Initial state ~ N(0, 1) (drawn first) and the fixed parameters."""
    rng = np.random.default_rng([seed, 2**31 - 1])
    f32 = np.float32
    state0 = rng.standard_normal((batch, d_inner, d_state), dtype=f32)
    v = rng.uniform(1e-3, 1e-1, size=d_inner)
    dt_bias = np.log(np.expm1(v)).astype(f32)
    A = np.tile(-np.arange(1, d_state + 1, dtype=f32), (d_inner, 1))
    D = np.ones(d_inner, dtype=f32)
    return DecodeParams(state0=state0, A=A, D=D, dt_bias=dt_bias, dtype=dtype)


def decode_step(batch: int, d_inner: int, d_state: int, step: int, *,
                seed: int = 4, dtype: str = "bf16") -> DecodeStep:
    """The inputs of decode step `step` (its own PCG64 stream)."""
    rng = np.random.default_rng([seed, step])
    f32 = np.float32
    u = _store(rng.standard_normal((batch, d_inner), dtype=f32), dtype)
    z = _store(rng.standard_normal((batch, d_inner), dtype=f32), dtype)
    B = _store(rng.standard_normal((batch, d_state), dtype=f32), dtype)
    C = _store(rng.standard_normal((batch, d_state), dtype=f32), dtype)
    dt_raw = _store(rng.standard_normal((batch, d_inner), dtype=f32)
                    * f32(0.5), dtype)
    return DecodeStep(u=u, dt_raw=dt_raw, z=z, B=B, C=C)
