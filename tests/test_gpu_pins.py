"""The oracle's closed-form pins rerun on the GPU path (fp32, rel-L2 1e-5):
the LTI convolution, the geometric series and the dt limits are checked
against their closed forms directly, not through the oracle."""
import math

import numpy as np
import pytest

import selective_state_space_144_b300 as msc
from selective_state_space_144_b300 import synth
from tests.helpers import from_device, rel_l2, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _gpu(u, dt_raw, A, B, C, D=None, z=None, dt_bias=None, chunks=0):
    f = lambda a: to_device(None if a is None else np.asarray(a, np.float32), "f32")
    msc.tuning_set("scan_chunks", chunks)
    try:
        out, last = msc.selective_scan_fwd(f(u), f(dt_raw), f(A), f(B), f(C),
                                           f(D), f(z), f(dt_bias))
        torch.cuda.synchronize()
    finally:
        msc.tuning_set("scan_chunks", 0)
    return from_device(out), from_device(last)


def _softplus(x):
    return np.logaddexp(0.0, np.asarray(x, np.float64))


@pytest.mark.parametrize("chunks", [1, 4])
def test_lti_convolution(chunks):
    batch, L, d_inner, N = 2, 256, 3, 4
    rng = np.random.default_rng(7)
    x = synth.scan_inputs(batch, L, d_inner, N, dtype="f32", seed=12,
                          D="normal", A_kind="random", with_z=False)
    raw = rng.normal(0.0, 0.5, size=d_inner).astype(np.float32)
    dt_raw = np.broadcast_to(raw[None, None, :], (batch, L, d_inner))
    Bc = rng.standard_normal((batch, N)).astype(np.float32)
    Cc = rng.standard_normal((batch, N)).astype(np.float32)
    B = np.broadcast_to(Bc[:, None, :], (batch, L, N))
    C = np.broadcast_to(Cc[:, None, :], (batch, L, N))
    y, _ = _gpu(x.u, dt_raw, x.A, B, C, x.D, None, x.dt_bias, chunks)
    A = x.A.astype(np.float64)
    dt = _softplus(raw.astype(np.float64) + x.dt_bias)
    k = np.arange(L, dtype=np.float64)
    y_ref = np.zeros((batch, L, d_inner))
    for b in range(batch):
        for d in range(d_inner):
            K = (Cc[b][None, :] * np.exp(k[:, None] * dt[d] * A[d][None, :])
                 * dt[d] * Bc[b][None, :]).sum(axis=1)
            ud = x.u[b, :, d].astype(np.float64)
            y_ref[b, :, d] = np.convolve(K, ud)[:L] + x.D[d] * ud
    assert rel_l2(y, y_ref) <= 1e-5


def test_geometric_series():
    L = 300
    A = np.array([[-0.7], [-2.0]], np.float32)
    raw = np.array([0.3, -1.1], np.float32)
    Dv = np.array([0.25, -1.5], np.float32)
    u = np.ones((1, L, 2), np.float32)
    dt_raw = np.broadcast_to(raw, (1, L, 2))
    ones = np.ones((1, L, 1), np.float32)
    y, last = _gpu(u, dt_raw, A, ones, ones, Dv, chunks=3)
    dt = _softplus(raw)
    t = np.arange(L, dtype=np.float64)[:, None]
    a = np.exp(dt * A[:, 0].astype(np.float64))
    h = dt * (1.0 - a ** (t + 1)) / (1.0 - a)
    assert rel_l2(y[0], h + Dv) <= 1e-5
    assert rel_l2(last[0, :, 0], h[-1]) <= 1e-5


def test_dt_limits():
    x = synth.scan_inputs(2, 64, 40, 16, dtype="f32", seed=14, D="normal")
    silu = lambda z: z / (1.0 + np.exp(-z.astype(np.float64)))
    small = np.full_like(x.dt_raw, -40.0)
    y, last = _gpu(x.u, small, x.A, x.B, x.C, x.D, x.z)
    assert np.max(np.abs(last)) < 1e-12
    assert rel_l2(y, x.D * x.u.astype(np.float64) * silu(x.z)) <= 1e-5
    big = np.full_like(x.dt_raw, 40.0)
    y, last = _gpu(x.u, big, x.A, x.B, x.C, x.D, x.z)
    CB = np.sum(x.C.astype(np.float64) * x.B, axis=-1)
    u = x.u.astype(np.float64)
    ref = (40.0 * CB[:, :, None] * u + x.D * u) * silu(x.z)
    assert rel_l2(y, ref) <= 1e-5
