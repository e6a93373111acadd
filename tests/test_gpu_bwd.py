"""GPU parity of the selective scan's backward pass against the fp64 oracle's
adjoint (itself pinned against finite differences and torch autograd).

Gradients stored in the input dtype (du, ddt, dz) are compared like the
forward outputs: rel-L2 <= 1e-5 for fp32 storage, <= 2e-3 for bf16 storage
(oracle rounded to bf16).  The fp32 gradients that are sums over steps or
channels (dA, dB, dC, dD, ddt_bias) and dh0 come from the same bf16-rounded
inputs on both sides and differ only by fp32 accumulation order: rel-L2 <=
2e-5 (fp32 and bf16 storage alike)."""
import numpy as np
import pytest

import oracle
import selective_state_space_144_b300 as msc
from selective_state_space_144_b300 import synth
from tests.helpers import TOL, as_stored, from_device, rel_l2, scan_device_args, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
SUM_TOL = 2e-5


def grads(x, *, h0=None, dlast=True, seed=0, want_dh0=True):
    rng = np.random.default_rng(seed)
    dout = rng.standard_normal(x.u.shape).astype(np.float32)
    if x.dtype == "bf16":
        dout = synth.round_bf16(dout)
    dl = rng.standard_normal((x.u.shape[0], x.u.shape[2], x.B.shape[-1])).astype(np.float32) \
        if dlast else None
    a = scan_device_args(x)
    g = msc.selective_scan_bwd(
        a["u"], a["dt"], a["A"], a["B"], a["C"], a["D"], a["z"], a["dt_bias"],
        h0=None if h0 is None else to_device(h0, "f32"), dout=to_device(dout, x.dtype),
        dlast_state=None if dl is None else to_device(dl, "f32"), want_dh0=want_dh0)
    torch.cuda.synchronize()
    ref = oracle.scan_bwd(x.u, x.dt_raw, x.A, x.B, x.C, x.D, x.z, x.dt_bias, h0,
                          dout=dout, dlast=dl)
    return {k: (None if v is None else from_device(v)) for k, v in g.items()}, ref


def check(x, **kw):
    got, ref = grads(x, **kw)
    for k in ("du", "ddt", "dz"):
        if got[k] is None:
            continue
        assert np.all(np.isfinite(got[k])), k
        e = rel_l2(got[k], as_stored(ref[k], x.dtype))
        assert e <= TOL[x.dtype], f"{k} rel-L2 {e:.3e}"
    for k in ("dA", "dB", "dC", "dD", "ddt_bias", "dh0"):
        if got[k] is None:
            continue
        e = rel_l2(got[k], ref[k])
        assert e <= SUM_TOL, f"{k} rel-L2 {e:.3e}"


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d_state", [1, 3, 4, 8, 16, 32, 33, 64])
def test_bwd_state_sizes(dtype, d_state):
    x = synth.scan_inputs(2, 77, 45, d_state, dtype=dtype, seed=800 + d_state,
                          D="normal", A_kind="random")
    check(x, seed=1)


@pytest.mark.parametrize("L", [1, 5, 31, 32, 33, 64, 100])
def test_bwd_lengths(L):
    """Segments of 32 recomputed steps: one partial, exactly one, ragged."""
    x = synth.scan_inputs(2, L, 64, 16, dtype="f32", seed=820 + L, D="normal")
    check(x, seed=2)


@pytest.mark.parametrize("drop", ["z", "D", "dt_bias", "all"])
def test_bwd_optional_inputs(drop):
    x = synth.scan_inputs(2, 90, 40, 16, dtype="f32", seed=840,
                          with_z=drop not in ("z", "all"), with_D=drop not in ("D", "all"),
                          with_bias=drop not in ("dt_bias", "all"))
    check(x, seed=3)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_bwd_h0_and_no_dlast(dtype):
    x = synth.scan_inputs(3, 70, 64, 16, dtype=dtype, seed=850, D="normal")
    h0 = np.random.default_rng(4).standard_normal((3, 64, 16)).astype(np.float32)
    check(x, h0=h0, seed=5)
    check(x, h0=h0, dlast=False, seed=6)


def test_bwd_empty_sequence():
    """L = 0: dh0 = dlast, dA = 0."""
    x = synth.scan_inputs(2, 0, 64, 16, dtype="f32", seed=860)
    got, ref = grads(x, seed=7)
    assert np.array_equal(got["dh0"], ref["dh0"].astype(np.float32))
    assert np.all(got["dA"] == 0.0)


def test_bwd_workload_reduced():
    """The 8 x 2048 x 1536 x 16 layer's distributions at reduced size."""
    x = synth.workload_inputs("mamba130m_layer", batch=2, L=300, d_inner=200)
    check(x, seed=8)


def test_bwd_mid_size():
    """Many channel tiles and segments: 2 x 512 x 512 x 16, bf16."""
    x = synth.scan_inputs(2, 512, 512, 16, dtype="bf16", seed=870, D="normal")
    check(x, seed=9, want_dh0=False)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d_state", [8, 16, 32, 64])
@pytest.mark.parametrize("L", [1, 8, 16, 17, 40])
def test_bwd_tma_tiles(dtype, d_state, L):
    """Shapes the TMA backward takes (d_inner % 8 == 0, N in {8, 16, 32, 64}):
    tiles of 16 steps (N <= 16) or 8 steps (N > 16), one tile or several,
    whole or ragged, with h0 so that the first tile's entering state is used."""
    x = synth.scan_inputs(2, L, 48, d_state, dtype=dtype, seed=900 + d_state + L,
                          D="normal", A_kind="random")
    h0 = np.random.default_rng(L).standard_normal((2, 48, d_state)).astype(np.float32)
    check(x, h0=h0, seed=11)


def test_bwd_after_scratch_release():
    """The scratch pool gives its memory back and the next call takes it again."""
    x = synth.scan_inputs(2, 40, 64, 16, dtype="bf16", seed=960, D="normal")
    check(x, seed=12)
    msc.scratch_release()
    check(x, seed=12)


def test_bwd_tma_one_channel_group_long():
    """One CTA (batch 1, 8 channels) over 17 tiles of 16 steps, the last
    ragged: every checkpoint of the forward walk is used by the reverse walk."""
    x = synth.scan_inputs(1, 257, 8, 16, dtype="bf16", seed=970, D="normal")
    h0 = np.random.default_rng(13).standard_normal((1, 8, 16)).astype(np.float32)
    check(x, h0=h0, seed=14)


def test_bwd_tma_d_state_64_many_tiles():
    """d_state 64 (16 states per lane, the largest register footprint) over
    38 tiles of 8 steps, fp32 storage."""
    x = synth.scan_inputs(2, 300, 16, 64, dtype="f32", seed=975, D="normal", A_kind="random")
    check(x, seed=15)


def test_bwd_tma_repeatable():
    """The gradients written without atomics (du, ddt, dz, dh0) are bitwise
    equal from call to call; the atomically summed ones agree to rounding."""
    x = synth.scan_inputs(2, 200, 64, 16, dtype="bf16", seed=980, D="normal")
    a = scan_device_args(x)
    dout = to_device(synth.round_bf16(np.random.default_rng(16).standard_normal(
        x.u.shape).astype(np.float32)), "bf16")
    g1 = msc.selective_scan_bwd(a["u"], a["dt"], a["A"], a["B"], a["C"], a["D"], a["z"],
                                a["dt_bias"], dout=dout, want_dh0=True)
    g2 = msc.selective_scan_bwd(a["u"], a["dt"], a["A"], a["B"], a["C"], a["D"], a["z"],
                                a["dt_bias"], dout=dout, want_dh0=True)
    torch.cuda.synchronize()
    for k in ("du", "ddt", "dz", "dh0"):
        assert torch.equal(g1[k], g2[k]), k
    for k in ("dA", "dB", "dC", "dD", "ddt_bias"):
        assert rel_l2(from_device(g1[k]), from_device(g2[k]).astype(np.float64)) <= 1e-6, k
