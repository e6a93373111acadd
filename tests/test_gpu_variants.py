"""GPU parity of the scan variants against the fp64 oracle: the
zero-order-hold input matrix ("State space models and Mamba", section on
discretisation; "Deep dive into Mamba", section 12) and the initial state h0
(split prefill), on every kernel family (TMA kernels with 4 and 2 lanes per
channel, element-load kernels), with and without time chunks, for the scan
and the decode step.  Same tolerances as the base scan: rel-L2 <= 1e-5 for
fp32 storage, <= 2e-3 for bf16 storage against the oracle rounded to bf16.
"""
import numpy as np
import pytest

import oracle
import selective_state_space_144_b300 as msc
from selective_state_space_144_b300 import synth
from tests.helpers import TOL, as_stored, from_device, rel_l2, scan_device_args, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _defaults():
    msc.tuning_set("scan_chunks", 0)
    msc.tuning_set("scan_min_chunk", 512)
    msc.tuning_set("scan_path", 0)
    msc.tuning_set("scan_lanes", 0)


@pytest.fixture(autouse=True)
def _reset_tuning():
    _defaults()
    yield
    torch.cuda.synchronize()
    msc.check_device_error()
    _defaults()


# (scan_path, scan_lanes): TMA 4 lanes, TMA 2 lanes, element-load kernels
KERNELS = [(0, 4), (0, 2), (1, 0)]


def zoh_inputs(batch, L, d_inner, N, dtype, seed, shift=0.0):
    """Workload-like inputs whose step sizes reach both ZOH branches
    (|delta*A| below and above 1/4); channel 0 has A = 0 in state 0."""
    x = synth.scan_inputs(batch, L, d_inner, N, dtype=dtype, seed=seed,
                          D="normal", A_kind="random")
    if shift:
        raw = x.dt_raw + shift
        x.dt_raw = synth.round_bf16(raw) if dtype == "bf16" else raw.astype(np.float32)
    x.A = x.A.copy()
    x.A[0, 0] = 0.0
    return x


def run(x, *, chunks=0, path=0, lanes=0, h0=None, zoh=False, with_last=True):
    msc.tuning_set("scan_path", path)
    msc.tuning_set("scan_lanes", lanes)
    msc.tuning_set("scan_chunks", chunks)
    a = scan_device_args(x)
    batch, L, d_inner, d_state = x.u.shape + (x.B.shape[-1],)
    out = torch.full((batch, L, d_inner), float("nan"), dtype=a["u"].dtype, device="cuda")
    last = torch.full((batch, d_inner, d_state), float("nan"), device="cuda") if with_last else None
    h0_d = None if h0 is None else torch.from_numpy(np.ascontiguousarray(h0, np.float32)).cuda()
    msc.selective_scan_fwd(a["u"], a["dt"], a["A"], a["B"], a["C"], a["D"], a["z"],
                           a["dt_bias"], out=out, last_state=last,
                           return_last_state=with_last, h0=h0_d, zoh=zoh)
    torch.cuda.synchronize()
    return from_device(out), (from_device(last) if with_last else None)


def check(x, **kw):
    h0 = kw.get("h0")
    y, last = run(x, **kw)
    y_ref, last_ref = oracle.scan_fwd(x.u, x.dt_raw, x.A, x.B, x.C, x.D, x.z, x.dt_bias,
                                      h0=h0, zoh=kw.get("zoh", False))
    tol = TOL[x.dtype]
    assert np.all(np.isfinite(y))
    e_y = rel_l2(y, as_stored(y_ref, x.dtype))
    assert e_y <= tol, f"out rel-L2 {e_y:.3e}"
    if last is not None:
        e_s = rel_l2(last, last_ref)
        assert e_s <= tol, f"last_state rel-L2 {e_s:.3e}"
    return y, last


# ---- zero-order hold ---------------------------------------------------------
@pytest.mark.parametrize("path,lanes", KERNELS)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d_state", [8, 16, 32, 64])
def test_zoh_state_sizes(dtype, d_state, path, lanes):
    x = zoh_inputs(2, 333, 96, d_state, dtype, seed=500 + d_state, shift=1.0)
    check(x, zoh=True, path=path, lanes=lanes)


@pytest.mark.parametrize("d_state", [1, 3, 5, 12, 33])
def test_zoh_odd_state_sizes(d_state):
    """Sizes only the element-load kernels take."""
    x = zoh_inputs(2, 150, 40, d_state, "f32", seed=520 + d_state, shift=1.0)
    check(x, zoh=True)


@pytest.mark.parametrize("path,lanes", KERNELS)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("chunks", [2, 3, 7])
def test_zoh_chunked(dtype, chunks, path, lanes):
    """The chunk summaries (backward walk on the TMA path) use the ZOH input."""
    x = zoh_inputs(3, 517, 208, 16, dtype, seed=540 + chunks)
    check(x, zoh=True, chunks=chunks, path=path, lanes=lanes)


@pytest.mark.parametrize("shift", [-4.0, 0.0, 3.0])
def test_zoh_step_size_ranges(shift):
    """Small steps (mostly the series branch), workload steps, large steps
    (mostly the (dA - 1)/A branch)."""
    x = zoh_inputs(2, 400, 64, 16, "f32", seed=560, shift=shift)
    check(x, zoh=True)
    check(x, zoh=True, path=1)


def test_zoh_differs_from_euler():
    """The variant is really taken: at workload step sizes ZOH and Euler
    outputs differ far beyond the tolerance."""
    x = zoh_inputs(2, 200, 64, 16, "f32", seed=570, shift=1.0)
    y_e, _ = run(x)
    y_z, _ = run(x, zoh=True)
    assert rel_l2(y_z, y_e) > 1e-2


def test_zoh_a_zero_equals_euler():
    """A = 0: the ZOH gain is delta exactly, so both discretisations give the
    same bits on every kernel family."""
    x = synth.scan_inputs(2, 150, 64, 16, dtype="f32", seed=571)
    x.A = np.zeros_like(x.A)
    for path, lanes in KERNELS:
        y_e, l_e = run(x, path=path, lanes=lanes)
        y_z, l_z = run(x, path=path, lanes=lanes, zoh=True)
        assert np.array_equal(y_e, y_z) and np.array_equal(l_e, l_z), (path, lanes)


# ---- initial state h0 -------------------------------------------------------
def _h0(x, seed):
    batch, _, d_inner = x.u.shape
    return np.random.default_rng(seed).standard_normal(
        (batch, d_inner, x.B.shape[-1])).astype(np.float32)


@pytest.mark.parametrize("path,lanes", KERNELS)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("chunks", [1, 4])
def test_h0(dtype, chunks, path, lanes):
    x = synth.scan_inputs(2, 300, 72, 16, dtype=dtype, seed=600 + chunks, D="normal")
    check(x, h0=_h0(x, 1), chunks=chunks, path=path, lanes=lanes)


@pytest.mark.parametrize("zoh", [False, True])
def test_h0_with_zoh(zoh):
    x = zoh_inputs(2, 260, 64, 32, "bf16", seed=610)
    check(x, h0=_h0(x, 2), zoh=zoh, chunks=3)


@pytest.mark.parametrize("path", [0, 1])
def test_h0_empty_sequence(path):
    """L = 0: the state after zero steps is h0."""
    x = synth.scan_inputs(2, 0, 64, 16, dtype="f32", seed=620)
    h0 = _h0(x, 3)
    _, last = run(x, path=path, h0=h0)
    assert np.array_equal(last, h0)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("zoh", [False, True])
def test_split_prefill(dtype, zoh):
    """A prompt scanned in three pieces, each seeded with the previous
    piece's last_state, reproduces the single scan (and the oracle)."""
    L = 700
    x = zoh_inputs(2, L, 128, 16, dtype, seed=630)
    y_one, last_one = run(x, zoh=zoh)
    a = scan_device_args(x)
    state = None
    ys = []
    for lo, hi in ((0, 250), (250, 251), (251, L)):
        part = {k: (v[:, lo:hi].contiguous() if k in ("u", "dt", "z", "B", "C") else v)
                for k, v in a.items()}
        y, state = msc.selective_scan_fwd(part["u"], part["dt"], part["A"], part["B"],
                                          part["C"], part["D"], part["z"], part["dt_bias"],
                                          h0=state, zoh=zoh)
        ys.append(y)
    torch.cuda.synchronize()
    y_split = from_device(torch.cat(ys, dim=1))
    assert rel_l2(y_split, y_one) <= 1e-5
    assert rel_l2(from_device(state), last_one) <= 1e-5
    y_ref, last_ref = oracle.scan_fwd(x.u, x.dt_raw, x.A, x.B, x.C, x.D, x.z, x.dt_bias,
                                      zoh=zoh)
    assert rel_l2(y_split, as_stored(y_ref, dtype)) <= TOL[dtype]
    assert rel_l2(from_device(state), last_ref) <= TOL[dtype]


def test_workload_reduced_zoh_h0():
    """The 8 x 2048 x 1536 x 16 layer's distributions at reduced size, with
    both variants."""
    x = synth.workload_inputs("mamba130m_layer", batch=2, L=300, d_inner=200)
    check(x, zoh=True, h0=_h0(x, 4))


# ---- decode -----------------------------------------------------------------
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d_state", [3, 8, 16, 32, 33])
def test_zoh_decode(dtype, d_state):
    batch, d_inner, steps = 3, 50, 5
    p = synth.decode_params(batch, d_inner, d_state, seed=40 + d_state, dtype=dtype)
    A = p.A.copy()
    A[0, 0] = 0.0
    state = torch.from_numpy(p.state0).cuda()
    ref = p.state0.astype(np.float64)
    A_d, D_d, b_d = (to_device(v, "f32") for v in (A, p.D, p.dt_bias))
    for k in range(steps):
        s = synth.decode_step(batch, d_inner, d_state, k, seed=40 + d_state, dtype=dtype)
        dv = {n: to_device(getattr(s, m), dtype)
              for n, m in (("u", "u"), ("dt", "dt_raw"), ("B", "B"), ("C", "C"), ("z", "z"))}
        out = msc.selective_state_update(state, dv["u"], dv["dt"], A_d, dv["B"], dv["C"],
                                         D_d, dv["z"], b_d, zoh=True)
        ref, ref_out = oracle.state_update(ref, s.u, s.dt_raw, A, s.B, s.C, p.D, s.z,
                                           p.dt_bias, zoh=True)
        assert rel_l2(from_device(out), as_stored(ref_out, dtype)) <= TOL[dtype], k
    torch.cuda.synchronize()
    assert rel_l2(from_device(state), ref) <= TOL[dtype]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_zoh_decode_steps_equal_scan(dtype):
    """ZOH decode steps from a zero state reproduce the ZOH scan."""
    batch, L, d_inner, N = 2, 40, 72, 16
    x = zoh_inputs(batch, L, d_inner, N, dtype, seed=650)
    dev = {k: to_device(getattr(x, k), dtype) for k in ("u", "dt_raw", "z", "B", "C")}
    A, D, bias = (to_device(v, "f32") for v in (x.A, x.D, x.dt_bias))
    msc.tuning_set("scan_chunks", 1)
    y, last = msc.selective_scan_fwd(dev["u"], dev["dt_raw"], A, dev["B"], dev["C"], D,
                                     dev["z"], bias, zoh=True)
    state = torch.zeros(batch, d_inner, N, device="cuda")
    outs = [msc.selective_state_update(state, dev["u"][:, t].contiguous(),
                                       dev["dt_raw"][:, t].contiguous(), A,
                                       dev["B"][:, t].contiguous(), dev["C"][:, t].contiguous(),
                                       D, dev["z"][:, t].contiguous(), bias, zoh=True)
            for t in range(L)]
    torch.cuda.synchronize()
    assert rel_l2(from_device(torch.stack(outs, dim=1)), from_device(y)) <= 1e-6
    assert rel_l2(from_device(state), from_device(last)) <= 1e-6
