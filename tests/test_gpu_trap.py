"""GPU parity of the Mamba-3 exponential-trapezoid scan ("State space models
and the Mamba series", section 2.1) and its decode step against the fp64
oracle, on every kernel family (TMA kernels with 4 and 2 lanes per channel,
element-load kernels), with and without time chunks.  Same tolerances as the
base scan: rel-L2 <= 1e-5 for fp32 storage, <= 2e-3 for bf16 storage
against the oracle rounded to bf16."""
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


KERNELS = [(0, 4), (0, 2), (1, 0)]   # (scan_path, scan_lanes)


def lam_for(x, seed, lo=0.0, hi=1.0):
    lam = np.random.default_rng(seed).uniform(lo, hi, x.u.shape).astype(np.float32)
    return synth.round_bf16(lam) if x.dtype == "bf16" else lam


def prev_for(x, seed):
    rng = np.random.default_rng(seed)
    batch, _, d_inner = x.u.shape
    up = rng.standard_normal((batch, d_inner)).astype(np.float32)
    Bp = rng.standard_normal((batch, x.B.shape[-1])).astype(np.float32)
    if x.dtype == "bf16":
        up, Bp = synth.round_bf16(up), synth.round_bf16(Bp)
    return up, Bp


def run(x, lam, *, chunks=0, path=0, lanes=0, h0=None, u_prev=None, B_prev=None):
    msc.tuning_set("scan_path", path)
    msc.tuning_set("scan_lanes", lanes)
    msc.tuning_set("scan_chunks", chunks)
    a = scan_device_args(x)
    d = x.dtype
    batch, L, d_inner, d_state = x.u.shape + (x.B.shape[-1],)
    out = torch.full((batch, L, d_inner), float("nan"), dtype=a["u"].dtype, device="cuda")
    last = torch.full((batch, d_inner, d_state), float("nan"), device="cuda")
    msc.selective_scan_trap_fwd(
        a["u"], a["dt"], to_device(lam, d), a["A"], a["B"], a["C"], a["D"], a["z"],
        a["dt_bias"], h0=None if h0 is None else to_device(h0, "f32"),
        u_prev=None if u_prev is None else to_device(u_prev, d),
        B_prev=None if B_prev is None else to_device(B_prev, d), out=out, last_state=last)
    torch.cuda.synchronize()
    return from_device(out), from_device(last)


def check(x, lam, **kw):
    y, last = run(x, lam, **kw)
    y_ref, last_ref = oracle.scan_fwd_trap(x.u, x.dt_raw, lam, x.A, x.B, x.C, x.D, x.z,
                                           x.dt_bias, h0=kw.get("h0"),
                                           u_prev=kw.get("u_prev"), B_prev=kw.get("B_prev"))
    tol = TOL[x.dtype]
    assert np.all(np.isfinite(y))
    e_y, e_s = rel_l2(y, as_stored(y_ref, x.dtype)), rel_l2(last, last_ref)
    assert e_y <= tol, f"out rel-L2 {e_y:.3e}"
    assert e_s <= tol, f"last_state rel-L2 {e_s:.3e}"


@pytest.mark.parametrize("path,lanes", KERNELS)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d_state", [8, 16, 32, 64])
def test_trap_state_sizes(dtype, d_state, path, lanes):
    x = synth.scan_inputs(2, 333, 96, d_state, dtype=dtype, seed=700 + d_state,
                          D="normal", A_kind="random")
    check(x, lam_for(x, 1), path=path, lanes=lanes)


@pytest.mark.parametrize("d_state", [1, 3, 5, 12, 33])
def test_trap_odd_state_sizes(d_state):
    x = synth.scan_inputs(2, 150, 40, d_state, dtype="f32", seed=720 + d_state, D="normal")
    check(x, lam_for(x, 2))


@pytest.mark.parametrize("path,lanes", KERNELS)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("chunks", [2, 3, 7])
def test_trap_chunked(dtype, chunks, path, lanes):
    """Chunk summaries carry the previous-step term across chunk borders."""
    x = synth.scan_inputs(3, 517, 208, 16, dtype=dtype, seed=740 + chunks, D="normal")
    check(x, lam_for(x, 3), chunks=chunks, path=path, lanes=lanes)


@pytest.mark.parametrize("path,lanes", KERNELS)
def test_trap_chunked_large_steps(path, lanes):
    """Large step sizes: the backward summary stops early; the deferred
    previous-step weight is then below resolution too."""
    x = synth.scan_inputs(2, 1024, 64, 16, dtype="f32", seed=750, D="normal")
    x.dt_raw = x.dt_raw + 3.0
    check(x, lam_for(x, 4), chunks=4, path=path, lanes=lanes)


@pytest.mark.parametrize("path,lanes", KERNELS)
def test_trap_previous_step_and_h0(path, lanes):
    x = synth.scan_inputs(2, 260, 64, 16, dtype="bf16", seed=760, D="normal")
    up, Bp = prev_for(x, 5)
    h0 = np.random.default_rng(6).standard_normal((2, 64, 16)).astype(np.float32)
    check(x, lam_for(x, 7), path=path, lanes=lanes, h0=h0, u_prev=up, B_prev=Bp)
    check(x, lam_for(x, 7), path=path, lanes=lanes, h0=h0, u_prev=up, B_prev=Bp, chunks=3)


@pytest.mark.parametrize("path,lanes", KERNELS)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_trap_lambda_one_is_euler_bitwise(dtype, path, lanes):
    """lambda = 1: the same operations as the Euler scan on every value."""
    x = synth.scan_inputs(2, 300, 128, 16, dtype=dtype, seed=770, D="normal")
    lam = np.ones_like(x.u, dtype=np.float32)
    for chunks in (1, 3):
        y1, l1 = run(x, lam, path=path, lanes=lanes, chunks=chunks)
        msc.tuning_set("scan_chunks", chunks)
        a = scan_device_args(x)
        y0, l0 = msc.selective_scan_fwd(a["u"], a["dt"], a["A"], a["B"], a["C"], a["D"],
                                        a["z"], a["dt_bias"])
        torch.cuda.synchronize()
        assert np.array_equal(y1, from_device(y0)), chunks
        assert np.array_equal(l1, from_device(l0)), chunks


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_trap_split_prefill(dtype):
    """Three pieces, each seeded with the previous piece's last state and its
    last step's u and B, equal one scan."""
    L = 600
    x = synth.scan_inputs(2, L, 128, 16, dtype=dtype, seed=780, D="normal")
    lam = lam_for(x, 8)
    y_one, last_one = run(x, lam)
    a = scan_device_args(x)
    lam_d = to_device(lam, dtype)
    ys, state, up, Bp = [], None, None, None
    for lo, hi in ((0, 250), (250, 251), (251, L)):
        part = {k: (v[:, lo:hi].contiguous() if k in ("u", "dt", "z", "B", "C") else v)
                for k, v in a.items()}
        y, state = msc.selective_scan_trap_fwd(part["u"], part["dt"],
                                               lam_d[:, lo:hi].contiguous(), part["A"],
                                               part["B"], part["C"], part["D"], part["z"],
                                               part["dt_bias"], h0=state, u_prev=up, B_prev=Bp)
        up = a["u"][:, hi - 1].contiguous()
        Bp = a["B"][:, hi - 1].contiguous()
        ys.append(y)
    torch.cuda.synchronize()
    assert rel_l2(from_device(torch.cat(ys, dim=1)), y_one) <= 1e-5
    assert rel_l2(from_device(state), last_one) <= 1e-5


def test_trap_workload_reduced():
    x = synth.workload_inputs("mamba130m_layer", batch=2, L=300, d_inner=200)
    check(x, lam_for(x, 9))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d_state", [3, 8, 16, 32, 33])
def test_trap_decode(dtype, d_state):
    batch, d_inner, steps = 3, 50, 5
    p = synth.decode_params(batch, d_inner, d_state, seed=80 + d_state, dtype=dtype)
    state = torch.from_numpy(p.state0).cuda()
    ref = p.state0.astype(np.float64)
    A_d, D_d, b_d = (to_device(v, "f32") for v in (p.A, p.D, p.dt_bias))
    up = Bp = None
    rng = np.random.default_rng(90 + d_state)
    for k in range(steps):
        s = synth.decode_step(batch, d_inner, d_state, k, seed=80 + d_state, dtype=dtype)
        lam = rng.uniform(0, 1, (batch, d_inner)).astype(np.float32)
        if dtype == "bf16":
            lam = synth.round_bf16(lam)
        dv = {n: to_device(getattr(s, m), dtype)
              for n, m in (("u", "u"), ("dt", "dt_raw"), ("B", "B"), ("C", "C"), ("z", "z"))}
        out = msc.selective_state_update_trap(
            state, None if up is None else to_device(up, dtype),
            None if Bp is None else to_device(Bp, dtype), dv["u"], dv["dt"],
            to_device(lam, dtype), A_d, dv["B"], dv["C"], D_d, dv["z"], b_d)
        ref, ref_out = oracle.state_update_trap(ref, up, Bp, s.u, s.dt_raw, lam, p.A, s.B,
                                                s.C, p.D, s.z, p.dt_bias)
        assert rel_l2(from_device(out), as_stored(ref_out, dtype)) <= TOL[dtype], k
        up, Bp = s.u, s.B
    torch.cuda.synchronize()
    assert rel_l2(from_device(state), ref) <= TOL[dtype]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_trap_decode_steps_equal_scan(dtype):
    batch, L, d_inner, N = 2, 40, 72, 16
    x = synth.scan_inputs(batch, L, d_inner, N, dtype=dtype, seed=790, D="normal")
    lam = lam_for(x, 10)
    dev = {k: to_device(getattr(x, k), dtype) for k in ("u", "dt_raw", "z", "B", "C")}
    lam_d = to_device(lam, dtype)
    A, D, bias = (to_device(v, "f32") for v in (x.A, x.D, x.dt_bias))
    msc.tuning_set("scan_chunks", 1)
    y, last = msc.selective_scan_trap_fwd(dev["u"], dev["dt_raw"], lam_d, A, dev["B"],
                                          dev["C"], D, dev["z"], bias)
    state = torch.zeros(batch, d_inner, N, device="cuda")
    outs = []
    for t in range(L):
        up = dev["u"][:, t - 1].contiguous() if t else None
        Bp = dev["B"][:, t - 1].contiguous() if t else None
        outs.append(msc.selective_state_update_trap(
            state, up, Bp, dev["u"][:, t].contiguous(), dev["dt_raw"][:, t].contiguous(),
            lam_d[:, t].contiguous(), A, dev["B"][:, t].contiguous(),
            dev["C"][:, t].contiguous(), D, dev["z"][:, t].contiguous(), bias))
    torch.cuda.synchronize()
    assert rel_l2(from_device(torch.stack(outs, dim=1)), from_device(y)) <= 1e-6
    assert rel_l2(from_device(state), from_device(last)) <= 1e-6
