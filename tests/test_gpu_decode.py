"""GPU parity of the single-token selective state update (decode) against
the fp64 oracle, and decode-versus-scan equivalence on the GPU."""
import numpy as np
import pytest

import oracle
import selective_state_space_144_b300 as msc
from selective_state_space_144_b300 import synth
from tests.helpers import TOL, as_stored, from_device, rel_l2, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _step_dev(s, dtype):
    return dict(u=to_device(s.u, dtype), dt=to_device(s.dt_raw, dtype),
                B=to_device(s.B, dtype), C=to_device(s.C, dtype),
                z=to_device(s.z, dtype))


def run_decode(batch, d_inner, d_state, steps, dtype, sel=None, seed=4,
               with_z=True, with_D=True, with_bias=True):
    """Run `steps` decode steps on the GPU and in the oracle (restricted to
    channels `sel` when given); return the worst rel-L2 over every step's
    output and over the final state."""
    p = synth.decode_params(batch, d_inner, d_state, seed=seed, dtype=dtype)
    D = p.D if with_D else None
    bias = p.dt_bias if with_bias else None
    state = torch.from_numpy(p.state0).cuda()
    A_d = to_device(p.A, "f32")
    D_d = to_device(D, "f32")
    b_d = to_device(bias, "f32")
    sel = np.arange(d_inner) if sel is None else sel
    ref_state = p.state0[:, sel].astype(np.float64)
    worst = 0.0
    for k in range(steps):
        s = synth.decode_step(batch, d_inner, d_state, k, seed=seed, dtype=dtype)
        dv = _step_dev(s, dtype)
        out = torch.full((batch, d_inner), float("nan"), dtype=dv["u"].dtype,
                         device="cuda")
        msc.selective_state_update(state, dv["u"], dv["dt"], A_d, dv["B"],
                                   dv["C"], D_d, dv["z"] if with_z else None,
                                   b_d, out=out)
        ref_state, ref_out = oracle.state_update(
            ref_state, s.u[:, sel], s.dt_raw[:, sel], p.A[sel], s.B, s.C,
            None if D is None else D[sel], s.z[:, sel] if with_z else None,
            None if bias is None else bias[sel])
        got = from_device(out)[:, sel]
        assert np.all(np.isfinite(got))
        worst = max(worst, rel_l2(got, as_stored(ref_out, dtype)))
    torch.cuda.synchronize()
    e_state = rel_l2(from_device(state)[:, sel], ref_state)
    return worst, e_state


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d_state", [1, 3, 4, 5, 8, 16, 32, 33, 64])
def test_decode_small(dtype, d_state):
    e_out, e_state = run_decode(3, 50, d_state, 6, dtype, seed=10 + d_state)
    assert e_out <= TOL[dtype], e_out
    assert e_state <= TOL[dtype], e_state


@pytest.mark.parametrize("drop", ["z", "D", "dt_bias"])
def test_decode_optional_inputs(drop):
    e_out, e_state = run_decode(2, 40, 16, 3, "f32", with_z=drop != "z",
                                with_D=drop != "D", with_bias=drop != "dt_bias")
    assert e_out <= TOL["f32"] and e_state <= TOL["f32"]


def test_decode_full_size_sampled():
    """The 256 x 5120 x 16 decode workload: 12 consecutive steps, every
    output and the final state compared on 64 sampled channels."""
    sel = np.sort(np.random.default_rng(0).choice(5120, 64, replace=False))
    e_out, e_state = run_decode(256, 5120, 16, 12, "bf16", sel=sel)
    assert e_out <= TOL["bf16"], e_out
    assert e_state <= TOL["bf16"], e_state


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_steps_equal_scan(dtype):
    """L decode steps from a zero state reproduce the scan's outputs and its
    last_state ("State space models and Mamba": recurrent decoding)."""
    batch, L, d_inner, N = 2, 40, 72, 16
    x = synth.scan_inputs(batch, L, d_inner, N, dtype=dtype, seed=21,
                          D="normal")
    dev = {k: to_device(getattr(x, k), dtype) for k in ("u", "dt_raw", "z", "B", "C")}
    A = to_device(x.A, "f32")
    D = to_device(x.D, "f32")
    bias = to_device(x.dt_bias, "f32")
    msc.tuning_set("scan_chunks", 1)
    try:
        y, last = msc.selective_scan_fwd(dev["u"], dev["dt_raw"], A, dev["B"],
                                         dev["C"], D, dev["z"], bias)
    finally:
        msc.tuning_set("scan_chunks", 0)
    state = torch.zeros(batch, d_inner, N, device="cuda")
    outs = []
    for t in range(L):
        outs.append(msc.selective_state_update(
            state, dev["u"][:, t].contiguous(), dev["dt_raw"][:, t].contiguous(),
            A, dev["B"][:, t].contiguous(), dev["C"][:, t].contiguous(), D,
            dev["z"][:, t].contiguous(), bias))
    torch.cuda.synchronize()
    y_dec = torch.stack(outs, dim=1)
    assert rel_l2(from_device(y_dec), from_device(y)) <= 1e-6
    assert rel_l2(from_device(state), from_device(last)) <= 1e-6


def test_decode_general_kernel_with_unaligned_A():
    """A whose rows are not 16-byte aligned takes the general decode kernel
    (a thread per 4 states); same parity bar."""
    batch, d_inner, N = 4, 64, 16
    p = synth.decode_params(batch, d_inner, N, seed=31, dtype="f32")
    s = synth.decode_step(batch, d_inner, N, 0, seed=31, dtype="f32")
    flat = torch.empty(d_inner * N + 1, device="cuda")
    A_d = flat[1:].view(d_inner, N)
    A_d.copy_(torch.from_numpy(p.A))
    state = torch.from_numpy(p.state0).cuda()
    dv = _step_dev(s, "f32")
    out = msc.selective_state_update(state, dv["u"], dv["dt"], A_d, dv["B"], dv["C"],
                                     to_device(p.D, "f32"), dv["z"],
                                     to_device(p.dt_bias, "f32"))
    torch.cuda.synchronize()
    ref_state, ref_out = oracle.state_update(p.state0, s.u, s.dt_raw, p.A, s.B, s.C,
                                             p.D, s.z, p.dt_bias)
    assert rel_l2(from_device(out), ref_out) <= TOL["f32"]
    assert rel_l2(from_device(state), ref_state) <= TOL["f32"]


@pytest.mark.parametrize("N", [8, 16, 32, 64])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("batch,d_inner", [(1, 8), (3, 136), (5, 1000), (7, 264), (40, 640)])
def test_decode_stream_kernel_shapes(N, dtype, batch, d_inner):
    """d_state 16-64 with aligned arrays takes the copy-engine streaming
    kernel (tiles of 2048/N channels; d_state 8 the thread-per-channel
    kernel on both paths): partial tiles, batch rows spread over
    CTAs, fp32 and bf16 storage.  Four steps against the oracle, and the
    state bit for bit against the thread-per-channel or general kernel (the
    same operations per state)."""
    steps = 4
    p = synth.decode_params(batch, d_inner, N, seed=60 + d_inner, dtype=dtype)
    A, D, bias = to_device(p.A, "f32"), to_device(p.D, "f32"), to_device(p.dt_bias, "f32")
    states = {}
    outs = {}
    try:
        for path in (0, 1):
            msc.tuning_set("update_path", path)
            state = torch.from_numpy(p.state0).cuda()
            ref_state = p.state0.astype(np.float64)
            worst = 0.0
            for k in range(steps):
                s = synth.decode_step(batch, d_inner, N, k, seed=60 + d_inner, dtype=dtype)
                dv = _step_dev(s, dtype)
                out = torch.full((batch, d_inner), float("nan"), dtype=dv["u"].dtype,
                                 device="cuda")
                msc.selective_state_update(state, dv["u"], dv["dt"], A, dv["B"], dv["C"], D,
                                           dv["z"], bias, out=out)
                ref_state, ref_out = oracle.state_update(ref_state, s.u, s.dt_raw, p.A, s.B,
                                                         s.C, p.D, s.z, p.dt_bias)
                got = from_device(out)
                assert np.all(np.isfinite(got))
                worst = max(worst, rel_l2(got, as_stored(ref_out, dtype)))
            torch.cuda.synchronize()
            assert worst <= TOL[dtype], (path, worst)
            assert rel_l2(from_device(state), ref_state) <= TOL[dtype]
            states[path] = state.cpu()
            outs[path] = out.float().cpu()
    finally:
        msc.tuning_set("update_path", 0)
    assert torch.equal(states[0], states[1])


@pytest.mark.parametrize("disc", ["zoh", "trapezoid"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("batch,d_inner,N", [(3, 136, 16), (5, 1000, 16), (40, 640, 16),
                                             (9, 264, 8), (6, 200, 32), (4, 72, 64)])
def test_decode_stream_kernel_variants(disc, dtype, batch, d_inner, N):
    """The streaming decode kernel with the zero-order-hold input and with
    the exponential trapezoid (lambda, and the previous token's u and B from
    the second step on): four steps against the oracle on both decode
    kernels, and the state bit for bit between them."""
    steps = 4
    p = synth.decode_params(batch, d_inner, N, seed=70 + d_inner, dtype=dtype)
    A, D, bias = to_device(p.A, "f32"), to_device(p.D, "f32"), to_device(p.dt_bias, "f32")
    states = {}
    try:
        for path in (0, 1):
            msc.tuning_set("update_path", path)
            state = torch.from_numpy(p.state0).cuda()
            ref_state = p.state0.astype(np.float64)
            rng = np.random.default_rng(71 + d_inner)
            up = Bp = None
            worst = 0.0
            for k in range(steps):
                s = synth.decode_step(batch, d_inner, N, k, seed=70 + d_inner, dtype=dtype)
                dv = _step_dev(s, dtype)
                if disc == "zoh":
                    out = msc.selective_state_update(state, dv["u"], dv["dt"], A, dv["B"],
                                                     dv["C"], D, dv["z"], bias, zoh=True)
                    ref_state, ref_out = oracle.state_update(ref_state, s.u, s.dt_raw, p.A,
                                                             s.B, s.C, p.D, s.z, p.dt_bias,
                                                             zoh=True)
                else:
                    lam = rng.uniform(0, 1, (batch, d_inner)).astype(np.float32)
                    if dtype == "bf16":
                        lam = synth.round_bf16(lam)
                    out = msc.selective_state_update_trap(
                        state, None if up is None else to_device(up, dtype),
                        None if Bp is None else to_device(Bp, dtype), dv["u"], dv["dt"],
                        to_device(lam, dtype), A, dv["B"], dv["C"], D, dv["z"], bias)
                    ref_state, ref_out = oracle.state_update_trap(
                        ref_state, up, Bp, s.u, s.dt_raw, lam, p.A, s.B, s.C, p.D, s.z,
                        p.dt_bias)
                    up, Bp = s.u, s.B
                got = from_device(out)
                assert np.all(np.isfinite(got))
                worst = max(worst, rel_l2(got, as_stored(ref_out, dtype)))
            torch.cuda.synchronize()
            assert worst <= TOL[dtype], (path, worst)
            assert rel_l2(from_device(state), ref_state) <= TOL[dtype]
            states[path] = state.cpu()
    finally:
        msc.tuning_set("update_path", 0)
    assert torch.equal(states[0], states[1])
