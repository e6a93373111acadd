"""Pins that tie the fp64 oracle to facts outside itself.

Each check takes an oracle object (``oracle.Oracle``) so that the same checks
can be run against builds of the oracle with a planted mistake
(tests/test_oracle_mutants.py): every plausible mistake must fail at least
one of them.  None of these checks re-types the oracle's loop; each uses a
different evaluation that the pages or plain mathematics fix:

  * softplus / silu identities and values (inverse of the bias recipe,
    softplus(x) - softplus(-x) = x, silu via tanh);
  * the unrolled state-space/attention dual sum ("Deep dive into Mamba"
    section 6.1 and the formula summary of section 12), evaluated with
    cumulative sums of the step size instead of running products;
  * the LTI special case as a causal convolution with kernel
    K = (C.B', C.A'.B', C.A'^2.B', ...) (presentation article, section 2.1);
  * the geometric-series closed form for a constant scalar system;
  * segmented scan == sequential scan (presentation article, section 3.2);
  * the dt -> 0 and dt -> infinity limits (presentation article, 4.1);
  * decode steps == scan ("State space models and Mamba", Mamba decoding);
  * the stability bound |h| <= sum |dt B u| when A < 0;
  * a hand-worked example with exactly representable decays
    (tests/golden/hand_worked_l3_n2.json);
  * split prefill: a scan over [0, k) whose last state seeds (h0) the scan
    over [k, L) reproduces the scan over [0, L);
  * zero-order hold ("State space models and Mamba", discretisation; "Deep
    dive into Mamba" section 12): with the input held constant over each
    step, the discrete state equals the continuous system's solution at the
    step ends -- checked against a fine Runge-Kutta integration of
    h' = A h + B u and against the closed-form step response
    h(t) = B (e^(A t) - 1) / A; ZOH reduces to delta*B when A = 0 and as
    delta -> 0;
  * the causal depthwise conv1d before the scan ("Deep dive into Mamba"
    sections 3.2 and 5.2): against torch's own conv1d in fp64 (groups =
    channels, padding d_conv - 1, first L outputs), identity and pure-delay
    kernels, its conv state equal to convolving the concatenated sequence,
    and decode steps equal to the prefill;
  * the Mamba-3 exponential-trapezoid scan (Mamba series article, 2.1):
    lambda = 1 is the Euler scan bit for bit, lambda = 0 is the Euler scan of
    the inputs delayed one step, a constant-input closed form, split prefill
    carrying the previous step's input, decode == scan;
  * the scan's backward pass: every gradient against central finite
    differences of the (pinned) forward oracle, and against torch autograd
    through an fp64 forward written here with tensor operations.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

from selective_state_space_144_b300 import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def rel_l2(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = float(np.linalg.norm(ref.ravel()))
    num = float(np.linalg.norm((got - ref).ravel()))
    if den == 0.0:
        return num
    return num / den


def _softplus_np(x):
    # library routine: log(e^0 + e^x)
    return np.logaddexp(0.0, np.asarray(x, dtype=np.float64))


def _silu_np(z):
    z = np.asarray(z, dtype=np.float64)
    return z * 0.5 * (1.0 + np.tanh(0.5 * z))


def _random_case(batch, L, d_inner, d_state, seed, with_z=True):
    x = synth.scan_inputs(batch, L, d_inner, d_state, dtype="f32", seed=seed,
                          D="normal", A_kind="random", with_z=with_z)
    # make the bias channel-dependent and the skip non-trivial
    return x


# --------------------------------------------------------------------------
def check_softplus(orc):
    for v in (1e-3, 0.0123, 0.1, 0.5, 3.0):
        got = orc.softplus(math.log(math.expm1(v)))
        assert abs(got - v) <= 1e-14 * v + 1e-300, (v, got)
    assert abs(orc.softplus(0.0) - math.log(2.0)) <= 1e-16
    for x in (-30.0, -5.0, -0.3, 0.7, 12.0, 40.0):
        d = orc.softplus(x) - orc.softplus(-x)
        assert abs(d - x) <= 1e-14 * max(1.0, abs(x)), (x, d)
    assert orc.softplus(800.0) == 800.0
    assert 0.0 <= orc.softplus(-800.0) < 1e-300


def check_silu(orc):
    assert orc.silu(0.0) == 0.0
    for zv in (-20.0, -3.0, -0.4, 0.25, 1.5, 9.0):
        ref = float(_silu_np(zv))
        assert abs(orc.silu(zv) - ref) <= 1e-14 * max(1.0, abs(ref)), zv
        assert abs(orc.silu(zv) - orc.silu(-zv) - zv) <= 1e-14 * max(1, abs(zv))


def _dual_form(x, h0=None):
    """y via the unrolled sum over j <= t of C_t (prod_{l=j+1..t} dA_l) dB_j u_j,
    the products taken as exp(A * (S_t - S_j)) with S the running sum of the
    step sizes; plus the h0 term exp(A * S_t) h0; then D*u and the gate."""
    u = x.u.astype(np.float64)
    batch, L, d_inner = u.shape
    N = x.B.shape[-1]
    A = x.A.astype(np.float64)
    Bm = x.B.astype(np.float64)
    Cm = x.C.astype(np.float64)
    bias = 0.0 if x.dt_bias is None else x.dt_bias.astype(np.float64)
    delta = _softplus_np(x.dt_raw.astype(np.float64) + bias)
    S = np.cumsum(delta, axis=1)                     # (b, t, d), inclusive
    y = np.zeros((batch, L, d_inner))
    last = np.zeros((batch, d_inner, N))
    for b in range(batch):
        for d in range(d_inner):
            for t in range(L):
                acc = 0.0
                for j in range(t + 1):
                    w = np.exp(A[d] * (S[b, t, d] - S[b, j, d]))
                    acc += float(np.sum(Cm[b, t] * w * delta[b, j, d]
                                        * Bm[b, j] * u[b, j, d]))
                if h0 is not None:
                    acc += float(np.sum(Cm[b, t] * np.exp(A[d] * S[b, t, d])
                                        * h0[b, d]))
                y[b, t, d] = acc
            for j in range(L):
                last[b, d] += (np.exp(A[d] * (S[b, L - 1, d] - S[b, j, d]))
                               * delta[b, j, d] * Bm[b, j] * u[b, j, d])
            if h0 is not None:
                last[b, d] += np.exp(A[d] * S[b, L - 1, d]) * h0[b, d]
    if x.D is not None:
        y += x.D.astype(np.float64)[None, None, :] * u
    if x.z is not None:
        y *= _silu_np(x.z)
    return y, last


def check_dual_form(orc):
    x = _random_case(2, 12, 3, 3, seed=11)
    y_ref, last_ref = _dual_form(x)
    y, last = orc.scan_fwd(x.u, x.dt_raw, x.A, x.B, x.C, x.D, x.z, x.dt_bias)
    assert rel_l2(y, y_ref) < 1e-12, rel_l2(y, y_ref)
    assert rel_l2(last, last_ref) < 1e-12, rel_l2(last, last_ref)
    # with a given initial state
    rng = np.random.default_rng(5)
    h0 = rng.standard_normal((2, 3, 3))
    y_ref, last_ref = _dual_form(x, h0=h0)
    y, last = orc.scan_fwd(x.u, x.dt_raw, x.A, x.B, x.C, x.D, x.z, x.dt_bias,
                           h0=h0)
    assert rel_l2(y, y_ref) < 1e-12, rel_l2(y, y_ref)
    assert rel_l2(last, last_ref) < 1e-12, rel_l2(last, last_ref)


def check_lti_convolution(orc):
    """Constant dt, B, C over time: y = K * u + D u with
    K_k = sum_n C_n exp(k dt A_n) dt B_n, evaluated directly per lag k."""
    batch, L, d_inner, N = 2, 256, 3, 4
    rng = np.random.default_rng(7)
    x = _random_case(batch, L, d_inner, N, seed=12, with_z=False)
    raw = rng.normal(0.0, 0.5, size=d_inner)
    x.dt_raw = np.broadcast_to(raw[None, None, :], (batch, L, d_inner)).copy()
    Bc = rng.standard_normal((batch, N))
    Cc = rng.standard_normal((batch, N))
    x.B = np.broadcast_to(Bc[:, None, :], (batch, L, N)).copy()
    x.C = np.broadcast_to(Cc[:, None, :], (batch, L, N)).copy()
    y, last = orc.scan_fwd(x.u, x.dt_raw, x.A, x.B, x.C, x.D, None, x.dt_bias)
    A = x.A.astype(np.float64)
    dt = _softplus_np(raw + x.dt_bias.astype(np.float64))
    k = np.arange(L, dtype=np.float64)
    y_ref = np.zeros((batch, L, d_inner))
    for b in range(batch):
        for d in range(d_inner):
            K = (Cc[b][None, :] * np.exp(k[:, None] * dt[d] * A[d][None, :])
                 * dt[d] * Bc[b][None, :]).sum(axis=1)
            ud = x.u[b, :, d].astype(np.float64)
            y_ref[b, :, d] = np.convolve(K, ud)[:L] + x.D[d] * ud
    assert rel_l2(y, y_ref) < 1e-12, rel_l2(y, y_ref)


def check_geometric_series(orc):
    """u = B = C = 1, N = 1, constant dt: h_t = dt (1 - a^(t+1)) / (1 - a),
    a = exp(dt A); y_t = h_t + D."""
    batch, L, d_inner, N = 1, 40, 2, 1
    A = np.array([[-0.7], [-2.0]])
    raw = np.array([0.3, -1.1])
    Dv = np.array([0.25, -1.5])
    u = np.ones((batch, L, d_inner))
    dt_raw = np.broadcast_to(raw, (batch, L, d_inner)).copy()
    ones = np.ones((batch, L, N))
    y, last = orc.scan_fwd(u, dt_raw, A, ones, ones, Dv, None, None)
    dt = _softplus_np(raw)
    t = np.arange(L, dtype=np.float64)[:, None]
    a = np.exp(dt * A[:, 0])
    h = dt * (1.0 - a ** (t + 1)) / (1.0 - a)
    assert rel_l2(y[0], h + Dv) < 1e-13, rel_l2(y[0], h + Dv)
    assert rel_l2(last[0, :, 0], h[-1]) < 1e-13


def check_segmented_equals_sequential(orc):
    L = 150
    x = _random_case(2, L, 3, 4, seed=13)
    y0, last0 = orc.scan_fwd(x.u, x.dt_raw, x.A, x.B, x.C, x.D, x.z, x.dt_bias)
    for seg in (1, 3, 64, L, 1000):
        y, last = orc.scan_fwd_segmented(x.u, x.dt_raw, x.A, x.B, x.C, x.D,
                                         x.z, x.dt_bias, seg=seg)
        assert rel_l2(y, y0) < 1e-12, (seg, rel_l2(y, y0))
        assert rel_l2(last, last0) < 1e-12, (seg, rel_l2(last, last0))


def check_dt_limits(orc):
    x = _random_case(2, 20, 3, 4, seed=14)
    # dt -> 0: state stays ~0, y -> D u silu(z)
    small = np.full_like(x.dt_raw, -40.0)
    y, last = orc.scan_fwd(x.u, small, x.A, x.B, x.C, x.D, x.z, None)
    assert np.max(np.abs(last)) < 1e-15
    ref = x.D[None, None, :] * x.u.astype(np.float64) * _silu_np(x.z)
    assert rel_l2(y, ref) < 1e-12
    # dt -> infinity with A <= -1: the state forgets everything but the
    # current input, h_t = dt B_t u_t, y_t = dt (C_t . B_t) u_t + D u_t
    big = np.full_like(x.dt_raw, 40.0)
    A = np.minimum(x.A, -1.0)
    y, last = orc.scan_fwd(x.u, big, A, x.B, x.C, x.D, x.z, None)
    dt = _softplus_np(40.0)
    CB = np.sum(x.C.astype(np.float64) * x.B.astype(np.float64), axis=-1)
    u = x.u.astype(np.float64)
    ref = (dt * CB[:, :, None] * u + x.D[None, None, :] * u) * _silu_np(x.z)
    assert rel_l2(y, ref) < 1e-12, rel_l2(y, ref)
    ref_last = dt * x.B[:, -1, None, :].astype(np.float64) * u[:, -1, :, None]
    assert rel_l2(last, ref_last) < 1e-12


def check_decode_equals_scan(orc):
    batch, L, d_inner, N = 3, 17, 4, 5
    x = _random_case(batch, L, d_inner, N, seed=15)
    y, last = orc.scan_fwd(x.u, x.dt_raw, x.A, x.B, x.C, x.D, x.z, x.dt_bias)
    st = np.zeros((batch, d_inner, N))
    for t in range(L):
        st, o = orc.state_update(st, x.u[:, t], x.dt_raw[:, t], x.A,
                                 x.B[:, t], x.C[:, t], x.D, x.z[:, t],
                                 x.dt_bias)
        assert np.array_equal(o, y[:, t]), t
    assert np.array_equal(st, last)


def check_stability_bound(orc):
    x = _random_case(2, 300, 3, 4, seed=16)
    _, last = orc.scan_fwd(x.u, x.dt_raw, x.A, x.B, x.C, x.D, x.z, x.dt_bias)
    delta = _softplus_np(x.dt_raw.astype(np.float64)
                         + x.dt_bias.astype(np.float64))
    bound = np.einsum("btd,btn->bdn", np.abs(delta * x.u),
                      np.abs(x.B.astype(np.float64)))
    assert np.all(np.abs(last) <= bound * (1 + 1e-12))
    # decays strictly inside (0, 1): the state must not simply accumulate
    assert np.all(np.abs(last) < bound)


def check_hand_worked(orc):
    with open(os.path.join(GOLDEN, "hand_worked_l3_n2.json")) as f:
        g = json.load(f)
    inp = g["inputs"]
    u = np.array(inp["u"], dtype=np.float64).reshape(1, -1, 1)
    L = u.shape[1]
    dt_raw = np.zeros((1, L, 1))
    A = np.array(inp["A"], dtype=np.float64).reshape(1, -1)
    B = np.array(inp["B"], dtype=np.float64).reshape(1, L, -1)
    C = np.array(inp["C"], dtype=np.float64).reshape(1, L, -1)
    D = np.array([inp["D"]], dtype=np.float64)
    y, last = orc.scan_fwd(u, dt_raw, A, B, C, D, None, None)
    ln2 = math.log(2.0)
    y_ref = np.array([p * ln2 + q for p, q in g["expected"]["y"]])
    last_ref = np.array([p * ln2 for p in g["expected"]["last_state_over_ln2"]])
    assert np.allclose(y[0, :, 0], y_ref, rtol=1e-14, atol=1e-15), (y, y_ref)
    assert np.allclose(last[0, 0], last_ref, rtol=1e-14, atol=1e-15)


def check_split_prefill(orc):
    """Scanning [0, k) and then [k, L) from the first part's last state (the
    h0 input) gives the outputs and last state of one scan over [0, L)."""
    L = 90
    x = _random_case(2, L, 3, 4, seed=17)
    y0, last0 = orc.scan_fwd(x.u, x.dt_raw, x.A, x.B, x.C, x.D, x.z, x.dt_bias)
    for k in (1, 37, 89):
        sl = lambda a, lo, hi: a[:, lo:hi]
        ya, la = orc.scan_fwd(sl(x.u, 0, k), sl(x.dt_raw, 0, k), x.A, sl(x.B, 0, k),
                              sl(x.C, 0, k), x.D, sl(x.z, 0, k), x.dt_bias)
        yb, lb = orc.scan_fwd(sl(x.u, k, L), sl(x.dt_raw, k, L), x.A, sl(x.B, k, L),
                              sl(x.C, k, L), x.D, sl(x.z, k, L), x.dt_bias, h0=la)
        assert rel_l2(np.concatenate([ya, yb], axis=1), y0) < 1e-13, k
        assert rel_l2(lb, last0) < 1e-13, k


def _rk4_piecewise(A, B, u, delta, h0, substeps=400):
    """Integrate h' = A h + B_t u_t (A diagonal, per state) over consecutive
    intervals of length delta_t with the input held constant on each, by the
    classical 4-stage Runge-Kutta method; return the state at every interval
    end.  Shapes: A (N,), B (L, N), u (L,), delta (L,), h0 (N,)."""
    h = np.array(h0, dtype=np.float64)
    out = np.zeros((len(u), len(h)))
    for t in range(len(u)):
        s = delta[t] / substeps
        f = lambda y: A * y + B[t] * u[t]
        for _ in range(substeps):
            k1 = f(h)
            k2 = f(h + 0.5 * s * k1)
            k3 = f(h + 0.5 * s * k2)
            k4 = f(h + s * k3)
            h = h + (s / 6.0) * (k1 + 2.0 * k2 + 2.0 * k3 + k4)
        out[t] = h
    return out


def check_zoh_matches_ode(orc):
    """Zero-order hold is exact for an input held over each step: the scan's
    states (and y = C.h + D u) match a fine RK4 integration of the continuous
    system, with step sizes up to ~2, both signs of A and a state with A = 0."""
    rng = np.random.default_rng(18)
    batch, L, d_inner, N = 1, 10, 2, 4
    u = rng.standard_normal((batch, L, d_inner))
    dt_raw = rng.normal(0.0, 1.0, (batch, L, d_inner))
    A = np.array([[-1.7, -0.4, 0.0, 0.3], [-3.0, -1.0, -0.05, 0.6]])
    B = rng.standard_normal((batch, L, N))
    C = rng.standard_normal((batch, L, N))
    Dv = np.array([0.5, -1.25])
    y, last = orc.scan_fwd(u, dt_raw, A, B, C, Dv, None, None, zoh=True)
    delta = _softplus_np(dt_raw)
    for d in range(d_inner):
        hs = _rk4_piecewise(A[d], B[0], u[0, :, d], delta[0, :, d], np.zeros(N))
        y_ref = np.sum(C[0] * hs, axis=1) + Dv[d] * u[0, :, d]
        assert rel_l2(y[0, :, d], y_ref) < 1e-10, (d, rel_l2(y[0, :, d], y_ref))
        assert rel_l2(last[0, d], hs[-1]) < 1e-10
    # and it is not the Euler input matrix at these step sizes
    ye, _ = orc.scan_fwd(u, dt_raw, A, B, C, Dv, None, None)
    assert rel_l2(ye, y) > 1e-2


def check_zoh_step_response(orc):
    """u = B = C = 1, N = 1, constant step size: the state after t+1 steps
    is the continuous step response (e^(A (t+1) delta) - 1) / A."""
    batch, L, d_inner = 1, 30, 3
    A = np.array([[-0.9], [-4.0], [0.2]])
    raw = np.array([0.4, -0.8, 1.3])
    u = np.ones((batch, L, d_inner))
    dt_raw = np.broadcast_to(raw, (batch, L, d_inner)).copy()
    ones = np.ones((batch, L, 1))
    y, last = orc.scan_fwd(u, dt_raw, A, ones, ones, None, None, None, zoh=True)
    dt = _softplus_np(raw)
    tt = (np.arange(L, dtype=np.float64)[:, None] + 1.0) * dt
    h = np.expm1(A[:, 0] * tt) / A[:, 0]
    assert rel_l2(y[0], h) < 1e-13, rel_l2(y[0], h)
    assert rel_l2(last[0, :, 0], h[-1]) < 1e-13


def check_zoh_limits(orc):
    """ZOH equals the Euler input matrix delta*B exactly when A = 0, to fp64
    rounding as delta -> 0; and its decode steps reproduce its scan."""
    x = _random_case(2, 20, 3, 4, seed=19)
    A0 = np.zeros_like(x.A)
    ye, le = orc.scan_fwd(x.u, x.dt_raw, A0, x.B, x.C, x.D, x.z, x.dt_bias)
    yz, lz = orc.scan_fwd(x.u, x.dt_raw, A0, x.B, x.C, x.D, x.z, x.dt_bias, zoh=True)
    assert np.array_equal(ye, yz) and np.array_equal(le, lz)
    small = np.full_like(x.dt_raw, -30.0)
    ye, le = orc.scan_fwd(x.u, small, x.A, x.B, x.C, x.D, x.z, None)
    yz, lz = orc.scan_fwd(x.u, small, x.A, x.B, x.C, x.D, x.z, None, zoh=True)
    assert rel_l2(lz, le) < 1e-12 and rel_l2(yz, ye) < 1e-14
    y, last = orc.scan_fwd(x.u, x.dt_raw, x.A, x.B, x.C, x.D, x.z, x.dt_bias, zoh=True)
    st = np.zeros_like(last)
    for t in range(x.u.shape[1]):
        st, o = orc.state_update(st, x.u[:, t], x.dt_raw[:, t], x.A, x.B[:, t],
                                 x.C[:, t], x.D, x.z[:, t], x.dt_bias, zoh=True)
        assert np.array_equal(o, y[:, t]), t
    assert np.array_equal(st, last)



def _conv_case(batch, L, d_inner, d_conv, seed):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((batch, L, d_inner)),
            rng.standard_normal((d_inner, d_conv)),
            rng.standard_normal(d_inner))


def check_conv_against_torch(orc):
    """The pages' module: nn.Conv1d(d, d, kernel_size=d_conv, padding=d_conv-1,
    groups=d, bias) on (batch, d, L), first L outputs, then SiLU -- here
    torch's functional conv1d in fp64 on the CPU."""
    import torch
    for d_conv, L in ((4, 37), (2, 5), (3, 2), (1, 6)):
        x, w, bias = _conv_case(2, L, 5, d_conv, seed=30 + d_conv)
        ref = torch.nn.functional.conv1d(
            torch.from_numpy(x).transpose(1, 2), torch.from_numpy(w)[:, None, :],
            torch.from_numpy(bias), padding=d_conv - 1, groups=5)[:, :, :L]
        ref = ref.transpose(1, 2).numpy()
        y, _ = orc.causal_conv1d(x, w, bias, silu=False)
        assert np.allclose(y, ref, rtol=1e-13, atol=1e-13), d_conv
        y, _ = orc.causal_conv1d(x, w, bias, silu=True)
        assert np.allclose(y, _silu_np(ref), rtol=1e-13, atol=1e-13), d_conv


def check_conv_special_kernels(orc):
    """w = e_last is the identity, w = e_first delays by d_conv - 1 steps
    (zeros enter first)."""
    x, _, _ = _conv_case(2, 20, 3, 4, seed=35)
    ident = np.zeros((3, 4)); ident[:, 3] = 1.0
    y, st = orc.causal_conv1d(x, ident, None, silu=False)
    assert np.array_equal(y, x)
    assert np.array_equal(st, np.transpose(x[:, -3:, :], (0, 2, 1)))
    delay = np.zeros((3, 4)); delay[:, 0] = 1.0
    y, _ = orc.causal_conv1d(x, delay, None, silu=False)
    assert np.array_equal(y[:, 3:], x[:, :-3]) and np.all(y[:, :3] == 0.0)


def check_conv_state(orc):
    """A conv state (the d_conv-1 inputs before t = 0, oldest first) acts as
    a prefix of the sequence; state_out holds the last d_conv-1 inputs, also
    when L < d_conv - 1; prefill in two pieces equals one prefill."""
    x, w, bias = _conv_case(2, 30, 4, 4, seed=36)
    prev = np.random.default_rng(37).standard_normal((2, 3, 4))   # (batch, time, d)
    st_in = np.transpose(prev, (0, 2, 1)).copy()                   # (batch, d, 3)
    y, st = orc.causal_conv1d(x, w, bias, state_in=st_in)
    y_cat, st_cat = orc.causal_conv1d(np.concatenate([prev, x], axis=1), w, bias)
    assert np.allclose(y, y_cat[:, 3:], rtol=1e-14, atol=1e-14)
    assert np.array_equal(st, st_cat)
    for k in (1, 2, 29):
        ya, sa = orc.causal_conv1d(x[:, :k], w, bias)
        yb, sb = orc.causal_conv1d(x[:, k:], w, bias, state_in=sa)
        y0, s0 = orc.causal_conv1d(x, w, bias)
        assert np.allclose(np.concatenate([ya, yb], axis=1), y0, rtol=1e-14, atol=1e-14)
        assert np.array_equal(sb, s0), k


def check_conv_decode_equals_prefill(orc):
    x, w, bias = _conv_case(3, 12, 5, 4, seed=38)
    y, st_ref = orc.causal_conv1d(x, w, bias)
    st = np.zeros((3, 5, 3))
    for t in range(12):
        st, o = orc.conv1d_update(st, x[:, t], w, bias)
        assert np.allclose(o, y[:, t], rtol=1e-14, atol=1e-14), t
    assert np.array_equal(st, st_ref)



def check_trap_lambda_one_is_euler(orc):
    x = _random_case(2, 30, 3, 4, seed=40)
    lam = np.ones_like(x.u, dtype=np.float64)
    y1, l1 = orc.scan_fwd_trap(x.u, x.dt_raw, lam, x.A, x.B, x.C, x.D, x.z, x.dt_bias)
    y0, l0 = orc.scan_fwd(x.u, x.dt_raw, x.A, x.B, x.C, x.D, x.z, x.dt_bias)
    assert np.array_equal(y1, y0) and np.array_equal(l1, l0)


def check_trap_lambda_zero_is_delayed_euler(orc):
    """lambda = 0 injects only B_{t-1} x_{t-1} with the step size of t: the
    Euler scan of (u, B) delayed one step (the step before t = 0 given by
    u_prev / B_prev), with delta and C not delayed (no skip, no gate)."""
    x = _random_case(2, 25, 3, 4, seed=41, with_z=False)
    rng = np.random.default_rng(42)
    u_prev = rng.standard_normal((2, 3))
    B_prev = rng.standard_normal((2, 4))
    lam = np.zeros_like(x.u, dtype=np.float64)
    y, last = orc.scan_fwd_trap(x.u, x.dt_raw, lam, x.A, x.B, x.C, None, None,
                                x.dt_bias, u_prev=u_prev, B_prev=B_prev)
    u_d = np.concatenate([u_prev[:, None, :], x.u[:, :-1]], axis=1)
    B_d = np.concatenate([B_prev[:, None, :], x.B[:, :-1]], axis=1)
    y0, l0 = orc.scan_fwd(u_d, x.dt_raw, x.A, B_d, x.C, None, None, x.dt_bias)
    assert rel_l2(y, y0) < 1e-14 and rel_l2(last, l0) < 1e-14


def check_trap_closed_form(orc):
    """u = B = C = 1, N = 1, constant delta and lambda, nothing before t = 0:
    h_0 = lambda*delta, h_t = a h_{t-1} + delta, so
    h_t = a^t lambda delta + delta (1 - a^t) / (1 - a), a = exp(delta A)."""
    batch, L, d_inner = 1, 40, 3
    A = np.array([[-0.6], [-2.5], [-0.05]])
    raw = np.array([0.2, -0.7, 1.1])
    lamv = np.array([0.5, 0.3, 0.9])
    u = np.ones((batch, L, d_inner))
    dt_raw = np.broadcast_to(raw, (batch, L, d_inner)).copy()
    lam = np.broadcast_to(lamv, (batch, L, d_inner)).copy()
    ones = np.ones((batch, L, 1))
    y, last = orc.scan_fwd_trap(u, dt_raw, lam, A, ones, ones, None, None, None)
    dt = _softplus_np(raw)
    a = np.exp(dt * A[:, 0])
    t = np.arange(L, dtype=np.float64)[:, None]
    h = a ** t * lamv * dt + dt * (1.0 - a ** t) / (1.0 - a)
    assert rel_l2(y[0], h) < 1e-13, rel_l2(y[0], h)
    assert rel_l2(last[0, :, 0], h[-1]) < 1e-13


def check_trap_split_and_decode(orc):
    """Two pieces (the second seeded with the first's last state and its last
    step's u and B) equal one scan; decode tokens equal the scan."""
    x = _random_case(2, 24, 3, 5, seed=43)
    lam = np.random.default_rng(44).uniform(0.0, 1.0, x.u.shape)
    y0, l0 = orc.scan_fwd_trap(x.u, x.dt_raw, lam, x.A, x.B, x.C, x.D, x.z, x.dt_bias)
    k = 11
    sl = lambda v, lo, hi: v[:, lo:hi]
    ya, la = orc.scan_fwd_trap(sl(x.u, 0, k), sl(x.dt_raw, 0, k), sl(lam, 0, k), x.A,
                               sl(x.B, 0, k), sl(x.C, 0, k), x.D, sl(x.z, 0, k), x.dt_bias)
    yb, lb = orc.scan_fwd_trap(sl(x.u, k, 24), sl(x.dt_raw, k, 24), sl(lam, k, 24), x.A,
                               sl(x.B, k, 24), sl(x.C, k, 24), x.D, sl(x.z, k, 24),
                               x.dt_bias, h0=la, u_prev=x.u[:, k - 1], B_prev=x.B[:, k - 1])
    assert rel_l2(np.concatenate([ya, yb], axis=1), y0) < 1e-14
    assert rel_l2(lb, l0) < 1e-14
    st = np.zeros_like(l0)
    for t in range(24):
        up = x.u[:, t - 1] if t else None
        Bp = x.B[:, t - 1] if t else None
        st, o = orc.state_update_trap(st, up, Bp, x.u[:, t], x.dt_raw[:, t], lam[:, t],
                                      x.A, x.B[:, t], x.C[:, t], x.D, x.z[:, t], x.dt_bias)
        assert np.array_equal(o, y0[:, t]), t
    assert np.array_equal(st, l0)



def _bwd_case(seed):
    x = _random_case(2, 5, 2, 3, seed=seed)
    rng = np.random.default_rng(seed + 1)
    h0 = rng.standard_normal((2, 2, 3))
    w_out = rng.standard_normal(x.u.shape)
    w_last = rng.standard_normal((2, 2, 3))
    return x, h0, w_out, w_last


def _bwd_inputs(x, h0):
    return dict(u=x.u, dt_raw=x.dt_raw, A=x.A, B=x.B, C=x.C, D=x.D, z=x.z,
                dt_bias=x.dt_bias, h0=h0)


def check_bwd_finite_differences(orc):
    """J = sum(out * w_out) + sum(last * w_last); every input element's
    gradient against a central difference of the forward oracle."""
    x, h0, w_out, w_last = _bwd_case(50)
    inp = {k: np.array(v, dtype=np.float64) for k, v in _bwd_inputs(x, h0).items()}
    g = orc.scan_bwd(inp["u"], inp["dt_raw"], inp["A"], inp["B"], inp["C"], inp["D"],
                     inp["z"], inp["dt_bias"], inp["h0"], dout=w_out, dlast=w_last)
    names = dict(u="du", dt_raw="ddt", A="dA", B="dB", C="dC", D="dD", z="dz",
                 dt_bias="ddt_bias", h0="dh0")

    def J(v):
        y, last = orc.scan_fwd(v["u"], v["dt_raw"], v["A"], v["B"], v["C"], v["D"],
                               v["z"], v["dt_bias"], h0=v["h0"])
        return float(np.sum(y * w_out) + np.sum(last * w_last))
    eps = 1e-6
    for key, gname in names.items():
        arr = inp[key]
        for idx in np.ndindex(arr.shape):
            old = arr[idx]
            arr[idx] = old + eps
            jp = J(inp)
            arr[idx] = old - eps
            jm = J(inp)
            arr[idx] = old
            fd = (jp - jm) / (2 * eps)
            got = g[gname][idx]
            assert abs(got - fd) <= 1e-6 * (1.0 + abs(fd)), (key, idx, got, fd)


def check_bwd_against_autograd(orc):
    """The same gradients from torch autograd through an fp64 forward written
    with tensor operations (softplus as log(1 + e^x), silu as z sigmoid z)."""
    import torch
    x, h0, w_out, w_last = _bwd_case(51)
    t = {k: torch.tensor(np.asarray(v, dtype=np.float64), requires_grad=True)
         for k, v in _bwd_inputs(x, h0).items()}
    delta = torch.logaddexp(torch.zeros((), dtype=torch.float64), t["dt_raw"] + t["dt_bias"])
    h = t["h0"]
    outs = []
    for s in range(x.u.shape[1]):
        a = torch.exp(delta[:, s, :, None] * t["A"][None])
        h = a * h + delta[:, s, :, None] * t["B"][:, s, None, :] * t["u"][:, s, :, None]
        y = (h * t["C"][:, s, None, :]).sum(-1) + t["D"] * t["u"][:, s]
        outs.append(y * t["z"][:, s] * torch.sigmoid(t["z"][:, s]))
    J = (torch.stack(outs, 1) * torch.from_numpy(w_out)).sum() + \
        (h * torch.from_numpy(w_last)).sum()
    keys = list(t)
    grads = torch.autograd.grad(J, [t[k] for k in keys])
    g = orc.scan_bwd(x.u, x.dt_raw, x.A, x.B, x.C, x.D, x.z, x.dt_bias, h0,
                     dout=w_out, dlast=w_last)
    names = dict(u="du", dt_raw="ddt", A="dA", B="dB", C="dC", D="dD", z="dz",
                 dt_bias="ddt_bias", h0="dh0")
    for k, gr in zip(keys, grads):
        assert rel_l2(g[names[k]], gr.numpy()) < 1e-12, k


ALL_CHECKS = [
    check_softplus,
    check_silu,
    check_dual_form,
    check_lti_convolution,
    check_geometric_series,
    check_segmented_equals_sequential,
    check_dt_limits,
    check_decode_equals_scan,
    check_stability_bound,
    check_hand_worked,
    check_split_prefill,
    check_zoh_matches_ode,
    check_zoh_step_response,
    check_zoh_limits,
    check_conv_against_torch,
    check_conv_special_kernels,
    check_conv_state,
    check_conv_decode_equals_prefill,
    check_trap_lambda_one_is_euler,
    check_trap_lambda_zero_is_delayed_euler,
    check_trap_closed_form,
    check_trap_split_and_decode,
    check_bwd_finite_differences,
    check_bwd_against_autograd,
]
