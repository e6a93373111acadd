"""GPU parity of the training path with forward-written checkpoints: the
forward scan that also stores the state entering every tile of the backward
pass, and the backward that reads those states instead of recomputing them
("Deep dive into Mamba", section 7.3: keep the states at chunk boundaries,
recompute inside a chunk).

Checked here:
* the checkpoint rows against the fp64 oracle's state after each prefix of
  the sequence (row k = the state entering step k * interval), at the same
  tolerance as last_state;
* out and last_state of the checkpointing forward equal the plain forward's
  bit for bit (the checkpoint store changes no arithmetic);
* with the forward in one time chunk, the backward reading the checkpoints
  gives du, ddt, dz, dh0 bit for bit as the self-checkpointing backward
  (the rows are the very states its forward walk computes) and the summed
  gradients to rounding; with time split into chunks, both agree with the
  oracle's adjoint at the backward's tolerances."""
import dataclasses

import numpy as np
import pytest

import oracle
import selective_state_space_144_b300 as msc
from selective_state_space_144_b300 import synth
from tests.helpers import TOL, as_stored, from_device, rel_l2, scan_device_args, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
SUM_TOL = 2e-5


def oracle_ckpt_rows(x, h0, interval):
    """The oracle's state entering step k * interval for every row k."""
    batch, L, d_inner = x.u.shape
    N = x.B.shape[-1]
    rows = (L + interval - 1) // interval
    ref = np.zeros((batch, rows, d_inner, N))
    for k in range(rows):
        t = k * interval
        if t == 0:
            ref[:, 0] = 0.0 if h0 is None else h0
            continue
        _, last = oracle.scan_fwd(x.u[:, :t], x.dt_raw[:, :t], x.A, x.B[:, :t], x.C[:, :t],
                                  x.D, None if x.z is None else x.z[:, :t], x.dt_bias, h0)
        ref[:, k] = last
    return ref


def fwd_ckpt(x, h0):
    a = scan_device_args(x)
    h0d = None if h0 is None else to_device(h0, "f32")
    out, last, ck = msc.selective_scan_fwd_ckpt(a["u"], a["dt"], a["A"], a["B"], a["C"],
                                                a["D"], a["z"], a["dt_bias"], h0=h0d)
    out0, last0 = msc.selective_scan_fwd(a["u"], a["dt"], a["A"], a["B"], a["C"], a["D"],
                                         a["z"], a["dt_bias"], h0=h0d)
    torch.cuda.synchronize()
    return a, h0d, (out, last, ck), (out0, last0)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d_state", [8, 16, 32, 64])
@pytest.mark.parametrize("L", [1, 16, 17, 100])
def test_ckpt_rows_are_the_prefix_states(dtype, d_state, L):
    """Every row against the oracle; out and last_state as the plain scan."""
    x = synth.scan_inputs(2, L, 48, d_state, dtype=dtype, seed=1200 + d_state + L,
                          D="normal", A_kind="random")
    h0 = np.random.default_rng(L + d_state).standard_normal((2, 48, d_state)).astype(np.float32)
    _, _, (out, last, ck), (out0, last0) = fwd_ckpt(x, h0)
    assert torch.equal(out, out0) and torch.equal(last, last0)
    interval, nbytes = msc.scan_checkpoint_size(2, L, 48, d_state)
    assert interval == (16 if d_state <= 16 else 8)
    assert ck.numel() * 4 == nbytes
    ref = oracle_ckpt_rows(x, h0, interval)
    got = from_device(ck)
    assert np.array_equal(got[:, 0], h0)          # row 0 is h0 itself
    e = rel_l2(got, ref)
    assert e <= TOL[dtype], f"checkpoint rows rel-L2 {e:.3e}"


def test_ckpt_rows_over_time_chunks():
    """Few channels over a long sequence: the forward splits time into
    chunks (several chunk starts fall on checkpoint rows); with no h0 row 0
    is zero."""
    x = synth.scan_inputs(1, 1000, 16, 16, dtype="bf16", seed=1300, D="normal")
    msc.tuning_set("scan_chunks", 5)
    try:
        _, _, (out, last, ck), (out0, last0) = fwd_ckpt(x, None)
    finally:
        msc.tuning_set("scan_chunks", 0)
    got = from_device(ck)
    assert np.all(got[:, 0] == 0.0)
    e = rel_l2(got, oracle_ckpt_rows(x, None, 16))
    assert e <= TOL["bf16"], f"checkpoint rows rel-L2 {e:.3e}"


def bwd_pair(x, h0, seed, chunks=1):
    rng = np.random.default_rng(seed)
    dout = rng.standard_normal(x.u.shape).astype(np.float32)
    if x.dtype == "bf16":
        dout = synth.round_bf16(dout)
    dl = rng.standard_normal((x.u.shape[0], x.u.shape[2], x.B.shape[-1])).astype(np.float32)
    msc.tuning_set("scan_chunks", chunks)
    try:
        a, h0d, (_, _, ck), _ = fwd_ckpt(x, h0)
    finally:
        msc.tuning_set("scan_chunks", 0)
    kw = dict(h0=h0d, dout=to_device(dout, x.dtype), dlast_state=to_device(dl, "f32"),
              want_dh0=True)
    args = (a["u"], a["dt"], a["A"], a["B"], a["C"], a["D"], a["z"], a["dt_bias"])
    g_ck = msc.selective_scan_bwd(*args, ckpt=ck, **kw)
    g_re = msc.selective_scan_bwd(*args, **kw)
    torch.cuda.synchronize()
    return g_ck, g_re, dout, dl


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d_state", [8, 16, 32, 64])
@pytest.mark.parametrize("L", [1, 15, 16, 40, 257])
def test_bwd_from_ckpt_equals_recompute(dtype, d_state, L):
    """One time chunk: the rows are the backward's own recomputed states."""
    x = synth.scan_inputs(2, L, 48, d_state, dtype=dtype, seed=1400 + d_state + L,
                          D="normal", A_kind="random")
    h0 = np.random.default_rng(L).standard_normal((2, 48, d_state)).astype(np.float32)
    g_ck, g_re, _, _ = bwd_pair(x, h0, seed=L)
    for k in ("du", "ddt", "dz", "dh0"):
        assert torch.equal(g_ck[k], g_re[k]), k
    for k in ("dA", "dB", "dC", "dD", "ddt_bias"):
        e = rel_l2(from_device(g_ck[k]), from_device(g_re[k]).astype(np.float64))
        assert e <= 1e-6, f"{k} rel-L2 {e:.3e}"


@pytest.mark.parametrize("chunks", [1, 3])
def test_bwd_from_ckpt_against_oracle(chunks):
    """Both backward forms against the oracle's adjoint, the forward in one
    time chunk or three."""
    x = synth.scan_inputs(2, 300, 64, 16, dtype="bf16", seed=1500 + chunks, D="normal")
    h0 = np.random.default_rng(21).standard_normal((2, 64, 16)).astype(np.float32)
    g_ck, g_re, dout, dl = bwd_pair(x, h0, seed=22, chunks=chunks)
    ref = oracle.scan_bwd(x.u, x.dt_raw, x.A, x.B, x.C, x.D, x.z, x.dt_bias, h0,
                          dout=dout, dlast=dl)
    for g in (g_ck, g_re):
        for k in ("du", "ddt", "dz"):
            e = rel_l2(from_device(g[k]), as_stored(ref[k], "bf16"))
            assert e <= TOL["bf16"], f"{k} rel-L2 {e:.3e}"
        for k in ("dA", "dB", "dC", "dD", "ddt_bias", "dh0"):
            e = rel_l2(from_device(g[k]), ref[k])
            assert e <= SUM_TOL, f"{k} rel-L2 {e:.3e}"


def test_ckpt_workload_layer_sampled():
    """The 8 x 2048 x 1536 x 16 layer at full size: checkpointing forward as
    the plain one bit for bit, the backward from checkpoints as the
    recomputing backward bit for bit (du, ddt, dz), and sampled checkpoint
    rows against the oracle on a few channels."""
    x = synth.workload_inputs("mamba130m_layer")
    a, _, (out, last, ck), (out0, last0) = fwd_ckpt(x, None)
    assert torch.equal(out, out0) and torch.equal(last, last0)
    rng = np.random.default_rng(23)
    dout = to_device(synth.round_bf16(rng.standard_normal(x.u.shape).astype(np.float32)),
                     "bf16")
    args = (a["u"], a["dt"], a["A"], a["B"], a["C"], a["D"], a["z"], a["dt_bias"])
    g_ck = msc.selective_scan_bwd(*args, ckpt=ck, dout=dout)
    g_re = msc.selective_scan_bwd(*args, dout=dout)
    torch.cuda.synchronize()
    for k in ("du", "ddt", "dz"):
        assert torch.equal(g_ck[k], g_re[k]), k
    ch = np.array([0, 1, 777, 1535])
    sub = dataclasses.replace(x, u=x.u[:1, :, ch], dt_raw=x.dt_raw[:1, :, ch],
                              z=x.z[:1, :, ch], B=x.B[:1], C=x.C[:1], A=x.A[ch], D=x.D[ch],
                              dt_bias=x.dt_bias[ch])
    ref = oracle_ckpt_rows(sub, None, 16)
    got = from_device(ck)[:1, :, ch]
    e = rel_l2(got, ref)
    assert e <= TOL["bf16"], f"checkpoint rows rel-L2 {e:.3e}"


def test_ckpt_unsupported_shapes_are_refused():
    """Shapes without the TMA kernels (d_inner not a multiple of 8, d_state
    outside 8/16/32/64) are refused by the checkpointing entry points -- the
    recomputing backward covers them -- and nothing is launched."""
    x = synth.scan_inputs(2, 40, 12, 16, dtype="bf16", seed=1600)
    a = scan_device_args(x)
    with pytest.raises(msc.MscError) as e:
        msc.selective_scan_fwd_ckpt(a["u"], a["dt"], a["A"], a["B"], a["C"], a["D"], a["z"],
                                    a["dt_bias"], ckpt=torch.empty(2, 3, 12, 16, device="cuda"))
    assert e.value.status == 2
    x = synth.scan_inputs(2, 40, 16, 12, dtype="bf16", seed=1601)
    with pytest.raises(msc.MscError) as e:
        msc.scan_checkpoint_size(2, 40, 16, 12)
    assert e.value.status == 2
    torch.cuda.synchronize()
    msc.check_device_error()


def test_ckpt_empty_and_single_step():
    """L = 0 writes nothing and returns last_state = h0; L = 1 is one row,
    h0 itself, and the backward from it matches the recomputing one."""
    h0 = np.random.default_rng(31).standard_normal((2, 16, 16)).astype(np.float32)
    x0 = synth.scan_inputs(2, 0, 16, 16, dtype="bf16", seed=1602)
    a0 = scan_device_args(x0)
    out, last, ck = msc.selective_scan_fwd_ckpt(a0["u"], a0["dt"], a0["A"], a0["B"], a0["C"],
                                                a0["D"], a0["z"], a0["dt_bias"],
                                                h0=to_device(h0, "f32"))
    torch.cuda.synchronize()
    assert ck.numel() == 0 and np.array_equal(from_device(last), h0)
    x1 = synth.scan_inputs(2, 1, 16, 16, dtype="bf16", seed=1603, D="normal")
    g_ck, g_re, _, _ = bwd_pair(x1, h0, seed=32)
    for k in ("du", "ddt", "dz", "dh0"):
        assert torch.equal(g_ck[k], g_re[k]), k


@pytest.mark.parametrize("d_state", [8, 16, 32])
def test_ckpt_rows_two_lanes_per_channel(d_state):
    """The TMA kernels with two lanes per channel (more states per lane)
    write the same checkpoint layout."""
    x = synth.scan_inputs(2, 100, 64, d_state, dtype="bf16", seed=1700 + d_state,
                          D="normal", A_kind="random")
    h0 = np.random.default_rng(d_state).standard_normal((2, 64, d_state)).astype(np.float32)
    msc.tuning_set("scan_lanes", 2)
    try:
        _, _, (out, last, ck), (out0, last0) = fwd_ckpt(x, h0)
    finally:
        msc.tuning_set("scan_lanes", 0)
    assert torch.equal(out, out0) and torch.equal(last, last0)
    interval, _ = msc.scan_checkpoint_size(2, 100, 64, d_state)
    e = rel_l2(from_device(ck), oracle_ckpt_rows(x, h0, interval))
    assert e <= TOL["bf16"], f"checkpoint rows rel-L2 {e:.3e}"


@pytest.mark.parametrize("d_inner", [64, 12])
def test_autograd_selective_scan_matches_direct_calls(d_inner):
    """selective_scan under torch autograd: the forward and the gradients
    equal the direct calls bit for bit (d_inner 64: checkpoints kept by the
    forward; 12: no TMA kernels, the plain forward and the recomputing
    backward)."""
    x = synth.scan_inputs(2, 70, d_inner, 16, dtype="bf16", seed=1800 + d_inner, D="normal")
    a = scan_device_args(x)
    h0 = to_device(np.random.default_rng(41).standard_normal((2, d_inner, 16))
                   .astype(np.float32), "f32")
    leaves = {k: a[k].clone().requires_grad_(True) for k in a}
    h0l = h0.clone().requires_grad_(True)
    rng = np.random.default_rng(42)
    W = to_device(synth.round_bf16(rng.standard_normal(x.u.shape).astype(np.float32)), "bf16")
    V = to_device(rng.standard_normal((2, d_inner, 16)).astype(np.float32), "f32")
    msc.tuning_set("scan_chunks", 1)  # one time chunk: checkpoint rows = recomputed states
    try:
        out, last = msc.selective_scan(leaves["u"], leaves["dt"], leaves["A"], leaves["B"],
                                       leaves["C"], leaves["D"], leaves["z"],
                                       leaves["dt_bias"], h0=h0l)
        loss = (out.float() * W.float()).sum() + (last * V).sum()
        loss.backward()
        out0, last0 = msc.selective_scan_fwd(a["u"], a["dt"], a["A"], a["B"], a["C"], a["D"],
                                             a["z"], a["dt_bias"], h0=h0)
    finally:
        msc.tuning_set("scan_chunks", 0)
    # d loss / d out, as autograd hands it over: W in fp32, rounded to out's dtype
    g = msc.selective_scan_bwd(a["u"], a["dt"], a["A"], a["B"], a["C"], a["D"], a["z"],
                               a["dt_bias"], h0=h0, dout=W, dlast_state=V, want_dh0=True)
    torch.cuda.synchronize()
    assert torch.equal(out, out0) and torch.equal(last, last0)
    for k, name in (("du", "u"), ("ddt", "dt"), ("dz", "z")):
        assert torch.equal(leaves[name].grad, g[k]), k
    assert torch.equal(h0l.grad, g["dh0"])
    for k, name in (("dA", "A"), ("dD", "D"), ("ddt_bias", "dt_bias")):
        e = rel_l2(from_device(leaves[name].grad), from_device(g[k]).astype(np.float64))
        assert e <= 1e-6, f"{k} rel-L2 {e:.3e}"
    for k, name in (("dB", "B"), ("dC", "C")):
        e = rel_l2(from_device(leaves[name].grad), from_device(g[k].to(torch.bfloat16)))
        assert e <= 1e-2, f"{k} rel-L2 {e:.3e}"   # bf16 gradients of bf16 inputs


def test_ckpt_forward_with_caller_workspace():
    """msc_selective_scan_fwd_ckpt with a caller workspace (sized by
    msc_selective_scan_workspace_size, filled with garbage) gives the same
    out, last_state and checkpoints as with library scratch."""
    x = synth.scan_inputs(1, 700, 64, 16, dtype="bf16", seed=1900, D="normal")
    a = scan_device_args(x)
    msc.tuning_set("scan_chunks", 3)  # time chunks: the workspace holds their carries
    try:
        out0, last0, ck0 = msc.selective_scan_fwd_ckpt(a["u"], a["dt"], a["A"], a["B"], a["C"],
                                                       a["D"], a["z"], a["dt_bias"])
        n = msc.scan_workspace_size(1, 700, 64, 16, torch.bfloat16)
        ws = torch.randint(0, 255, (max(n, 1),), dtype=torch.uint8, device="cuda")
        out = torch.empty_like(out0)
        last = torch.empty_like(last0)
        ck = torch.empty_like(ck0)
        P = lambda t: None if t is None else t.data_ptr()
        st = msc.load().msc_selective_scan_fwd_ckpt(
            P(a["u"]), P(a["dt"]), P(a["A"]), P(a["B"]), P(a["C"]), P(a["D"]), P(a["z"]),
            P(a["dt_bias"]), None, P(out), P(last), P(ck), 1, 700, 64, 16, 1, P(ws), n,
            torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
    finally:
        msc.tuning_set("scan_chunks", 0)
    assert st == 0
    assert torch.equal(out, out0) and torch.equal(last, last0) and torch.equal(ck, ck0)
