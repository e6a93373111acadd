"""Failure detection on the GPU without a fault: a bounded wait that runs out.

Every wait of the forward scan's TMA kernels for a data copy gives up after a
fixed number of polls, sets a device word and lets the kernel return early.
The debug key "debug_starve_copies" makes those kernels issue none of their
copies and give up after a few polls, so each wait runs out while nothing is
in flight.  The tests check that msc_check_device_error then reports
MSC_ERR_TIMEOUT, that clearing the word works, that the outputs were not
written, and that the context stays usable: a normal scan right afterwards
matches the fp64 oracle.
"""
import numpy as np
import pytest

import oracle
import selective_state_space_144_b300 as msc
from selective_state_space_144_b300 import synth
from tests.helpers import TOL, as_stored, from_device, rel_l2, scan_device_args, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

MSC_ERR_TIMEOUT = 6


def _reset():
    msc.tuning_set("debug_starve_copies", 0)
    msc.tuning_set("scan_chunks", 0)


@pytest.fixture(autouse=True)
def _clean_state():
    _reset()
    torch.cuda.synchronize()
    msc.load().msc_check_device_error(1)
    yield
    _reset()
    torch.cuda.synchronize()
    msc.load().msc_check_device_error(1)


def _scan(x, out, last):
    a = scan_device_args(x)
    msc.selective_scan_fwd(a["u"], a["dt"], a["A"], a["B"], a["C"], a["D"],
                           a["z"], a["dt_bias"], out=out, last_state=last)
    torch.cuda.synchronize()


@pytest.mark.parametrize("chunks", [1, 2])
def test_starved_waits_report_timeout_and_context_survives(chunks):
    """chunks = 1: the output kernel alone (one CTA); chunks = 2: the chunk
    summary kernel and the output kernel both run out."""
    batch, L, d_inner, N = 1, 64, 8, 16          # one 8-channel tile: one CTA per chunk
    x = synth.scan_inputs(batch, L, d_inner, N, dtype="bf16", seed=77)
    lib = msc.load()
    out = torch.full((batch, L, d_inner), float("nan"), dtype=torch.bfloat16,
                     device="cuda")
    last = torch.full((batch, d_inner, N), float("nan"), device="cuda")

    msc.tuning_set("scan_chunks", chunks)
    msc.tuning_set("debug_starve_copies", 64)
    _scan(x, out, last)
    assert lib.msc_check_device_error(0) == MSC_ERR_TIMEOUT   # read, keep
    assert lib.msc_check_device_error(1) == MSC_ERR_TIMEOUT   # read, clear
    assert lib.msc_check_device_error(0) == 0                 # cleared
    # the kernels returned through the bounded-wait exit: nothing written
    assert torch.isnan(out.float()).all()
    assert torch.isnan(last).all()

    # the context is intact: the same scan without starvation is correct
    msc.tuning_set("debug_starve_copies", 0)
    _scan(x, out, last)
    assert lib.msc_check_device_error(0) == 0
    y_ref, s_ref = oracle.scan_fwd(x.u, x.dt_raw, x.A, x.B, x.C, x.D, x.z,
                                   x.dt_bias)
    got = from_device(out)
    assert np.all(np.isfinite(got))
    assert rel_l2(got, as_stored(y_ref, "bf16")) <= TOL["bf16"]
    assert rel_l2(from_device(last), s_ref) <= TOL["bf16"]


@pytest.mark.parametrize("disc", ["euler", "zoh", "trapezoid"])
def test_starved_decode_reports_timeout_and_context_survives(disc):
    """The streaming decode kernel (d_state 16, aligned arrays; every
    discretisation it takes): its waits run out with no copy issued; the
    state is left untouched; a normal step afterwards matches the oracle."""
    batch, d_inner, N = 2, 256, 16
    p = synth.decode_params(batch, d_inner, N)
    s = synth.decode_step(batch, d_inner, N, 0)
    lib = msc.load()
    dev = {k: to_device(getattr(s, k), "bf16") for k in ("u", "dt_raw", "z", "B", "C")}
    A, D, bias = (to_device(p.A, "f32"), to_device(p.D, "f32"), to_device(p.dt_bias, "f32"))
    lam = synth.round_bf16(np.random.default_rng(5).uniform(0, 1, (batch, d_inner))
                           .astype(np.float32))
    lam_d = to_device(lam, "bf16")
    state = torch.from_numpy(p.state0).cuda()
    out = torch.full((batch, d_inner), float("nan"), dtype=torch.bfloat16, device="cuda")

    def step():
        if disc == "trapezoid":
            msc.selective_state_update_trap(state, None, None, dev["u"], dev["dt_raw"], lam_d,
                                            A, dev["B"], dev["C"], D, dev["z"], bias, out=out)
        else:
            msc.selective_state_update(state, dev["u"], dev["dt_raw"], A, dev["B"], dev["C"],
                                       D, dev["z"], bias, out=out, zoh=disc == "zoh")
        torch.cuda.synchronize()

    msc.tuning_set("debug_starve_copies", 64)
    step()
    assert lib.msc_check_device_error(1) == MSC_ERR_TIMEOUT
    assert lib.msc_check_device_error(0) == 0
    assert torch.isnan(out.float()).all()
    assert torch.equal(state.cpu(), torch.from_numpy(p.state0))

    msc.tuning_set("debug_starve_copies", 0)
    step()
    assert lib.msc_check_device_error(0) == 0
    if disc == "trapezoid":
        ref_state, ref_out = oracle.state_update_trap(p.state0, None, None, s.u, s.dt_raw, lam,
                                                      p.A, s.B, s.C, p.D, s.z, p.dt_bias)
    else:
        ref_state, ref_out = oracle.state_update(p.state0, s.u, s.dt_raw, p.A, s.B, s.C, p.D,
                                                 s.z, p.dt_bias, zoh=disc == "zoh")
    assert rel_l2(from_device(out), as_stored(ref_out, "bf16")) <= TOL["bf16"]
    assert rel_l2(from_device(state), ref_state) <= TOL["bf16"]
