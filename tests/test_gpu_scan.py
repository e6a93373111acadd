"""GPU parity of the selective scan forward against the fp64 oracle.

Every case draws seeded inputs (selective_state_space_144_b300.synth), runs
the sm_103a kernels through the C ABI, and compares element by element with
the oracle on the same inputs: rel-L2 <= 1e-5 for fp32 storage and <= 2e-3
for bf16 storage (oracle output rounded to bf16), for out and last_state.
Outputs are poisoned with NaN first so an unwritten element fails.
"""
import numpy as np
import pytest

import oracle
import selective_state_space_144_b300 as msc
from selective_state_space_144_b300 import synth
from tests.helpers import TOL, as_stored, from_device, rel_l2, scan_device_args

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
    msc.check_device_error()      # no bounded wait gave up during the test
    _defaults()


# 0: automatic (the TMA kernels where the shape allows), 1: element-load kernels
PATHS = [0, 1]
# lanes per channel of the TMA kernels: 4 (N/4 states each) or 2 (N/2 each)
LANES = [4, 2]


def run_gpu(x, chunks=0, with_last=True, path=0, lanes=0):
    msc.tuning_set("scan_path", path)
    msc.tuning_set("scan_lanes", lanes)
    if chunks:
        msc.tuning_set("scan_chunks", chunks)
    a = scan_device_args(x)
    batch, L, d_inner, d_state = x.u.shape + (x.B.shape[-1],)
    out = torch.full((batch, L, d_inner), float("nan"), dtype=a["u"].dtype,
                     device="cuda")
    last = (torch.full((batch, d_inner, d_state), float("nan"),
                       dtype=torch.float32, device="cuda") if with_last else None)
    msc.selective_scan_fwd(a["u"], a["dt"], a["A"], a["B"], a["C"], a["D"],
                           a["z"], a["dt_bias"], out=out, last_state=last,
                           return_last_state=with_last)
    torch.cuda.synchronize()
    return from_device(out), (from_device(last) if with_last else None)


def check(x, chunks=0, with_last=True, path=0, lanes=0):
    y, last = run_gpu(x, chunks, with_last, path, lanes)
    y_ref, last_ref = oracle.scan_fwd(x.u, x.dt_raw, x.A, x.B, x.C, x.D, x.z,
                                      x.dt_bias)
    tol = TOL[x.dtype]
    assert np.all(np.isfinite(y)), "unwritten or non-finite output"
    e_y = rel_l2(y, as_stored(y_ref, x.dtype))
    assert e_y <= tol, f"out rel-L2 {e_y:.3e} > {tol}"
    if with_last:
        assert np.all(np.isfinite(last))
        e_s = rel_l2(last, last_ref)
        assert e_s <= tol, f"last_state rel-L2 {e_s:.3e} > {tol}"
    return e_y


def test_tiny_f32_workload():
    """The 1 x 64 x 8 x 4 fp32 oracle-check workload, at full size."""
    x = synth.workload_inputs("tiny_f32")
    check(x)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d_state", [1, 2, 3, 4, 5, 8, 12, 16, 24, 32, 33, 64])
@pytest.mark.parametrize("d_inner", [45, 64])
def test_state_sizes(dtype, d_state, d_inner):
    """d_inner = 64 takes the TMA kernels for d_state in {8, 16, 32, 64};
    45 channels (not a multiple of 8) and other d_state take the
    element-load kernels."""
    x = synth.scan_inputs(2, 77, d_inner, d_state, dtype=dtype,
                          seed=100 + d_state, D="normal", A_kind="random")
    check(x)


@pytest.mark.parametrize("lanes", LANES)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d_state", [8, 16, 32, 64])
def test_tma_lane_splits(dtype, d_state, lanes):
    """Both lane splits of the TMA kernels (2 lanes per channel is taken for
    d_state <= 32 only), 3 chunks, ragged tail."""
    x = synth.scan_inputs(2, 333, 96, d_state, dtype=dtype,
                          seed=200 + d_state, D="normal", A_kind="random")
    check(x, chunks=3, lanes=lanes)


@pytest.mark.parametrize("path,lanes", [(0, 4), (0, 2), (1, 0)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("chunks", [1, 2, 3, 7, 64])
def test_chunked_carry(dtype, chunks, path, lanes):
    """Time cut into chunks joined by the carry pass, ragged last chunk."""
    x = synth.scan_inputs(3, 517, 208, 16, dtype=dtype, seed=7 + chunks,
                          D="normal")
    check(x, chunks=chunks, path=path, lanes=lanes)


@pytest.mark.parametrize("lanes", LANES)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_chunk_summary_stops_early(dtype, lanes):
    """Large step sizes (delta ~ 3) make the product of later decays fall
    below 2^-40 within a few steps, so the backward chunk summary stops
    early; the carries must still be exact to fp32."""
    x = synth.scan_inputs(2, 1024, 64, 16, dtype=dtype, seed=51, D="normal")
    x.dt_raw = synth.round_bf16(x.dt_raw + 3.0) if dtype == "bf16" else x.dt_raw + 3.0
    check(x, chunks=4, lanes=lanes)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_chunk_summary_growing_state(dtype):
    """A > 0: the decays exceed 1, the later-decay product grows and the
    backward summary walks every step of every chunk."""
    x = synth.scan_inputs(2, 640, 64, 16, dtype=dtype, seed=52, D="normal")
    x.A = np.full_like(x.A, 0.02)
    check(x, chunks=5)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_tma_path_is_taken(dtype):
    """Aligned 16-state shapes run the TMA kernels: for bf16 a B/C
    conversion kernel plus the scan kernel, for fp32 the scan kernel alone
    (the element-load kernels would launch one)."""
    x = synth.scan_inputs(2, 256, 64, 16, dtype=dtype, seed=31)
    msc.tuning_set("scan_chunks", 1)
    msc.profile_read()
    msc.profile_enable(True)
    try:
        check(x, chunks=1)
        launches, kinds = msc.profile_read()
    finally:
        msc.profile_enable(False)
    timed, ms = kinds["scan"]
    assert timed == 1 and ms > 0.0 and kinds["update"][0] == 0
    assert launches == (2 if dtype == "bf16" else 1)


@pytest.mark.parametrize("d_inner,lanes", [(33, 0), (40, 4), (48, 2)])
@pytest.mark.parametrize("L", [1, 2, 5, 7, 8, 9, 31, 32, 33, 129])
def test_short_sequences(L, d_inner, lanes):
    x = synth.scan_inputs(2, L, d_inner, 16, dtype="f32", seed=L)
    check(x, lanes=lanes)
    check(x, chunks=L, lanes=lanes)   # one step (or one tile) per chunk


@pytest.mark.parametrize("path", PATHS)
def test_empty_sequence_zeroes_last_state(path):
    x = synth.scan_inputs(2, 0, 40, 16, dtype="bf16", seed=1)
    y, last = run_gpu(x, path=path)
    assert y.size == 0
    assert np.all(last == 0.0)


@pytest.mark.parametrize("d_inner", [70, 72])
@pytest.mark.parametrize("drop", ["z", "D", "dt_bias", "all"])
def test_optional_inputs_absent(drop, d_inner):
    x = synth.scan_inputs(2, 300, d_inner, 16, dtype="f32", seed=3, D="normal")
    if drop in ("z", "all"):
        x.z = None
    if drop in ("D", "all"):
        x.D = None
    if drop in ("dt_bias", "all"):
        x.dt_bias = None
    check(x)


def test_no_last_state():
    x = synth.scan_inputs(2, 200, 64, 16, dtype="bf16", seed=4)
    check(x, with_last=False)


def test_unaligned_pointers_take_element_loads():
    """Views starting one element into their storage: 2-byte-aligned bf16
    pointers that the 4-wide loads cannot use."""
    x = synth.scan_inputs(2, 150, 48, 16, dtype="bf16", seed=5)
    a = scan_device_args(x)
    def shifted(t):
        flat = torch.empty(t.numel() + 1, dtype=t.dtype, device="cuda")
        v = flat[1:].view(t.shape)
        v.copy_(t)
        return v
    args = {k: (shifted(v) if k in ("u", "dt", "B", "C", "z") else v)
            for k, v in a.items()}
    out, last = msc.selective_scan_fwd(**args)
    torch.cuda.synchronize()
    y_ref, last_ref = oracle.scan_fwd(x.u, x.dt_raw, x.A, x.B, x.C, x.D, x.z,
                                      x.dt_bias)
    assert rel_l2(from_device(out), as_stored(y_ref, "bf16")) <= TOL["bf16"]
    assert rel_l2(from_device(last), last_ref) <= TOL["bf16"]


def test_auto_plan_many_chunks():
    """Few channels and a long sequence: the automatic plan cuts time."""
    msc.tuning_set("scan_min_chunk", 64)
    x = synth.scan_inputs(1, 4096, 64, 16, dtype="bf16", seed=6)
    assert msc.scan_workspace_size(1, 4096, 64, 16, torch.bfloat16) > 0
    check(x)


def test_caller_workspace_variant():
    msc.tuning_set("scan_chunks", 5)
    x = synth.scan_inputs(2, 600, 96, 16, dtype="f32", seed=8)
    a = scan_device_args(x)
    n = msc.scan_workspace_size(2, 600, 96, 16, torch.float32)
    assert n > 0
    ws = torch.full((n,), 255, dtype=torch.uint8, device="cuda")   # garbage
    out, last = msc.selective_scan_fwd_ws(**a, workspace=ws)
    torch.cuda.synchronize()
    y_ref, last_ref = oracle.scan_fwd(x.u, x.dt_raw, x.A, x.B, x.C, x.D, x.z,
                                      x.dt_bias)
    assert rel_l2(from_device(out), y_ref) <= TOL["f32"]
    assert rel_l2(from_device(last), last_ref) <= TOL["f32"]


@pytest.mark.parametrize("path", PATHS)
def test_repeatable_bitwise(path):
    x = synth.scan_inputs(2, 700, 128, 16, dtype="bf16", seed=9)
    y1, l1 = run_gpu(x, chunks=3, path=path)
    y2, l2 = run_gpu(x, chunks=3, path=path)
    assert np.array_equal(y1, y2) and np.array_equal(l1, l2)


def test_paths_agree():
    """TMA (both lane splits) and element-load kernels compute the same
    recurrence; they may differ only by fp32 rounding."""
    x = synth.scan_inputs(2, 900, 64, 16, dtype="f32", seed=10, D="normal")
    y0, l0 = run_gpu(x, chunks=2, path=0, lanes=4)
    y1, l1 = run_gpu(x, chunks=2, path=1)
    y2, l2 = run_gpu(x, chunks=2, path=0, lanes=2)
    assert rel_l2(y0, y1) <= 1e-6 and rel_l2(l0, l1) <= 1e-6
    assert rel_l2(y2, y1) <= 1e-6 and rel_l2(l2, l1) <= 1e-6


# ---- the workloads at reduced size (several tiles, ragged tails) ---------
@pytest.mark.parametrize("name,over", [
    ("mamba130m_layer", dict(batch=2, L=300, d_inner=200)),
    ("long_seq_64k", dict(L=5000, d_inner=136)),
    ("mamba2p8b_layer", dict(batch=2, L=400, d_inner=330)),
])
def test_workloads_reduced(name, over):
    x = synth.workload_inputs(name, **over)
    check(x)


# ---- the workloads at full size: sampled channels, every time step -------
def _sampled_check(x, n_channels=24, seed=0):
    y, last = run_gpu(x)
    batch, L, d_inner = x.u.shape
    rng = np.random.default_rng(seed)
    sel = np.sort(rng.choice(d_inner, size=min(n_channels, d_inner),
                             replace=False))
    y_ref, last_ref = oracle.scan_fwd(
        x.u[:, :, sel], x.dt_raw[:, :, sel], x.A[sel], x.B, x.C,
        None if x.D is None else x.D[sel], None if x.z is None else x.z[:, :, sel],
        None if x.dt_bias is None else x.dt_bias[sel])
    tol = TOL[x.dtype]
    assert np.all(np.isfinite(y))
    assert rel_l2(y[:, :, sel], as_stored(y_ref, x.dtype)) <= tol
    assert rel_l2(last[:, sel], last_ref) <= tol


@pytest.mark.parametrize("name", ["mamba130m_layer", "long_seq_64k",
                                  "mamba2p8b_layer"])
def test_workloads_full_size_sampled(name):
    x = synth.workload_inputs(name)
    _sampled_check(x)
