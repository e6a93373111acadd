"""GPU parity on the full-size workloads, whole tensors against the fp64 oracle.

  * the three scan workloads (the Mamba-130M-like layer 8 x 2048 x 1536 x 16,
    the 64K-step sequence 1 x 65536 x 2048 x 16, the Mamba-2.8B-like layer
    4 x 4096 x 5120 x 16; bf16 storage, fp32 state): every output element and
    the whole last state, in the launch configuration the bench times;
  * the decode workload as it is defined: 1000 sequential single-token steps
    at 256 x 5120 x 16 with the fp32 state resident and updated in place from
    its N(0, 1) initial state, every step's output and the final state
    compared on sampled channels (every batch row, every step) -- the state
    of a channel depends only on that channel's inputs and the shared B, C,
    so the oracle advances the sampled channels alone;
  * the backward pass on the Mamba-130M-like layer: every gradient whole.

Tolerances are the parity tolerances of the other tests (rel-L2 over a whole
tensor <= 2e-3 for bf16 storage against the oracle rounded to bf16; the fp32
sums of the backward <= 2e-5).  Per-batch-row rel-L2 is checked as well, so a
wrong batch row cannot hide in the norm of the others."""
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest

import oracle
import selective_state_space_144_b300 as msc
from selective_state_space_144_b300 import synth
from tests.helpers import TOL, as_stored, from_device, rel_l2, scan_device_args, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _defaults():
    for key, v in (("scan_chunks", 0), ("scan_min_chunk", 512), ("scan_path", 0),
                   ("scan_lanes", 0)):
        msc.tuning_set(key, v)
    yield
    torch.cuda.synchronize()
    msc.check_device_error()


def _rows_rel(got, ref):
    return max(rel_l2(got[b], ref[b]) for b in range(got.shape[0]))


@pytest.mark.parametrize("name", ["mamba130m_layer", "long_seq_64k", "mamba2p8b_layer"])
def test_scan_workload_whole_tensor(name):
    x = synth.workload_inputs(name)
    a = scan_device_args(x)
    batch, L, d_inner = x.u.shape
    N = x.B.shape[-1]
    out = torch.full((batch, L, d_inner), float("nan"), dtype=torch.bfloat16, device="cuda")
    last = torch.full((batch, d_inner, N), float("nan"), device="cuda")
    nws = msc.scan_workspace_size(batch, L, d_inner, N, torch.bfloat16)
    wsp = torch.empty(max(nws, 1), dtype=torch.uint8, device="cuda")
    msc.selective_scan_fwd_ws(**a, out=out, last_state=last, workspace=wsp)
    torch.cuda.synchronize()
    del a, wsp
    y = from_device(out)
    s = from_device(last)
    del out, last
    torch.cuda.empty_cache()
    y_ref, s_ref = oracle.scan_fwd(x.u, x.dt_raw, x.A, x.B, x.C, x.D, x.z, x.dt_bias)
    y_ref = as_stored(y_ref, "bf16")
    assert np.all(np.isfinite(y)) and np.all(np.isfinite(s))
    tol = TOL["bf16"]
    e_y, e_s = rel_l2(y, y_ref), rel_l2(s, s_ref)
    assert e_y <= tol, f"out rel-L2 {e_y:.3e}"
    assert e_s <= tol, f"last_state rel-L2 {e_s:.3e}"
    assert _rows_rel(y, y_ref) <= tol
    assert _rows_rel(s, s_ref) <= tol


def test_decode_workload_1000_steps():
    """Every one of the 1000 steps' outputs (not a subset) against the oracle,
    on sampled channels: the oracle's outputs are kept for all steps."""
    w = synth.WORKLOADS["decode_256x5120"]
    batch, d_inner, N, steps = w["batch"], w["d_inner"], w["d_state"], w["steps"]
    p = synth.decode_params(batch, d_inner, N)
    sel = np.sort(np.random.default_rng(6).choice(d_inner, 64, replace=False))
    sel_d = torch.from_numpy(sel).cuda()
    state = torch.from_numpy(p.state0).cuda()
    A, D, bias = to_device(p.A, "f32"), to_device(p.D, "f32"), to_device(p.dt_bias, "f32")
    out = torch.empty(batch, d_inner, dtype=torch.bfloat16, device="cuda")
    got_out = torch.empty(steps, batch, len(sel), dtype=torch.bfloat16, device="cuda")
    ref_out = np.empty((steps, batch, len(sel)))
    ref_state = p.state0[:, sel].astype(np.float64)
    with ThreadPoolExecutor(max_workers=8) as pool:
        futs = [pool.submit(synth.decode_step, batch, d_inner, N, k) for k in range(min(16, steps))]
        for k in range(steps):
            s = futs[k].result()
            if k + 16 < steps:
                futs.append(pool.submit(synth.decode_step, batch, d_inner, N, k + 16))
            futs[k] = None
            msc.selective_state_update(state, to_device(s.u, "bf16"), to_device(s.dt_raw, "bf16"),
                                       A, to_device(s.B, "bf16"), to_device(s.C, "bf16"), D,
                                       to_device(s.z, "bf16"), bias, out=out)
            got_out[k].copy_(out.index_select(1, sel_d))
            ref_state, y = oracle.state_update(
                ref_state, s.u[:, sel], s.dt_raw[:, sel], p.A[sel], s.B, s.C, p.D[sel],
                s.z[:, sel], p.dt_bias[sel])
            ref_out[k] = as_stored(y, "bf16")
    torch.cuda.synchronize()
    got = from_device(got_out)
    assert np.all(np.isfinite(got))
    per_step = [rel_l2(got[k], ref_out[k]) for k in range(steps)]
    k = int(np.argmax(per_step))
    assert per_step[k] <= TOL["bf16"], f"step {k}: out rel-L2 {per_step[k]:.3e}"
    assert rel_l2(got, ref_out) <= TOL["bf16"]
    assert rel_l2(from_device(state)[:, sel], ref_state) <= TOL["bf16"]


@pytest.mark.parametrize("name,from_ckpt", [("mamba130m_layer", False),
                                            ("mamba130m_layer", True),
                                            ("mamba2p8b_layer", True)])
def test_backward_workload_whole_tensors(name, from_ckpt):
    """The backward on the 8 x 2048 x 1536 x 16 layer (the size the bench
    times) and on the 4 x 4096 x 5120 x 16 layer: every gradient of every
    input, whole -- recomputing its checkpoints, or from the ones the
    checkpointing forward wrote (the training path)."""
    x = synth.workload_inputs(name)
    rng = np.random.default_rng(14)
    dout = synth.round_bf16(rng.standard_normal(x.u.shape).astype(np.float32))
    a = scan_device_args(x)
    ck = None
    if from_ckpt:
        ck = msc.selective_scan_fwd_ckpt(a["u"], a["dt"], a["A"], a["B"], a["C"], a["D"],
                                         a["z"], a["dt_bias"])[2]
    g = msc.selective_scan_bwd(a["u"], a["dt"], a["A"], a["B"], a["C"], a["D"], a["z"],
                               a["dt_bias"], dout=to_device(dout, "bf16"), want_dh0=True,
                               ckpt=ck)
    del ck
    torch.cuda.synchronize()
    got = {k: (None if v is None else from_device(v)) for k, v in g.items()}
    del a, g
    torch.cuda.empty_cache()
    ref = oracle.scan_bwd(x.u, x.dt_raw, x.A, x.B, x.C, x.D, x.z, x.dt_bias, None,
                          dout=dout, dlast=None)
    for k in ("du", "ddt", "dz"):
        r = as_stored(ref[k], "bf16")
        assert np.all(np.isfinite(got[k])), k
        e = rel_l2(got[k], r)
        assert e <= TOL["bf16"], f"{k} rel-L2 {e:.3e}"
        assert _rows_rel(got[k], r) <= TOL["bf16"], k
    for k in ("dA", "dB", "dC", "dD", "ddt_bias", "dh0"):
        e = rel_l2(got[k], ref[k])
        assert e <= 2e-5, f"{k} rel-L2 {e:.3e}"


def test_bench_step_graph_replay_bitwise():
    """The bench's timed step -- the 130M-like layer's scan with a caller
    workspace, then one decode token from its last state -- replayed from a
    CUDA graph gives the eager step's outputs bit for bit (so the graph-timed
    launches compute what the whole-tensor test above checked)."""
    x = synth.workload_inputs("mamba130m_layer")
    a = scan_device_args(x)
    batch, L, d_inner = x.u.shape
    N = x.B.shape[-1]
    tok = synth.decode_step(batch, d_inner, N, 0, seed=11)
    t = {k: to_device(getattr(tok, k), "bf16") for k in ("u", "dt_raw", "z", "B", "C")}
    nws = msc.scan_workspace_size(batch, L, d_inner, N, torch.bfloat16)
    wsp = torch.empty(max(nws, 1), dtype=torch.uint8, device="cuda")
    out = torch.empty(batch, L, d_inner, dtype=torch.bfloat16, device="cuda")
    last = torch.empty(batch, d_inner, N, device="cuda")
    tout = torch.empty(batch, d_inner, dtype=torch.bfloat16, device="cuda")

    def step():
        msc.selective_scan_fwd_ws(**a, out=out, last_state=last, workspace=wsp)
        msc.selective_state_update(last, t["u"], t["dt_raw"], a["A"], t["B"], t["C"], a["D"],
                                   t["z"], a["dt_bias"], out=tout)

    step()
    torch.cuda.synchronize()
    ref = (out.clone(), last.clone(), tout.clone())
    for buf in (out, last, tout):
        buf.fill_(float("nan"))
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for buf in (out, last, tout):
        buf.fill_(float("nan"))
    graph.replay()
    torch.cuda.synchronize()
    for got, want in zip((out, last, tout), ref):
        assert torch.equal(got.view(torch.int16) if got.dtype == torch.bfloat16 else got,
                           want.view(torch.int16) if want.dtype == torch.bfloat16 else want)
