#!/usr/bin/env python3
"""Throughput of the selective scan (S6) and decode step on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

A step is one pass of the whole hot path over one batch of synthetic input:
the fused selective-scan forward over the Mamba-130M-like layer
(batch 8, L 2048, d_inner 1536, d_state 16; bf16 storage, fp32 state),
which produces the outputs and the last state, then one single-token decode
step that continues from that last state.  The metric is state updates per
second, batch*L*d_inner*d_state (+ batch*d_inner*d_state for the decode
token) per step, over all GPUs.  For N > 1 each rank runs its own batch
(weak scaling; no collective on the data path -- the scan shards by batch
row with no exchange), launched by torch.distributed.run.

The JSON line also carries: the roofline of the dominant kernel (the scan's
output kernel, timed live with CUDA events on its launch stream through the
library's measurement hook) against the MUFU ex2 peak measured in this run
and against the measured HBM copy peak; the fp64 CPU oracle timed on a
bounded sample on this host; an end-to-end figure through the Python API
with host buffers (pinned host->device copies of each step's inputs and a
device->host read of its outputs inside the timed region); the SM clocks
sampled by nvidia-smi during the timed region; and the other workloads
(64K-step sequence, 2.8B-like layer, 256 x 5120 decode) measured alone.

--impl reference times the fp64 CPU oracle (the only reference this method
has) on the same workload, a bounded sample per step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from selective_state_space_144_b300 import synth  # noqa: E402

METRIC = ("scan state-updates/s (B·L·D·N) and % of HBM/MUFU "
          "roofline, 1×B300")
UNIT = "state-updates/s"
MAIN = "mamba130m_layer"
L2_BYTES = 126 * 2**20


def parse():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=40)
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="target host time of the CPU-oracle sample")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the other workloads")
    ap.add_argument("--profile", default=None, metavar="WORKLOAD",
                    help="profiling driver: run only the scan (or, for "
                         "decode_256x5120, the decode step; for conv1d_prefill "
                         "/ conv1d_update, the conv; for scan_bwd, the backward "
                         "pass on the 130M layer; for scan_bwd_ckpt, the backward "
                         "from forward-written checkpoints) on WORKLOAD "
                         "--warmup + --steps times, print nothing else "
                         "(for ncu; see profiles/); a scan workload with the "
                         "suffix _zoh or _trapezoid runs that discretisation")
    return ap.parse_args()


# ---------------------------------------------------------------------------
def algorithmic(batch, L, d_inner, N, es=2):
    """Algorithmic work of one scan over (batch, L, d_inner, N): state
    updates, MUFU operations (one ex2 per update; ex2 + lg2 for softplus and
    ex2 + rcp for silu per (step, channel)), and HBM bytes (read u, dt, z,
    B, C, A, D, dt_bias; write out and last_state)."""
    upd = batch * L * d_inner * N
    mufu = upd * (1.0 + 4.0 / N)
    byt = (4 * batch * L * d_inner * es + 2 * batch * L * N * es
           + d_inner * N * 4 + 2 * d_inner * 4 + batch * d_inner * N * 4)
    return upd, mufu, byt


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0}, "fallback"


class ClockSampler:
    """nvidia-smi SM clock / throttle-reason samples during a region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                    "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def kernel_source_hash():
    """Hash of the scan kernels' code (comments and white space removed, so
    that a comment edit keeps the recorded counters valid)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "selective_state_space_144_b300", "csrc")
    for name in ("scan_tma.cu", "msc_device.cuh", "msc_ptx.cuh"):
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        h.update("".join(text.split()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str, field: str = "dram_bytes_per_launch"):
    """A per-launch counter (default: DRAM bytes) of `kernel` on `workload`
    from the committed ncu summary, or None when absent or taken on a
    different kernel source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    r = rec.get(f"{kernel}:{workload}")
    if not r or r.get("source_hash") != kernel_source_hash():
        return None
    return r.get(field)


# ---------------------------------------------------------------------------
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def combine_ranks(elapsed_ms: float, units_per_step: float, steps: int,
                  world: int, device=None) -> tuple[float, float]:
    """Whole-job timing of a weak-scaling run: the slowest rank's elapsed
    time (all_reduce MAX over the default process group when world > 1) and
    the throughput of all ranks' units over it."""
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([elapsed_ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        elapsed_ms = float(t.item())
    return elapsed_ms, units_per_step * steps * world / (elapsed_ms * 1e-3)


def cpu_oracle_sample(name: str, target_s: float, max_channels=None):
    """Time the fp64 oracle on a channel subset of workload `name` (every
    batch row, every step) sized to about `target_s` seconds of host time.
    Returns (updates/s, cores, description)."""
    import oracle
    w = synth.WORKLOADS[name]
    x = synth.workload_inputs(name, d_inner=64)
    cores = oracle.threads()
    # calibrate on 8 channels, then size the sample
    sel = np.arange(8)
    t0 = time.perf_counter()
    oracle.scan_fwd(x.u[:, :, sel], x.dt_raw[:, :, sel], x.A[sel], x.B, x.C,
                    x.D[sel], x.z[:, :, sel], x.dt_bias[sel])
    dt = time.perf_counter() - t0
    per_ch = max(dt / 8, 1e-6)
    nch = int(min(max(target_s / per_ch, 8), max_channels or w["d_inner"]))
    x = synth.workload_inputs(name, d_inner=nch)
    t0 = time.perf_counter()
    oracle.scan_fwd(x.u, x.dt_raw, x.A, x.B, x.C, x.D, x.z, x.dt_bias)
    el = time.perf_counter() - t0
    upd = w["batch"] * w["L"] * nch * w["d_state"]
    desc = (f"{name} restricted to {nch} of {w['d_inner']} channels "
            f"(all {w['batch']} batch rows, all {w['L']} steps): {upd} updates "
            f"in {el:.2f} s")
    return upd / el, cores, desc


# ---------------------------------------------------------------------------
def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    w = synth.WORKLOADS[MAIN]
    cores = oracle.threads()
    # per-step sample sized so that warmup + steps take about a minute
    x = synth.workload_inputs(MAIN, d_inner=8)
    t0 = time.perf_counter()
    oracle.scan_fwd(x.u, x.dt_raw, x.A, x.B, x.C, x.D, x.z, x.dt_bias)
    per_ch = (time.perf_counter() - t0) / 8
    budget = 60.0 / max(args.steps + args.warmup, 1)
    nch = int(max(1, min(w["d_inner"], budget / max(per_ch, 1e-9))))
    x = synth.workload_inputs(MAIN, d_inner=nch)
    run = lambda: oracle.scan_fwd(x.u, x.dt_raw, x.A, x.B, x.C, x.D, x.z,
                                  x.dt_bias)
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    el = time.perf_counter() - t0
    upd = w["batch"] * w["L"] * nch * w["d_state"]
    value = upd * args.steps / el
    sample = (f"each step: {MAIN} restricted to {nch} of {w['d_inner']} "
              f"channels (all batch rows and steps, {upd} updates)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": f"{MAIN}: batch 8, L 2048, d_inner 1536, "
                               "d_state 16 (bf16-rounded inputs)",
                   "parallelism": "host cores (OpenMP over channels)"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
def run_ours(args):
    import torch
    import selective_state_space_144_b300 as msc
    from selective_state_space_144_b300 import build as msc_build
    import ctypes

    ws_n, rank, local = dist_env()
    if ws_n > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    msc_build.build()
    msc.load()

    w = synth.WORKLOADS[MAIN]
    B_, L_, D_, N_ = w["batch"], w["L"], w["d_inner"], w["d_state"]
    x = synth.scan_inputs(B_, L_, D_, N_, dtype="bf16", seed=w["seed"] + 1000 * rank,
                          D=w["D"])
    tok = synth.decode_step(B_, D_, N_, 0, seed=w["seed"] + 1000 * rank)

    def dev_t(arr, kind):
        if kind == "bf16":
            bits = synth.bf16_bits(arr).view(np.int16)
            return torch.from_numpy(bits.copy()).to(dev).view(torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(arr, np.float32)).to(dev)

    u, dt, z = dev_t(x.u, "bf16"), dev_t(x.dt_raw, "bf16"), dev_t(x.z, "bf16")
    Bm, Cm = dev_t(x.B, "bf16"), dev_t(x.C, "bf16")
    A, Dv, bias = dev_t(x.A, "f32"), dev_t(x.D, "f32"), dev_t(x.dt_bias, "f32")
    tu, tdt, tz = dev_t(tok.u, "bf16"), dev_t(tok.dt_raw, "bf16"), dev_t(tok.z, "bf16")
    tB, tC = dev_t(tok.B, "bf16"), dev_t(tok.C, "bf16")
    out = torch.empty_like(u)
    last = torch.empty(B_, D_, N_, dtype=torch.float32, device=dev)
    tout = torch.empty_like(tu)
    nws = msc.scan_workspace_size(B_, L_, D_, N_, torch.bfloat16)
    wsp = torch.empty(max(nws, 1), dtype=torch.uint8, device=dev)

    def step():
        msc.selective_scan_fwd_ws(u, dt, A, Bm, Cm, Dv, z, bias, out=out,
                                  last_state=last, workspace=wsp)
        msc.selective_state_update(last, tu, tdt, A, tB, tC, Dv, tz, bias,
                                   out=tout)

    upd_scan, mufu_scan, bytes_scan = algorithmic(B_, L_, D_, N_)
    upd_step = upd_scan + B_ * D_ * N_

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)

    # MUFU ex2 peak on this GPU now (sustained ~0.4 s), for the roofline; the
    # FP32 FFMA / packed FFMA2 rates for the diagnostic issue bound
    pk = ctypes.CDLL(msc_build.lib_path("libmsc_peaks.so"))
    for fn in ("msc_peak_ex2", "msc_peak_ffma", "msc_peak_ffma2", "msc_peak_scan_core"):
        getattr(pk, fn).restype = ctypes.c_int
        getattr(pk, fn).argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_int64, ctypes.c_void_p,
                                    ctypes.POINTER(ctypes.c_float)]
    pk.msc_peak_copy.restype = ctypes.c_int
    pk.msc_peak_copy.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                 ctypes.c_int, ctypes.c_void_p, ctypes.POINTER(ctypes.c_float)]
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    sink = torch.zeros(4, device=dev)
    msf = ctypes.c_float(0)
    stream = torch.cuda.current_stream(dev).cuda_stream
    iters = 80000
    pk.msc_peak_ex2(sink.data_ptr(), sms * 8, 256, 2000, stream, ctypes.byref(msf))
    pk.msc_peak_ex2(sink.data_ptr(), sms * 8, 256, iters, stream, ctypes.byref(msf))
    ex2_peak = sms * 8 * 256 * iters * 8 / (msf.value * 1e-3)
    pk.msc_peak_ffma(sink.data_ptr(), sms * 8, 256, 2000, stream, ctypes.byref(msf))
    pk.msc_peak_ffma(sink.data_ptr(), sms * 8, 256, iters, stream, ctypes.byref(msf))
    ffma_peak = sms * 8 * 256 * iters * 8 / (msf.value * 1e-3)          # fp32 FMA/s
    pk.msc_peak_ffma2(sink.data_ptr(), sms * 8, 256, iters, stream, ctypes.byref(msf))
    ffma2_peak = sms * 8 * 256 * iters * 16 / (msf.value * 1e-3)        # fp32 FMA/s
    # the scan's update arithmetic alone (registers only), 16 warps per SM
    core_iters = 20000
    pk.msc_peak_scan_core(sink.data_ptr(), sms * 4, 128, 500, stream, ctypes.byref(msf))
    pk.msc_peak_scan_core(sink.data_ptr(), sms * 4, 128, core_iters, stream, ctypes.byref(msf))
    core_peak = sms * 4 * 128 * core_iters * 32 / (msf.value * 1e-3)     # updates/s
    # MUFU with 0 and 4 packed FMAs per pair of ex2: how far the pipes overlap
    pk.msc_peak_mufu_fma.restype = ctypes.c_int
    pk.msc_peak_mufu_fma.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_int64, ctypes.c_int, ctypes.c_void_p,
                                     ctypes.POINTER(ctypes.c_float)]
    mix = {}
    for k2 in (0, 4):
        pk.msc_peak_mufu_fma(sink.data_ptr(), sms * 4, 128, 20000, k2, stream, ctypes.byref(msf))
        mix[k2] = sms * 4 * 128 * 20000 * 8 / (msf.value * 1e-3)       # ex2/s
    # the same groups (2 ex2 + their 2 operand FMAs) with packed or scalar
    # FMAs, or the FMAs alone, as SM sub-partition cycles per warp and group
    pk.msc_peak_mix.restype = ctypes.c_int
    pk.msc_peak_mix.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int64,
                                ctypes.c_int, ctypes.c_void_p, ctypes.POINTER(ctypes.c_float)]
    mix_cycles = {}
    mix_names = ("ex2", "ex2 + 2 fma.f32x2", "ex2 + 4 fma.f32x2", "ex2 + 8 fma.f32",
                 "4 fma.f32x2 alone")
    warps_per_smsp = sms * 8 * 256 / 32 / (sms * 4.0)
    for m, mname in enumerate(mix_names):
        pk.msc_peak_mix(sink.data_ptr(), sms * 8, 256, 100, m, stream, ctypes.byref(msf))
        pk.msc_peak_mix(sink.data_ptr(), sms * 8, 256, 20000, m, stream, ctypes.byref(msf))
        mix_cycles[mname] = msf.value   # ms; cycles once the SM clock is known
    # streaming copy of 1 GiB (read + write bytes), the HBM figure of this run
    cp_src = torch.empty(2**28, dtype=torch.float32, device=dev)
    cp_dst = torch.empty_like(cp_src)
    copy_gbs = 0.0
    for _ in range(3):
        pk.msc_peak_copy(cp_dst.data_ptr(), cp_src.data_ptr(), 2**30 // 16, sms * 8, stream,
                         ctypes.byref(msf))
        copy_gbs = max(copy_gbs, 2 * 2**30 / (msf.value * 1e-3) / 1e9)
    del cp_src, cp_dst

    # ---- the step as a CUDA graph -----------------------------------------
    # The scan with a caller workspace and the decode step allocate nothing,
    # so the step (B/C conversion, scan, decode) is captured once and
    # replayed: the timed region then measures the kernels back to back,
    # not the Python and C host path of each call (tens to hundreds of
    # microseconds per call on a busy host, the same order as the kernels).
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream(dev).wait_stream(side)
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(max(3, args.warmup)):
        graph.replay()
    torch.cuda.synchronize(dev)

    # ---- timed region: K steps, nothing else on the path -------------------
    if ws_n > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        e0.record()
        for _ in range(args.steps):
            graph.replay()
        e1.record()
        e1.synchronize()
    if ws_n > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    msc.check_device_error()
    el_ms, value = combine_ranks(e0.elapsed_time(e1), upd_step, args.steps,
                                 ws_n, device=dev)

    # ---- the same K steps as eager calls through the Python API ------------
    torch.cuda.synchronize(dev)
    host_s = 0.0
    e0.record()
    for _ in range(args.steps):
        h0_ = time.perf_counter()
        step()
        host_s += time.perf_counter() - h0_
    e1.record()
    e1.synchronize()
    eager_ms = e0.elapsed_time(e1) / args.steps

    # ---- kernel times, in a separate pass of the same steps ----------------
    # The library's measurement hook brackets each call's main kernel with an
    # event pair on its launch stream and counts the kernels launched; it is
    # kept out of the timed region above so that its event records and host
    # bookkeeping do not stretch the step.
    # Each step is queued behind three reads of 512 MiB (about 0.25 ms of GPU
    # work): the L2 starts cold, and the GPU is busy while the host enqueues
    # the step, so an event pair holds the kernel alone and not the host's
    # launch latency (eager steps are host-bound, and an idle GPU would run
    # the opening event at once).
    lead = torch.ones(128 * 2**20, dtype=torch.float32, device=dev)
    nk = max(3, min(args.steps, 50))
    msc.profile_read()
    msc.profile_enable(True)
    for _ in range(nk):
        for _ in range(3):
            lead.sum()
        step()
    torch.cuda.synchronize(dev)
    del lead
    msc.profile_enable(False)
    launches, kinds = msc.profile_read()
    launches_per_step = launches / nk

    if rank != 0:
        dist.destroy_process_group()
        return 0

    peaks, peak_src = measured_peaks()
    n_scan, ms_scan = kinds["scan"]
    scan_ms = ms_scan / max(n_scan, 1)
    n_upd, ms_upd = kinds["update"]
    upd_ms = ms_upd / max(n_upd, 1)
    achieved_mufu = mufu_scan / (scan_ms * 1e-3)
    hbm = peaks["hbm_gbs"] * 1e9
    traffic = recorded_traffic("scan_tma_kernel", MAIN)
    inst = recorded_traffic("scan_tma_kernel", MAIN, field="warp_instructions_per_launch")
    # issue bound: one warp instruction per clock per SM sub-partition; the
    # FP32 FFMA rate measured above is that rate times 32 lanes
    issue_peak = ffma_peak / 32.0
    packed = recorded_traffic("scan_tma_kernel", MAIN,
                              field="packed_fp32x2_warp_instructions_per_launch")
    mufu_inst = recorded_traffic("scan_tma_kernel", MAIN, field="mufu_warp_instructions_per_launch")
    issue = None
    if inst:
        issue = {"warp_instructions_per_launch": inst,
                 "per_1024_updates": inst / (upd_scan / 1024.0),
                 "issue_peak_warp_instr_per_s": issue_peak,
                 "bound_ms": inst / issue_peak * 1e3,
                 "frac": (inst / issue_peak) / (scan_ms * 1e-3),
                 "source": "warp instructions from an ncu capture of this kernel source "
                           "(profiles/traffic.json); issue rate = measured FFMA rate / 32"}
        if packed and mufu_inst:
            # a packed fp32x2 instruction and an ex2 each hold a sub-partition's
            # dispatch for two cycles (msc_peak_mix), every other instruction one
            disp = inst + packed + mufu_inst
            issue["dispatch_cycles_per_launch"] = disp
            issue["dispatch_bound_ms"] = disp / issue_peak * 1e3
            issue["dispatch_frac"] = (disp / issue_peak) / (scan_ms * 1e-3)
    roofline = {
        "bound": "alu", "kernel": "scan_tma_kernel (output pass)",
        "achieved": achieved_mufu / 1e12, "peak": ex2_peak / 1e12,
        "unit": "Tops/s (MUFU: ex2 per update + ex2,lg2,ex2,rcp per step-channel)",
        "frac": achieved_mufu / ex2_peak,
        "peak_source": ("MUFU ex2 rate measured in this run by libmsc_peaks "
                        f"({sms} SMs x 8 CTAs x 256 threads x 8 chains)"),
        "traffic": traffic,
        "kernel_ms": scan_ms,
        "kernel_timing": (f"mean of {n_scan} launches, event pairs on the launch stream "
                          "in a pass after the timed region, each step queued behind three "
                          "512 MiB reads (L2 cold; host launch latency outside the pair)"),
        "hbm": {"achieved_gbs": bytes_scan / (scan_ms * 1e-3) / 1e9,
                "peak_gbs": peaks["hbm_gbs"], "peak_source": peak_src,
                "frac": bytes_scan / (scan_ms * 1e-3) / hbm,
                "algorithmic_bytes": bytes_scan},
        "diagnostic": {
            "ffma_tflops_measured": ffma_peak * 2 / 1e12,
            "ffma2_tflops_measured": ffma2_peak * 2 / 1e12,
            "update_core_ceiling": {
                "updates_per_s": core_peak,
                "frac_of_mufu_roofline": core_peak * (1.0 + 4.0 / N_) / ex2_peak,
                "achieved_frac": (upd_scan / (scan_ms * 1e-3)) / core_peak,
                "what": ("the scan's per-update instruction mix (mul.f32x2, 2 ex2, mul.f32x2, "
                         "fma.f32x2, fma.f32x2 per state pair) run from registers with no "
                         "memory traffic at 16 warps per SM: the rate MUFU and the FMA pipe "
                         "reach together, the ceiling of the update core"),
            },
            "mufu_fma_overlap": {
                "ex2_per_s_alone": mix[0],
                "ex2_per_s_with_4_ffma2_per_2_ex2": mix[4],
                "cycles_per_warp_group": None,   # filled in once the clock is known
                "cycles_reading": ("per SM sub-partition and warp, a group = 2 ex2 + 2 fma.f32 "
                                   "(+ the listed FMAs); the clock is the SM clock sampled in "
                                   "this run"),
                "what": ("ex2 throughput with only its operand arithmetic, and with four "
                         "packed FMAs per pair of ex2 (the update core's ratio); equal rates "
                         "would mean the FMA work hides under MUFU"),
            },
            "copy_gbs_this_run": copy_gbs,
            "issue": issue,
        },
    }
    step_kernels_ms = scan_ms + upd_ms
    # ---- CPU oracle baseline (rank 0, N = 1) ------------------------------
    cpu = None
    if ws_n == 1:
        v, cores, desc = cpu_oracle_sample(MAIN, args.cpu_seconds)
        cpu = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": desc}

    # ---- end to end through the Python API with host buffers --------------
    pin = lambda t: t.cpu().pin_memory()
    hu, hdt, hz, hB, hC = pin(u), pin(dt), pin(z), pin(Bm), pin(Cm)
    htu, htdt, htz, htB, htC = pin(tu), pin(tdt), pin(tz), pin(tB), pin(tC)
    hout, hlast, htout = pin(out), pin(last), pin(tout)
    h2d = sum(t.numel() * t.element_size()
              for t in (hu, hdt, hz, hB, hC, htu, htdt, htz, htB, htC))
    d2h = sum(t.numel() * t.element_size() for t in (hout, hlast, htout))

    # Two device buffer sets and three streams: the inputs of step k+1 cross
    # the link (host -> device) while step k computes and while the results
    # of step k-1 come back (device -> host; the link is full duplex).  Every
    # step still copies its own inputs from pinned host memory and reads its
    # results back; a set is refilled only after the compute that read it,
    # and its outputs are rewritten only after they reached the host.
    pairs_in = ((u, hu), (dt, hdt), (z, hz), (Bm, hB), (Cm, hC), (tu, htu), (tdt, htdt),
                (tz, htz), (tB, htB), (tC, htC))
    sets = []
    for _ in range(2):
        ins = [torch.empty_like(d_) for d_, _h in pairs_in]
        sets.append({"in": ins, "out": torch.empty_like(out), "last": torch.empty_like(last),
                     "tout": torch.empty_like(tout)})
    s_in, s_cp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_cp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def e2e_step(k):
        S = sets[k % 2]
        with torch.cuda.stream(s_in):
            if k >= 2:
                s_in.wait_event(ev_cp[k % 2])      # step k-2 has read this set
            for d_, (_dd, h_) in zip(S["in"], pairs_in):
                d_.copy_(h_, non_blocking=True)
            ev_in[k % 2].record(s_in)
        with torch.cuda.stream(s_cp):
            s_cp.wait_event(ev_in[k % 2])
            if k >= 2:
                s_cp.wait_event(ev_out[k % 2])     # step k-2's results are home
            su, sdt, sz, sB, sC, stu, stdt, stz, stB, stC = S["in"]
            msc.selective_scan_fwd_ws(su, sdt, A, sB, sC, Dv, sz, bias, out=S["out"],
                                      last_state=S["last"], workspace=wsp)
            msc.selective_state_update(S["last"], stu, stdt, A, stB, stC, Dv, stz, bias,
                                       out=S["tout"])
            ev_cp[k % 2].record(s_cp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_cp[k % 2])
            hout.copy_(S["out"], non_blocking=True)
            hlast.copy_(S["last"], non_blocking=True)
            htout.copy_(S["tout"], non_blocking=True)
            ev_out[k % 2].record(s_out)

    def join_streams():
        cur = torch.cuda.current_stream(dev)
        for st_ in (s_in, s_cp, s_out):
            cur.wait_stream(st_)

    ne = max(1, min(args.e2e_steps, args.steps))
    for st_ in (s_in, s_cp, s_out):
        st_.wait_stream(torch.cuda.current_stream(dev))
    for k in range(3):
        e2e_step(k)
    join_streams()
    torch.cuda.synchronize(dev)
    e0.record()
    for st_ in (s_in, s_cp, s_out):
        st_.wait_stream(torch.cuda.current_stream(dev))
    for k in range(ne):
        e2e_step(k)
    join_streams()
    e1.record()
    e1.synchronize()
    e2e_ms = e0.elapsed_time(e1) / ne
    e2e = {"value": upd_step / (e2e_ms * 1e-3), "unit": UNIT,
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "steps": ne, "ms_per_step": e2e_ms,
           "pipeline": "host->device copies, compute and device->host copies on three "
                       "streams with two device buffer sets"}
    del sets

    extras = {}
    if ws_n == 1 and not args.no_extras:
        del hu, hdt, hz, hB, hC, hout
        extras = run_extras(torch, msc, dev, ex2_peak, peaks)

    clocks = clk.summary()
    mhz = clocks["sm_mhz"] or 2032.0
    roofline["diagnostic"]["mufu_fma_overlap"]["cycles_per_warp_group"] = {
        k: v * 1e-3 * mhz * 1e6 / (warps_per_smsp * 20000 * 4) for k, v in mix_cycles.items()}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws_n,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {
            "workload": (f"{MAIN}: fused selective scan batch {B_}, L {L_}, "
                         f"d_inner {D_}, d_state {N_} (bf16 u/dt/z/B/C, fp32 "
                         "A/D/dt_bias/state) + one decode token from its "
                         "last state"),
            "storage": "bf16", "global_batch": B_ * ws_n, "seq_len": L_,
            "parallelism": f"{ws_n} independent replicas (batch-sharded)",
            "l2": (f"inputs larger than L2: {(4 * B_ * L_ * D_ * 2) / 2**20:.0f}"
                   " MiB of u/dt/z/out streamed per step vs 126 MiB L2"),
        },
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": int(round(launches_per_step * args.steps)),
        "step_timing": {
            "timed": "CUDA-graph replays of the captured step (3 kernels each)",
            "main_kernels_ms_per_step": step_kernels_ms,
            "scan_kernel_ms": scan_ms, "decode_kernel_ms": upd_ms,
            "kernels_per_step": launches_per_step,
            "eager_ms_per_step": eager_ms,
            "eager_host_us_per_step": host_s / args.steps * 1e6,
            "note": ("eager = the same K steps as Python API calls after the timed region, "
                     "host time = perf_counter around each step; kernel times from the "
                     "separate hook pass (the B/C fp32 conversion kernel, a few us, is not "
                     "in the sum)"),
        },
        "clocks": clocks,
        "workloads": extras,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_extras(torch, msc, dev, ex2_peak, peaks):
    """The other workloads, each measured alone: median kernel time of a few
    calls, each after reading a 512 MiB buffer (which leaves L2 holding only
    clean lines of that buffer), via the measurement hook."""
    res = {}
    flush_buf = torch.ones(128 * 2**20, dtype=torch.float32, device=dev)

    def flush():
        # a read, not a write: a written buffer would leave dirty lines in L2
        # that the timed kernel would then pay to write back
        return flush_buf.sum()

    def dev_t(arr, kind):
        if kind == "bf16":
            bits = synth.bf16_bits(arr).view(np.int16)
            return torch.from_numpy(bits.copy()).to(dev).view(torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(arr, np.float32)).to(dev)

    def hook_cold_ms(call, kind, reps=20):
        """Median device time of one launch after an L2 flush, from the event
        pair the library records around its kernel (no host time inside)."""
        ts = []
        for k in range(reps):
            flush()
            torch.cuda.synchronize(dev)
            msc.profile_read()
            msc.profile_enable(True)
            call(k)
            torch.cuda.synchronize(dev)
            msc.profile_enable(False)
            _, kinds = msc.profile_read()
            ts.append(kinds[kind][1])
        return statistics.median(ts)

    def back_to_back_ms(call, n):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        for k in range(10):
            call(k)
        torch.cuda.synchronize(dev)
        e0.record()
        for k in range(n):
            call(k)
        e1.record()
        e1.synchronize()
        return e0.elapsed_time(e1) / n

    # causal conv1d (+ SiLU) before the scan: prefill on the layer's shape,
    # and the decode token on the decode shape; d_conv 4, bf16
    rng = np.random.default_rng(12)
    Bc, Lc, Dc, Kc = 8, 2048, 1536, 4
    xc = dev_t(synth.round_bf16(rng.standard_normal((Bc, Lc, Dc)).astype(np.float32)), "bf16")
    wc = dev_t((rng.standard_normal((Dc, Kc)) / 2).astype(np.float32), "f32")
    bc = dev_t((0.1 * rng.standard_normal(Dc)).astype(np.float32), "f32")
    oc = torch.empty_like(xc)
    sc = torch.empty(Bc, Dc, Kc - 1, dtype=torch.bfloat16, device=dev)
    cstep = lambda k: msc.causal_conv1d_fwd(xc, wc, bc, out=oc, state_out=sc)
    c_cold = hook_cold_ms(cstep, "conv")
    c_b2b = back_to_back_ms(cstep, 200)
    c_bytes = 2 * Bc * Lc * Dc * 2 + Dc * Kc * 4 + Dc * 4 + Bc * Dc * (Kc - 1) * 2

    # device time per launch without launch latency: 30 launches in a CUDA
    # graph cycling over 3 input / output sets (300 MB, more than L2)
    def conv_graph_us(nset=3, reps=30):
        xs = [xc] + [xc.clone() for _ in range(nset - 1)]
        outs_ = [torch.empty_like(xc) for _ in range(nset)]
        sts = [torch.empty_like(sc) for _ in range(nset)]
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            for k in range(nset):
                msc.causal_conv1d_fwd(xs[k], wc, bc, out=outs_[k], state_out=sts[k])
        torch.cuda.current_stream(dev).wait_stream(side)
        torch.cuda.synchronize(dev)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for k in range(reps):
                msc.causal_conv1d_fwd(xs[k % nset], wc, bc, out=outs_[k % nset],
                                      state_out=sts[k % nset])
        graph.replay()
        torch.cuda.synchronize(dev)
        ts = []
        for _ in range(5):
            flush()
            torch.cuda.synchronize(dev)
            g0 = torch.cuda.Event(enable_timing=True)
            g1 = torch.cuda.Event(enable_timing=True)
            g0.record()
            graph.replay()
            g1.record()
            g1.synchronize()
            ts.append(g0.elapsed_time(g1) * 1e3 / reps)
        del xs, outs_, sts
        return statistics.median(ts)

    try:
        c_graph = conv_graph_us()
    except RuntimeError as exc:  # capture unavailable: report the others
        print(f"conv prefill graph timing skipped: {exc}", file=sys.stderr)
        c_graph = None
    res["conv1d_prefill_8x2048x1536_k4"] = {
        "shape": [Bc, Lc, Dc, Kc], "us_l2_flushed": c_cold * 1e3, "us_back_to_back": c_b2b * 1e3,
        "us_graph_streamed": c_graph,
        "algorithmic_bytes": c_bytes,
        "hbm_frac_l2_flushed": (c_bytes / (c_cold * 1e-3)) / (peaks["hbm_gbs"] * 1e9),
        "hbm_frac_graph_streamed": (None if c_graph is None else
                                    (c_bytes / (c_graph * 1e-6)) / (peaks["hbm_gbs"] * 1e9)),
        "note": ("x read and u written once (50 MB each); a single launch after an L2 flush "
                 "includes the launch latency (a few us of a ~25 us kernel); the graph replay "
                 "streams 3 sets of 100 MB back to back; back to back on one set, part of x "
                 "stays in L2"),
    }
    del xc, oc
    Bu, Du = 256, 5120
    xu = [dev_t(synth.round_bf16(rng.standard_normal((Bu, Du)).astype(np.float32)), "bf16")
          for _ in range(4)]
    wu = dev_t((rng.standard_normal((Du, Kc)) / 2).astype(np.float32), "f32")
    bu = dev_t((0.1 * rng.standard_normal(Du)).astype(np.float32), "f32")
    su = torch.zeros(Bu, Du, Kc - 1, dtype=torch.bfloat16, device=dev)
    ou = torch.empty(Bu, Du, dtype=torch.bfloat16, device=dev)
    ustep = lambda k: msc.causal_conv1d_update(su, xu[k % 4], wu, bu, out=ou)
    u_cold = hook_cold_ms(ustep, "conv_update")
    u_b2b = back_to_back_ms(ustep, 1000)
    u_bytes = 2 * Bu * Du * (Kc - 1) * 2 + 2 * Bu * Du * 2 + Du * Kc * 4 + Du * 4

    # device time per launch without launch latency: 160 launches captured in
    # a CUDA graph, cycling over 16 sets of state / x / out (210 MB, more than
    # L2), so that each launch streams its data from HBM
    def graph_us(nset=16, reps=160):
        sts = [torch.zeros_like(su) for _ in range(nset)]
        xs = [xu[k % 4].clone() for k in range(nset)]
        outs = [torch.empty_like(ou) for _ in range(nset)]
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            for k in range(nset):
                msc.causal_conv1d_update(sts[k], xs[k], wu, bu, out=outs[k])
        torch.cuda.current_stream(dev).wait_stream(side)
        torch.cuda.synchronize(dev)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for k in range(reps):
                msc.causal_conv1d_update(sts[k % nset], xs[k % nset], wu, bu, out=outs[k % nset])
        graph.replay()
        torch.cuda.synchronize(dev)
        ts = []
        for _ in range(5):
            flush()
            torch.cuda.synchronize(dev)
            g0 = torch.cuda.Event(enable_timing=True)
            g1 = torch.cuda.Event(enable_timing=True)
            g0.record()
            graph.replay()
            g1.record()
            g1.synchronize()
            ts.append(g0.elapsed_time(g1) * 1e3 / reps)
        return statistics.median(ts)

    try:
        u_graph = graph_us()
    except RuntimeError as exc:  # capture unavailable: report the others
        print(f"conv update graph timing skipped: {exc}", file=sys.stderr)
        u_graph = None
    res["conv1d_update_256x5120_k4"] = {
        "shape": [Bu, Du, Kc], "us_l2_flushed": u_cold * 1e3, "us_back_to_back": u_b2b * 1e3,
        "us_graph_streamed": u_graph,
        "algorithmic_bytes": u_bytes,
        "hbm_frac_l2_flushed": (u_bytes / (u_cold * 1e-3)) / (peaks["hbm_gbs"] * 1e9),
        "hbm_frac_graph_streamed": (None if u_graph is None else
                                    (u_bytes / (u_graph * 1e-6)) / (peaks["hbm_gbs"] * 1e9)),
        "note": ("21 MB per token: single launches and Python-issued back-to-back calls "
                 "include launch and call latency; the graph replay measures the kernel "
                 "streaming from HBM, with the gap between consecutive kernels"),
    }
    del xu, su, ou

    # backward pass of the scan on the 8 x 2048 x 1536 x 16 layer (bf16):
    # checkpoint pass + adjoint pass, gradients of every input
    xb = synth.workload_inputs("mamba130m_layer")
    ab = dict(u=dev_t(xb.u, "bf16"), dt=dev_t(xb.dt_raw, "bf16"), A=dev_t(xb.A, "f32"),
              B=dev_t(xb.B, "bf16"), C=dev_t(xb.C, "bf16"), D=dev_t(xb.D, "f32"),
              z=dev_t(xb.z, "bf16"), dt_bias=dev_t(xb.dt_bias, "f32"))
    gout = dev_t(synth.round_bf16(np.random.default_rng(14).standard_normal(
        xb.u.shape).astype(np.float32)), "bf16")
    Bb_, Lb_, Db_, Nb_ = xb.u.shape + (xb.B.shape[-1],)
    del xb
    def call_ms(fn, kind, reps=5):
        """Median (whole-call ms, main-kernel ms) over reps calls, L2 flushed."""
        for _ in range(2):
            fn()
        tb, kb = [], []
        for _ in range(reps):
            flush()
            torch.cuda.synchronize(dev)
            msc.profile_read()
            msc.profile_enable(True)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            e1.synchronize()
            msc.profile_enable(False)
            _, kinds = msc.profile_read()
            kb.append(kinds[kind][1])
            tb.append(e0.elapsed_time(e1))
        return statistics.median(tb), statistics.median(kb)

    updb = Bb_ * Lb_ * Db_ * Nb_
    bms, bkms = call_ms(lambda: msc.selective_scan_bwd(**ab, dout=gout), "scan_bwd")
    # algorithmic work of a recompute backward: the forward exponential again
    # and the adjoint's, 2 ex2 per update, plus softplus, sigmoid(dt), sigmoid(z)
    # per (step, channel); HBM: u, dt, z, dout read, du, ddt, dz written (2 B
    # each), B, C read and dB, dC written per (step, state)
    b_mufu = updb * (2 + 6.0 / Nb_)
    b_bytes = Bb_ * Lb_ * Db_ * 7 * 2 + Bb_ * Lb_ * Nb_ * (2 * 2 + 2 * 4) + Db_ * Nb_ * 8
    res["scan_bwd_mamba130m_layer"] = {
        "shape": [Bb_, Lb_, Db_, Nb_], "ms": bms, "adjoint_kernel_ms": bkms,
        "updates_per_s": updb / (bms * 1e-3),
        "mufu_frac": (b_mufu / (bms * 1e-3)) / ex2_peak,
        "hbm_frac": (b_bytes / (bms * 1e-3)) / (peaks["hbm_gbs"] * 1e9),
        "timing": "whole call (memsets, checkpoint and adjoint kernels, stream-ordered scratch)",
    }
    # training with forward-written checkpoints: the forward also stores the
    # state entering every 16 steps, the backward reads them and skips its
    # own forward re-walk (one of its three exponentials per update)
    _, ck_bytes = msc.scan_checkpoint_size(Bb_, Lb_, Db_, Nb_)
    ck = torch.empty(ck_bytes // 4, dtype=torch.float32, device=dev).view(
        Bb_, -1, Db_, Nb_)
    fo = torch.empty(Bb_, Lb_, Db_, dtype=torch.bfloat16, device=dev)
    fl = torch.empty(Bb_, Db_, Nb_, dtype=torch.float32, device=dev)
    f_ms, f_kms = call_ms(lambda: msc.selective_scan_fwd(**ab, out=fo, last_state=fl), "scan")
    fc_ms, fc_kms = call_ms(lambda: msc.selective_scan_fwd_ckpt(
        **ab, out=fo, last_state=fl, ckpt=ck), "scan")
    bc_ms, bc_kms = call_ms(lambda: msc.selective_scan_bwd(**ab, dout=gout, ckpt=ck),
                            "scan_bwd")
    res["scan_train_ckpt_mamba130m_layer"] = {
        "shape": [Bb_, Lb_, Db_, Nb_], "checkpoint_bytes": ck_bytes,
        "fwd_ms": f_ms, "fwd_kernel_ms": f_kms,
        "fwd_ckpt_ms": fc_ms, "fwd_ckpt_kernel_ms": fc_kms,
        "bwd_recompute_ms": bms, "bwd_from_ckpt_ms": bc_ms, "bwd_from_ckpt_kernel_ms": bc_kms,
        "fwd_plus_bwd_recompute_ms": f_ms + bms, "fwd_ckpt_plus_bwd_ms": fc_ms + bc_ms,
        "bwd_from_ckpt_mufu_frac": (b_mufu / (bc_ms * 1e-3)) / ex2_peak,
        "timing": "whole calls, L2 flushed before each; kernel ms from the library's "
                  "event pair around its main kernel",
    }
    del ab, gout, ck, fo, fl
    torch.cuda.empty_cache()

    # (workload, discretisation): the other two scan workloads, and the
    # 8 x 2048 x 1536 x 16 layer once more with the ZOH input matrix and with
    # the exponential-trapezoid input (lambda ~ U[0, 1])
    for name, disc in (("long_seq_64k", "euler"), ("mamba2p8b_layer", "euler"),
                       ("mamba130m_layer", "zoh"), ("mamba130m_layer", "trapezoid")):
        zoh = disc == "zoh"
        w = synth.WORKLOADS[name]
        x = synth.workload_inputs(name)
        a = dict(u=dev_t(x.u, "bf16"), dt=dev_t(x.dt_raw, "bf16"),
                 A=dev_t(x.A, "f32"), B=dev_t(x.B, "bf16"), C=dev_t(x.C, "bf16"),
                 D=dev_t(x.D, "f32"), z=dev_t(x.z, "bf16"),
                 dt_bias=dev_t(x.dt_bias, "f32"))
        lam = None
        if disc == "trapezoid":
            lam = dev_t(synth.round_bf16(np.random.default_rng(13).uniform(
                0.0, 1.0, x.u.shape).astype(np.float32)), "bf16")
        del x
        B_, L_, D_, N_ = w["batch"], w["L"], w["d_inner"], w["d_state"]
        out = torch.empty_like(a["u"])
        last = torch.empty(B_, D_, N_, dtype=torch.float32, device=dev)
        nws = msc.scan_workspace_size(B_, L_, D_, N_, torch.bfloat16)
        wsp = torch.empty(max(nws, 1), dtype=torch.uint8, device=dev)

        def call():
            if lam is not None:
                msc.selective_scan_trap_fwd(a["u"], a["dt"], lam, a["A"], a["B"], a["C"],
                                            a["D"], a["z"], a["dt_bias"], out=out,
                                            last_state=last, workspace=wsp)
            else:
                msc.selective_scan_fwd_ws(**a, out=out, last_state=last, workspace=wsp,
                                          zoh=zoh)
        for _ in range(3):
            call()
        times, total = [], []
        for _ in range(7):
            flush()
            torch.cuda.synchronize(dev)
            msc.profile_read()
            msc.profile_enable(True)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            call()
            e1.record()
            e1.synchronize()
            msc.profile_enable(False)
            _, kinds = msc.profile_read()
            times.append(kinds["scan"][1])
            total.append(e0.elapsed_time(e1))
        upd, mufu, byt = algorithmic(B_, L_, D_, N_)
        ms = statistics.median(total)
        kms = statistics.median(times)
        res[name + ("" if disc == "euler" else "_" + disc)] = {
            "shape": [B_, L_, D_, N_], "discretization": disc,
            "ms": ms,
            "updates_per_s": upd / (ms * 1e-3),
            "output_kernel_ms": kms,
            "mufu_frac": (mufu / (ms * 1e-3)) / ex2_peak,
            "hbm_frac": (byt / (ms * 1e-3)) / (peaks["hbm_gbs"] * 1e9),
            "timing": "whole call (all kernels), L2 flushed by a 512 MiB read before each",
        }
        del a, out, last, wsp, lam
        torch.cuda.empty_cache()

    # decode: 256 x 5120 x 16, 1000 steps, state in place
    name = "decode_256x5120"
    w = synth.WORKLOADS[name]
    Bb, Dd, Nn, steps = w["batch"], w["d_inner"], w["d_state"], w["steps"]
    p = synth.decode_params(Bb, Dd, Nn)
    state = torch.from_numpy(p.state0).to(dev)
    A = dev_t(p.A, "f32")
    Dv = dev_t(p.D, "f32")
    bias = dev_t(p.dt_bias, "f32")
    pool = []
    for k in range(8):   # 8 distinct token inputs, cycled over the steps
        s = synth.decode_step(Bb, Dd, Nn, k)
        pool.append(tuple(dev_t(v, "bf16") for v in (s.u, s.dt_raw, s.z, s.B, s.C)))
    out = torch.empty(Bb, Dd, dtype=torch.bfloat16, device=dev)
    def dstep(k):
        uu, dd, zz, BB, CC = pool[k % 8]
        msc.selective_state_update(state, uu, dd, A, BB, CC, Dv, zz, bias, out=out)
    # the workload as defined: `steps` sequential tokens, each with its own
    # inputs pre-staged on the device (7.9 GB for 1000 tokens, drawn from a
    # seeded device generator with the workload's distributions), the state
    # updated in place; the steps are replayed from one CUDA graph, so the
    # timed region holds the kernels back to back and no host work
    gen = torch.Generator(device=dev)
    gen.manual_seed(w["seed"])

    def draw(shape, scale=1.0):
        return (torch.randn(shape, generator=gen, device=dev) * scale).to(torch.bfloat16)

    Us, Zs = draw((steps, Bb, Dd)), draw((steps, Bb, Dd))
    Ts = draw((steps, Bb, Dd), 0.5)
    Bs, Cs = draw((steps, Bb, Nn)), draw((steps, Bb, Nn))

    def gstep(k):
        msc.selective_state_update(state, Us[k], Ts[k], A, Bs[k], Cs[k], Dv, Zs[k], bias,
                                   out=out)
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        for k in range(3):
            gstep(k)
    torch.cuda.current_stream(dev).wait_stream(side)
    torch.cuda.synchronize(dev)
    dgraph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(dgraph):
        for k in range(steps):
            gstep(k)
    dgraph.replay()
    torch.cuda.synchronize(dev)
    flush()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    dgraph.replay()
    e1.record()
    e1.synchronize()
    b2b_ms = e0.elapsed_time(e1) / steps
    del dgraph, Us, Zs, Ts, Bs, Cs
    torch.cuda.empty_cache()
    cold_ms = hook_cold_ms(dstep, "update")
    byt = 2 * Bb * Dd * Nn * 4 + 4 * Bb * Dd * 2 + 2 * Bb * Nn * 2 + Dd * Nn * 4 + 2 * Dd * 4
    upd = Bb * Dd * Nn
    res[name] = {
        "shape": [Bb, Dd, Nn], "steps": steps,
        "us_per_step_back_to_back": b2b_ms * 1e3,
        "us_per_step_l2_flushed": cold_ms * 1e3,
        "updates_per_s_back_to_back": upd / (b2b_ms * 1e-3),
        "hbm_frac_l2_flushed": (byt / (cold_ms * 1e-3)) / (peaks["hbm_gbs"] * 1e9),
        "hbm_frac_back_to_back": (byt / (b2b_ms * 1e-3)) / (peaks["hbm_gbs"] * 1e9),
        "algorithmic_bytes_per_step": byt,
        "note": ("back to back: the workload's 1000 tokens with distinct pre-staged inputs, "
                 "replayed from one CUDA graph (part of the 84 MB state stays in the "
                 "126 MB L2 from token to token); l2_flushed: one token after a 512 MiB "
                 "read, the cold-cache bound"),
    }
    # the same step with the zero-order-hold input and with the exponential
    # trapezoid (lambda ~ U[0, 1]; the previous token's u and B from the pool)
    lam = dev_t(synth.round_bf16(np.random.default_rng(15).uniform(
        0.0, 1.0, (Bb, Dd)).astype(np.float32)), "bf16")
    def zstep(k):
        uu, dd, zz, BB, CC = pool[k % 8]
        msc.selective_state_update(state, uu, dd, A, BB, CC, Dv, zz, bias, out=out, zoh=True)
    def tstep(k):
        uu, dd, zz, BB, CC = pool[k % 8]
        up, _, _, Bq, _ = pool[(k + 7) % 8]
        msc.selective_state_update_trap(state, up, Bq, uu, dd, lam, A, BB, CC, Dv, zz, bias,
                                        out=out)
    trap_extra = 2 * Bb * Dd * 2 + Bb * Nn * 2   # lambda and u_prev, the B_prev rows
    for vname, call, extra in (("zoh", zstep, 0), ("trapezoid", tstep, trap_extra)):
        v_ms = hook_cold_ms(call, "update")
        res[f"{name}_{vname}"] = {
            "shape": [Bb, Dd, Nn], "us_per_step_l2_flushed": v_ms * 1e3,
            "hbm_frac_l2_flushed": ((byt + extra) / (v_ms * 1e-3)) / (peaks["hbm_gbs"] * 1e9),
            "algorithmic_bytes_per_step": byt + extra,
        }
    del lam
    return res


def run_profile(args):
    """Run one workload's main kernel alone, for ncu captures: W + K calls
    of the scan (or of the decode step), nothing timed, nothing printed but
    a completion line."""
    import torch
    import selective_state_space_144_b300 as msc
    from selective_state_space_144_b300 import build as msc_build
    msc_build.build()
    dev = torch.device("cuda", 0)
    name = args.profile

    def dev_t(arr, kind):
        if kind == "bf16":
            bits = synth.bf16_bits(arr).view(np.int16)
            return torch.from_numpy(bits.copy()).to(dev).view(torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(arr, np.float32)).to(dev)

    if name in ("scan_bwd", "scan_bwd_ckpt"):
        # backward pass of the scan on the 8 x 2048 x 1536 x 16 layer, bf16;
        # scan_bwd_ckpt: the checkpointing forward once, then the backward
        # from its checkpoints
        x = synth.workload_inputs("mamba130m_layer")
        a = dict(u=dev_t(x.u, "bf16"), dt=dev_t(x.dt_raw, "bf16"), A=dev_t(x.A, "f32"),
                 B=dev_t(x.B, "bf16"), C=dev_t(x.C, "bf16"), D=dev_t(x.D, "f32"),
                 z=dev_t(x.z, "bf16"), dt_bias=dev_t(x.dt_bias, "f32"))
        gout = dev_t(synth.round_bf16(np.random.default_rng(14).standard_normal(
            x.u.shape).astype(np.float32)), "bf16")
        del x
        ck = msc.selective_scan_fwd_ckpt(**a)[2] if name == "scan_bwd_ckpt" else None
        for _ in range(args.warmup + args.steps):
            msc.selective_scan_bwd(**a, dout=gout, ckpt=ck)
        torch.cuda.synchronize(dev)
        msc.check_device_error()
        print(f"profile run done: {name}, {args.warmup + args.steps} calls", flush=True)
        return 0
    if name in ("conv1d_prefill", "conv1d_update"):
        # the conv before the scan: prefill on the 8 x 2048 x 1536 layer, or
        # the decode token on 256 x 5120; d_conv 4, bf16
        rng = np.random.default_rng(12)
        if name == "conv1d_prefill":
            Bc, Lc, Dc = 8, 2048, 1536
            x = dev_t(synth.round_bf16(rng.standard_normal((Bc, Lc, Dc)).astype(np.float32)),
                      "bf16")
        else:
            Bc, Dc = 256, 5120
            x = dev_t(synth.round_bf16(rng.standard_normal((Bc, Dc)).astype(np.float32)), "bf16")
        wc = dev_t((rng.standard_normal((Dc, 4)) / 2).astype(np.float32), "f32")
        bc = dev_t((0.1 * rng.standard_normal(Dc)).astype(np.float32), "f32")
        st = torch.zeros(Bc, Dc, 3, dtype=torch.bfloat16, device=dev)
        for _ in range(args.warmup + args.steps):
            if name == "conv1d_prefill":
                msc.causal_conv1d_fwd(x, wc, bc, state_out=st)
            else:
                msc.causal_conv1d_update(st, x, wc, bc)
        torch.cuda.synchronize(dev)
        msc.check_device_error()
        print(f"profile run done: {name}, {args.warmup + args.steps} calls", flush=True)
        return 0
    # a scan workload with a suffix runs that discretisation: NAME_zoh (the
    # zero-order-hold input) or NAME_trapezoid (lambda ~ U[0, 1])
    disc = "euler"
    for sfx in ("_zoh", "_trapezoid"):
        if name.endswith(sfx):
            name, disc = name[:-len(sfx)], sfx[1:]
    w = synth.WORKLOADS[name]
    if name.startswith("decode"):
        Bb, Dd, Nn = w["batch"], w["d_inner"], w["d_state"]
        p = synth.decode_params(Bb, Dd, Nn)
        s = synth.decode_step(Bb, Dd, Nn, 0)
        state = torch.from_numpy(p.state0).to(dev)
        args_ = (dev_t(s.u, "bf16"), dev_t(s.dt_raw, "bf16"), dev_t(p.A, "f32"),
                 dev_t(s.B, "bf16"), dev_t(s.C, "bf16"), dev_t(p.D, "f32"),
                 dev_t(s.z, "bf16"), dev_t(p.dt_bias, "f32"))
        for _ in range(args.warmup + args.steps):
            msc.selective_state_update(state, *args_)
    else:
        x = synth.workload_inputs(name)
        kind = w["dtype"]
        a = dict(u=dev_t(x.u, kind), dt=dev_t(x.dt_raw, kind), A=dev_t(x.A, "f32"),
                 B=dev_t(x.B, kind), C=dev_t(x.C, kind), D=dev_t(x.D, "f32"),
                 z=dev_t(x.z, kind), dt_bias=dev_t(x.dt_bias, "f32"))
        lam = None
        if disc == "trapezoid":  # the same lambda as the bench's trapezoid workload
            lam = dev_t(synth.round_bf16(np.random.default_rng(13).uniform(
                0.0, 1.0, x.u.shape).astype(np.float32)), kind)
        del x
        B_, L_, D_, N_ = w["batch"], w["L"], w["d_inner"], w["d_state"]
        out = torch.empty_like(a["u"])
        last = torch.empty(B_, D_, N_, dtype=torch.float32, device=dev)
        n = msc.scan_workspace_size(B_, L_, D_, N_, a["u"].dtype)
        wsp = torch.empty(max(n, 1), dtype=torch.uint8, device=dev)
        for _ in range(args.warmup + args.steps):
            if lam is not None:
                msc.selective_scan_trap_fwd(a["u"], a["dt"], lam, a["A"], a["B"], a["C"],
                                            a["D"], a["z"], a["dt_bias"], out=out,
                                            last_state=last, workspace=wsp)
            else:
                msc.selective_scan_fwd_ws(**a, out=out, last_state=last, workspace=wsp,
                                          zoh=disc == "zoh")
    torch.cuda.synchronize(dev)
    msc.check_device_error()
    print(f"profile run done: {name}, {args.warmup + args.steps} calls", flush=True)
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    if args.profile:
        return run_profile(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
