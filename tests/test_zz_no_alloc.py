"""The allocation-free scan entry point, msc_selective_scan_fwd_noalloc.

Callers that may not allocate device memory while they serve requests -- a
runtime whose own allocator owns the GPU -- use this entry point: the
scratch the scan needs lives in a fixed device array inside the library, so
the call allocates nothing.  This test calls it through the C ABI twice in a
row, on two different problems that both use the scratch (bf16 inputs need
fp32 copies of B and C; three time chunks need chunk carries), and checks
  * each result against the fp64 oracle on the same inputs, within the
    parity tolerance of the other tests, and against the allocating entry
    point msc_selective_scan_fwd;
  * that the call allocated nothing: after a first call (which, with lazy
    module loading, maps the library's module and its scratch array), the
    device's free memory (cudaMemGetInfo) and torch's allocated and reserved
    byte counts are the same before and after a synchronised call.
The file is named to be collected last; it also passes run alone in a
fresh process.
"""
import ctypes

import numpy as np
import pytest

import oracle
import selective_state_space_144_b300 as msc
from selective_state_space_144_b300 import synth
from tests.helpers import TOL, as_stored, from_device, rel_l2, scan_device_args

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _noalloc_entry():
    f = msc.load().msc_selective_scan_fwd_noalloc
    f.restype = ctypes.c_int
    f.argtypes = ([ctypes.c_void_p] * 10 + [ctypes.c_int64] * 4
                  + [ctypes.c_int, ctypes.c_void_p])
    return f


def _ptr(t):
    return None if t is None else t.data_ptr()


def _call(entry, a, out, last, dims):
    batch, L, d_inner, N = dims
    return entry(_ptr(a["u"]), _ptr(a["dt"]), _ptr(a["A"]), _ptr(a["B"]),
                 _ptr(a["C"]), _ptr(a["D"]), _ptr(a["z"]), _ptr(a["dt_bias"]),
                 _ptr(out), _ptr(last), batch, L, d_inner, N, msc.MSC_BF16,
                 torch.cuda.current_stream().cuda_stream)


def _memory():
    free, _total = torch.cuda.mem_get_info()
    return free, torch.cuda.memory_allocated(), torch.cuda.memory_reserved()


def test_noalloc_scan_matches_oracle_twice_and_allocates_nothing():
    entry = _noalloc_entry()
    msc.tuning_set("scan_chunks", 3)
    try:
        problems = [(2, 700, 128, 16, 41), (3, 517, 96, 16, 42)]
        for batch, L, d_inner, N, seed in problems:
            x = synth.scan_inputs(batch, L, d_inner, N, dtype="bf16", seed=seed,
                                  D="normal")
            a = scan_device_args(x)
            dims = (batch, L, d_inner, N)
            assert msc.scan_workspace_size(batch, L, d_inner, N, torch.bfloat16) > 0
            ref_out, ref_last = msc.selective_scan_fwd(**a)
            out = torch.full_like(ref_out, float("nan"))
            last = torch.full_like(ref_last, float("nan"))
            # a first call maps what lazy loading maps; then nothing may change
            assert _call(entry, a, out, last, dims) == 0
            out.fill_(float("nan"))
            last.fill_(float("nan"))
            torch.cuda.synchronize()
            before = _memory()
            st = _call(entry, a, out, last, dims)
            assert st == 0, msc.load().msc_status_string(st)
            torch.cuda.synchronize()
            after = _memory()
            assert after == before, f"device memory changed: {before} -> {after}"
            got_out, got_last = from_device(out), from_device(last)
            assert np.all(np.isfinite(got_out)) and np.all(np.isfinite(got_last))
            y_ref, s_ref = oracle.scan_fwd(x.u, x.dt_raw, x.A, x.B, x.C, x.D, x.z,
                                           x.dt_bias)
            assert rel_l2(got_out, as_stored(y_ref, "bf16")) <= TOL["bf16"]
            assert rel_l2(got_last, s_ref) <= TOL["bf16"]
            assert rel_l2(got_out, from_device(ref_out)) <= TOL["bf16"]
            assert rel_l2(got_last, from_device(ref_last)) <= TOL["bf16"]
        msc.check_device_error()
    finally:
        msc.tuning_set("scan_chunks", 0)
