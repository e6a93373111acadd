"""The C ABI on the host: the library loads, exports every symbol that
include/msc.h declares, and rejects bad arguments synchronously, before any
launch (so none of these tests needs a GPU)."""
import ctypes
import os
import re

import pytest

import selective_state_space_144_b300 as msc
from selective_state_space_144_b300 import build as msc_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "msc.h")


@pytest.fixture(scope="module")
def lib():
    msc_build.build()
    return msc.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(msc_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("msc_selective_scan_fwd", "msc_selective_state_update",
                     "msc_selective_scan_fwd_ws",
                     "msc_selective_scan_workspace_size", "msc_status_string"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"libmsc.so does not export {name}"


def test_status_strings(lib):
    for code in range(8):
        s = lib.msc_status_string(code)
        assert s and s != b"unknown status"
    assert lib.msc_status_string(99) == b"unknown status"
    assert lib.msc_version() >= 100


V = ctypes.c_void_p
FAKE = 0x10000          # never dereferenced: validation fails first


def scan(lib, *, u=FAKE, dt=FAKE, A=FAKE, B=FAKE, C=FAKE, D=None, z=None,
         bias=None, out=FAKE, last=None, batch=2, L=8, d_inner=16, d_state=16,
         dtype=1):
    return lib.msc_selective_scan_fwd(u, dt, A, B, C, D, z, bias, out, last,
                                      batch, L, d_inner, d_state, dtype, None)


def test_scan_rejects_bad_sizes(lib):
    assert scan(lib, d_state=0) == 2
    assert scan(lib, d_state=65) == 2
    assert scan(lib, batch=-1) == 1
    assert scan(lib, L=-1) == 1
    assert scan(lib, d_inner=-3) == 1
    assert scan(lib, dtype=7) == 1
    big = 2**62
    assert scan(lib, batch=big, L=big) == 2        # element count overflow


def test_scan_rejects_null_and_misaligned(lib):
    assert scan(lib, u=None) == 1
    assert scan(lib, out=None) == 1
    assert scan(lib, A=None) == 1
    assert scan(lib, u=FAKE + 1) == 3              # bf16 needs 2-byte alignment
    assert scan(lib, u=FAKE + 2, dtype=0) == 3     # fp32 needs 4-byte alignment
    assert scan(lib, D=FAKE + 2) == 3              # D is fp32
    assert scan(lib, last=FAKE + 1) == 3


def test_scan_empty_is_a_no_op(lib):
    # nothing to compute: returns OK without touching (fake) pointers
    assert scan(lib, batch=0) == 0
    assert scan(lib, d_inner=0) == 0


def test_workspace_size_query(lib):
    n = ctypes.c_size_t(123)
    assert lib.msc_selective_scan_workspace_size(8, 2048, 1536, 16, 1,
                                                 ctypes.byref(n)) == 0
    assert lib.msc_selective_scan_workspace_size(0, 2048, 1536, 16, 1,
                                                 ctypes.byref(n)) == 0
    assert n.value == 0
    assert lib.msc_selective_scan_workspace_size(1, 2048, 1536, 0, 1,
                                                 ctypes.byref(n)) == 2
    assert lib.msc_selective_scan_workspace_size(1, 2048, 1536, 16, 1,
                                                 None) == 1
    # one chunk -> no carry workspace
    assert lib.msc_tuning_set(b"scan_chunks", 1) == 0
    try:
        assert lib.msc_selective_scan_workspace_size(
            1, 4096, 64, 16, 1, ctypes.byref(n)) == 0
        assert n.value == 0
        assert lib.msc_tuning_set(b"scan_chunks", 4) == 0
        assert lib.msc_selective_scan_workspace_size(
            2, 4096, 64, 16, 1, ctypes.byref(n)) == 0
        assert n.value == 2 * 2 * 3 * 64 * 16 * 4   # (a, b) x batch x (K-1) x D x N
    finally:
        lib.msc_tuning_set(b"scan_chunks", 0)


def test_workspace_variant_rejects_small_workspace(lib):
    assert lib.msc_tuning_set(b"scan_chunks", 4) == 0
    try:
        st = lib.msc_selective_scan_fwd_ws(
            FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None, FAKE, None,
            2, 4096, 64, 16, 1, None, 0, None)
        assert st == 5
        st = lib.msc_selective_scan_fwd_ws(
            FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None, FAKE, None,
            2, 4096, 64, 16, 1, FAKE + 16, 1 << 30, None)
        assert st == 5                              # not 256-byte aligned
    finally:
        lib.msc_tuning_set(b"scan_chunks", 0)


def test_tuning_keys(lib):
    assert lib.msc_tuning_set(b"no_such_key", 1) == 1
    assert lib.msc_tuning_set(b"scan_chunks", -1) == 1
    assert lib.msc_tuning_set(None, 1) == 1
    assert lib.msc_tuning_set(b"scan_min_chunk", 512) == 0
    assert lib.msc_tuning_set(b"debug_starve_copies", -1) == 1
    assert lib.msc_tuning_set(b"debug_starve_copies", (1 << 22) + 1) == 1
    assert lib.msc_tuning_set(b"debug_starve_copies", 0) == 0
    for key in (b"update_path",):
        assert lib.msc_tuning_set(key, 2) == 1
        assert lib.msc_tuning_set(key, 1) == 0
        assert lib.msc_tuning_set(key, 0) == 0


def upd(lib, *, state=FAKE, u=FAKE, dt=FAKE, A=FAKE, B=FAKE, C=FAKE, D=None,
        z=None, bias=None, out=FAKE, batch=4, d_inner=16, d_state=16, dtype=1):
    return lib.msc_selective_state_update(state, u, dt, A, B, C, D, z, bias,
                                          out, batch, d_inner, d_state, dtype,
                                          None)


def test_state_update_validation(lib):
    assert upd(lib, d_state=0) == 2
    assert upd(lib, d_state=100) == 2
    assert upd(lib, batch=-1) == 1
    assert upd(lib, state=None) == 1
    assert upd(lib, out=None) == 1
    assert upd(lib, state=FAKE + 2) == 3
    assert upd(lib, z=FAKE + 1) == 3
    assert upd(lib, dtype=5) == 1
    assert upd(lib, batch=0) == 0


def test_python_binding_fails_loudly_without_cuda_tensors():
    torch = pytest.importorskip("torch")
    x = torch.zeros(1, 4, 8)
    with pytest.raises(ValueError):
        msc.selective_scan_fwd(x, x, torch.zeros(8, 4), torch.zeros(1, 4, 4),
                               torch.zeros(1, 4, 4))


def test_noalloc_rejects_problems_beyond_its_scratch(lib):
    """The allocation-free entry point refuses, before any device work, a
    problem whose scratch exceeds its fixed 16 MiB: 64 time chunks of a
    4 x 4096 x 1024 x 16 scan need 33 MB of chunk carries under either
    kernel family."""
    f = lib.msc_selective_scan_fwd_noalloc
    f.restype = ctypes.c_int
    f.argtypes = ([ctypes.c_void_p] * 10 + [ctypes.c_int64] * 4
                  + [ctypes.c_int, ctypes.c_void_p])
    assert lib.msc_tuning_set(b"scan_chunks", 64) == 0
    try:
        st = f(FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None, FAKE, None,
               4, 4096, 1024, 16, 1, None)
    finally:
        lib.msc_tuning_set(b"scan_chunks", 0)
    assert st == 7
    assert lib.msc_status_string(7) != b"unknown status"


def test_extended_entry_points_validate(lib):
    """msc_selective_scan_fwd_ex / msc_selective_state_update_ex: unknown
    discretisation and a misaligned h0 are refused before any launch."""
    f = lib.msc_selective_scan_fwd_ex
    f.restype = ctypes.c_int
    f.argtypes = ([ctypes.c_void_p] * 11 + [ctypes.c_int64] * 4
                  + [ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t,
                     ctypes.c_void_p])
    args = lambda h0, disc: (FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None, h0,
                             FAKE, None, 2, 8, 16, 16, 1, disc, None, 0, None)
    assert f(*args(None, 2)) == 1
    assert f(*args(None, -1)) == 1
    assert f(*args(FAKE + 2, 1)) == 3               # h0 is fp32
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None, FAKE, FAKE, None,
             0, 8, 16, 16, 1, 1, None, 0, None) == 0   # empty batch: no-op
    g = lib.msc_selective_state_update_ex
    g.restype = ctypes.c_int
    g.argtypes = [ctypes.c_void_p] * 10 + [ctypes.c_int64] * 3 + [ctypes.c_int] * 2 + [
        ctypes.c_void_p]
    assert g(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None, FAKE,
             4, 16, 16, 1, 7, None) == 1
    assert g(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None, FAKE,
             4, 16, 0, 1, 1, None) == 2


def test_conv_entry_points_validate(lib):
    f = lib.msc_causal_conv1d_fwd
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p] * 6 + [ctypes.c_int64] * 4 + [ctypes.c_int] * 2 + [
        ctypes.c_void_p]
    c = lambda **k: f(k.get("x", FAKE), k.get("w", FAKE), None, k.get("st", None),
                      k.get("out", FAKE), None, k.get("batch", 2), k.get("L", 8),
                      k.get("d", 16), k.get("K", 4), k.get("silu", 1), k.get("dt", 1), None)
    assert c(K=0) == 2 and c(K=9) == 2 and c(K=-1) == 1
    assert c(silu=2) == 1 and c(dt=3) == 1 and c(L=-1) == 1
    assert c(x=None) == 1 and c(w=None) == 1
    assert c(x=FAKE + 1) == 3 and c(st=FAKE + 1) == 3
    assert c(batch=70000) == 2
    assert c(batch=0) == 0
    g = lib.msc_causal_conv1d_update
    g.restype = ctypes.c_int
    g.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int64] * 3 + [ctypes.c_int] * 2 + [
        ctypes.c_void_p]
    assert g(None, FAKE, FAKE, None, FAKE, 2, 16, 4, 1, 1, None) == 1   # state needed
    assert g(FAKE, FAKE, FAKE, None, FAKE, 2, 16, 12, 1, 1, None) == 2


def test_bwd_entry_point_validates(lib):
    """msc_selective_scan_bwd refuses bad arguments before touching the GPU;
    an empty batch is a no-op."""
    f = lib.msc_selective_scan_bwd
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p] * 20 + [ctypes.c_int64] * 4 + [ctypes.c_int, ctypes.c_void_p]

    def bwd(**k):
        p = {n: k.get(n, FAKE) for n in ("u", "dt", "A", "B", "C", "dout", "du", "ddt",
                                         "dA", "dB", "dC")}
        return f(p["u"], p["dt"], p["A"], p["B"], p["C"], None, None, None, None, p["dout"],
                 None, p["du"], p["ddt"], p["dA"], p["dB"], p["dC"], None, None, None,
                 k.get("dh0", None), k.get("batch", 2), k.get("L", 8), 16, k.get("N", 16),
                 k.get("dtype", 1), None)

    assert bwd(dtype=3) == 1                       # unknown dtype
    assert bwd(N=0) == 2 and bwd(N=65) == 2        # d_state outside 1..64
    assert bwd(L=-1) == 1
    assert bwd(dout=None) == 1 and bwd(dA=None) == 1 and bwd(dB=None) == 1
    assert bwd(u=FAKE + 1) == 3                    # bf16 storage: 2-byte alignment
    assert bwd(dA=FAKE + 2) == 3 and bwd(dh0=FAKE + 2) == 3   # fp32 outputs
    assert bwd(batch=70000) == 2
    assert bwd(batch=0) == 0                       # nothing to do


def test_checkpoint_entry_points_validate(lib):
    """msc_scan_checkpoint_size on the host, and the checkpointing forward
    and backward refusing bad arguments before any launch."""
    q = lib.msc_scan_checkpoint_size
    tt, n = ctypes.c_int64(0), ctypes.c_size_t(0)
    assert q(2, 100, 24, 16, ctypes.byref(tt), ctypes.byref(n)) == 0
    assert tt.value == 16 and n.value == 2 * 7 * 24 * 16 * 4   # ceil(100 / 16) rows
    assert q(3, 64, 8, 32, ctypes.byref(tt), ctypes.byref(n)) == 0
    assert tt.value == 8 and n.value == 3 * 8 * 8 * 32 * 4
    assert q(2, 0, 8, 64, ctypes.byref(tt), ctypes.byref(n)) == 0 and n.value == 0
    assert q(2, 8, 8, 12, ctypes.byref(tt), ctypes.byref(n)) == 2    # no TMA path for 12
    assert q(2, -1, 8, 16, ctypes.byref(tt), ctypes.byref(n)) == 1
    assert q(2, 8, 8, 16, None, ctypes.byref(n)) == 1
    assert q(1 << 40, 1 << 20, 1 << 10, 16, ctypes.byref(tt), ctypes.byref(n)) == 2

    f = lib.msc_selective_scan_fwd_ckpt
    ck = lambda ckpt, N=16, batch=2: f(FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None,
                                       None, FAKE, None, ckpt, batch, 40, 16, N, 1,
                                       None, 0, None)
    assert ck(None) == 1                         # checkpoints required
    assert ck(FAKE + 8) == 3                     # 16-byte aligned
    assert ck(FAKE, N=12) == 2                   # TMA kernel only
    assert ck(None, batch=0) == 0                # nothing to do

    g = lib.msc_selective_scan_bwd_ckpt

    def bwd(ckpt, batch=2):
        return g(FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None, None, ckpt, FAKE, None,
                 FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None, None, batch, 40, 16, 16,
                 1, None)

    assert bwd(None) == 1
    assert bwd(FAKE + 4) == 3
    assert bwd(None, batch=0) == 0


def test_scratch_release_without_pools(lib):
    """Before any call has taken scratch there is no pool to trim."""
    lib.msc_scratch_release.restype = ctypes.c_int
    assert lib.msc_scratch_release() == 0


def test_trapezoid_entry_points_validate(lib):
    """The exponential-trapezoid scan and decode token need lam; its
    alignment is checked like the other storage arrays; an empty batch is a
    no-op."""
    f = lib.msc_selective_scan_trap_fwd
    f.restype = ctypes.c_int
    f.argtypes = ([ctypes.c_void_p] * 14 + [ctypes.c_int64] * 4
                  + [ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p])

    def trap(lam=FAKE, batch=2, prev=None):
        return f(FAKE, FAKE, lam, FAKE, FAKE, FAKE, None, None, None, None, prev, prev,
                 FAKE, None, batch, 8, 16, 16, 1, None, 0, None)

    assert trap(lam=None) == 1
    assert trap(lam=FAKE + 1) == 3                 # bf16 storage
    assert trap(prev=FAKE + 1) == 3                # u_prev / B_prev too
    assert trap(batch=0) == 0
    g = lib.msc_selective_state_update_trap
    g.restype = ctypes.c_int
    g.argtypes = [ctypes.c_void_p] * 13 + [ctypes.c_int64] * 3 + [ctypes.c_int, ctypes.c_void_p]
    assert g(FAKE, None, None, FAKE, FAKE, None, FAKE, FAKE, FAKE, None, None, None, FAKE,
             4, 16, 16, 1, None) == 1              # lam required
    assert g(FAKE, None, None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None, FAKE,
             4, 16, 0, 1, None) == 2               # d_state 0
