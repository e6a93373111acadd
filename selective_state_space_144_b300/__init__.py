"""Mamba selective scan (S6) on NVIDIA B300 -- Python binding of libmsc.so.

Argument marshalling only: every step of the computation runs in the sm_103a
kernels behind the C ABI of ``include/msc.h``.  PyTorch supplies device
memory and streams.  There is no CPU fallback: if ``libmsc.so`` has not been
built, every call raises ``RuntimeError``.

    selective_scan_fwd(u, dt, A, B, C, D=None, z=None, dt_bias=None,
                       out=None, last_state=None, return_last_state=True)
    selective_state_update(state, u, dt, A, B, C, D=None, z=None,
                           dt_bias=None, out=None)

Shapes: u, dt, z: (batch, L, d_inner); B, C: (batch, L, d_state);
A: (d_inner, d_state); D, dt_bias: (d_inner,); state / last_state:
(batch, d_inner, d_state).  u, dt, z, B, C share one dtype (float32 or
bfloat16); A, D, dt_bias and the state are float32.
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "MscError", "selective_scan", "selective_scan_fwd", "selective_scan_fwd_ws",
    "selective_scan_fwd_ckpt", "scan_checkpoint_size", "selective_scan_bwd",
    "selective_scan_trap_fwd", "selective_state_update_trap",
    "causal_conv1d_fwd", "causal_conv1d_update",
    "selective_state_update", "scan_workspace_size", "tuning_set",
    "check_device_error", "scratch_release", "profile_enable", "profile_read",
    "library_path", "load",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIBNAME = "libmsc.so"

MSC_F32, MSC_BF16 = 0, 1
MSC_DISC_EULER, MSC_DISC_ZOH = 0, 1
_STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported size",
           3: "pointer not aligned to its element size",
           4: "CUDA runtime error",
           5: "workspace missing, too small or misaligned",
           6: "a kernel's bounded wait for a data copy gave up",
           7: "scratch need exceeds the allocation-free entry point's buffer"}


class MscError(RuntimeError):
    """A non-zero msc_status returned by the library."""

    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {_STATUS.get(status, 'unknown status')} "
                         f"(status {status})")


_lib = None


def library_path() -> str:
    return os.path.join(_PKG, _LIBNAME)


def load():
    """Load libmsc.so (once).  Raises RuntimeError when it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it with "
            "`python -m selective_state_space_144_b300.build` "
            "(there is no CPU fallback)")
    lib = ctypes.CDLL(path)
    vp, i64, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
    st = ctypes.c_int
    lib.msc_selective_scan_fwd.restype = st
    lib.msc_selective_scan_fwd.argtypes = [vp] * 10 + [i64] * 4 + [st, vp]
    lib.msc_selective_scan_fwd_ws.restype = st
    lib.msc_selective_scan_fwd_ws.argtypes = ([vp] * 10 + [i64] * 4
                                              + [st, vp, sz, vp])
    lib.msc_selective_scan_fwd_ex.restype = st
    lib.msc_selective_scan_fwd_ex.argtypes = ([vp] * 11 + [i64] * 4
                                              + [st, st, vp, ctypes.c_size_t, vp])
    lib.msc_selective_state_update_ex.restype = st
    lib.msc_selective_state_update_ex.argtypes = [vp] * 10 + [i64] * 3 + [st, st, vp]
    lib.msc_selective_scan_trap_fwd.restype = st
    lib.msc_selective_scan_trap_fwd.argtypes = ([vp] * 14 + [i64] * 4
                                                + [st, vp, ctypes.c_size_t, vp])
    lib.msc_selective_state_update_trap.restype = st
    lib.msc_selective_state_update_trap.argtypes = [vp] * 13 + [i64] * 3 + [st, vp]
    lib.msc_selective_scan_bwd.restype = st
    lib.msc_selective_scan_bwd.argtypes = [vp] * 20 + [i64] * 4 + [st, vp]
    lib.msc_selective_scan_bwd_ckpt.restype = st
    lib.msc_selective_scan_bwd_ckpt.argtypes = [vp] * 21 + [i64] * 4 + [st, vp]
    lib.msc_selective_scan_fwd_ckpt.restype = st
    lib.msc_selective_scan_fwd_ckpt.argtypes = ([vp] * 12 + [i64] * 4
                                                + [st, vp, sz, vp])
    lib.msc_scan_checkpoint_size.restype = st
    lib.msc_scan_checkpoint_size.argtypes = [i64] * 4 + [ctypes.POINTER(i64),
                                                         ctypes.POINTER(sz)]
    lib.msc_causal_conv1d_fwd.restype = st
    lib.msc_causal_conv1d_fwd.argtypes = [vp] * 6 + [i64] * 4 + [ctypes.c_int, st, vp]
    lib.msc_causal_conv1d_update.restype = st
    lib.msc_causal_conv1d_update.argtypes = [vp] * 5 + [i64] * 3 + [ctypes.c_int, st, vp]
    lib.msc_selective_scan_workspace_size.restype = st
    lib.msc_selective_scan_workspace_size.argtypes = [i64] * 4 + [
        st, ctypes.POINTER(sz)]
    lib.msc_selective_state_update.restype = st
    lib.msc_selective_state_update.argtypes = [vp] * 10 + [i64] * 3 + [st, vp]
    lib.msc_tuning_set.restype = st
    lib.msc_tuning_set.argtypes = [ctypes.c_char_p, i64]
    lib.msc_status_string.restype = ctypes.c_char_p
    lib.msc_status_string.argtypes = [st]
    lib.msc_version.restype = ctypes.c_int
    lib.msc_version.argtypes = []
    lib.msc_check_device_error.restype = st
    lib.msc_check_device_error.argtypes = [ctypes.c_int]
    lib.msc_scratch_release.restype = st
    lib.msc_scratch_release.argtypes = []
    lib.msc_profile_enable.restype = st
    lib.msc_profile_enable.argtypes = [ctypes.c_int]
    lib.msc_profile_read.restype = st
    lib.msc_profile_read.argtypes = [ctypes.POINTER(i64), ctypes.POINTER(i64),
                                     ctypes.POINTER(ctypes.c_double)]
    _lib = lib
    return lib


def _check(fn: str, status: int):
    if status != 0:
        raise MscError(fn, status)


def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return MSC_BF16
    if t.dtype == torch.float32:
        return MSC_F32
    raise TypeError(f"unsupported storage dtype {t.dtype} "
                    "(float32 or bfloat16)")


def _ptr(t, name, dtype=None, shape=None, device=None):
    if t is None:
        return None
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, "
                         f"expected {tuple(shape)}")
    return t.data_ptr()


def _stream(device):
    return _torch().cuda.current_stream(device).cuda_stream


def _scan_args(u, dt, A, B, C, D, z, dt_bias, out, last_state,
               return_last_state):
    torch = _torch()
    if u.dim() != 3 or B.dim() != 3:
        raise ValueError("u must be (batch, L, d_inner), B (batch, L, d_state)")
    batch, L, d_inner = u.shape
    d_state = B.shape[-1]
    dev = u.device
    code = _dtype_code(u)
    sdt = u.dtype
    f32 = torch.float32
    p = dict(
        u=_ptr(u, "u", sdt, (batch, L, d_inner), dev),
        dt=_ptr(dt, "dt", sdt, (batch, L, d_inner), dev),
        A=_ptr(A, "A", f32, (d_inner, d_state), dev),
        B=_ptr(B, "B", sdt, (batch, L, d_state), dev),
        C=_ptr(C, "C", sdt, (batch, L, d_state), dev),
        D=_ptr(D, "D", f32, (d_inner,), dev),
        z=_ptr(z, "z", sdt, (batch, L, d_inner), dev),
        dt_bias=_ptr(dt_bias, "dt_bias", f32, (d_inner,), dev),
    )
    if out is None:
        out = torch.empty((batch, L, d_inner), dtype=sdt, device=dev)
    p["out"] = _ptr(out, "out", sdt, (batch, L, d_inner), dev)
    if last_state is None and return_last_state:
        last_state = torch.empty((batch, d_inner, d_state), dtype=f32,
                                 device=dev)
    p["last_state"] = _ptr(last_state, "last_state", f32,
                           (batch, d_inner, d_state), dev)
    return p, out, last_state, (batch, L, d_inner, d_state), code, dev


def _scan_ex(fn, u, dt, A, B, C, D, z, dt_bias, out, last_state,
             return_last_state, h0, zoh, workspace):
    lib = load()
    p, out, last_state, dims, code, dev = _scan_args(
        u, dt, A, B, C, D, z, dt_bias, out, last_state, return_last_state)
    batch, _, d_inner, d_state = dims
    h0p = _ptr(h0, "h0", _torch().float32, (batch, d_inner, d_state), dev)
    wp = _ptr(workspace, "workspace", None, None, dev)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.msc_selective_scan_fwd_ex(
        p["u"], p["dt"], p["A"], p["B"], p["C"], p["D"], p["z"],
        p["dt_bias"], h0p, p["out"], p["last_state"], *dims, code,
        MSC_DISC_ZOH if zoh else MSC_DISC_EULER, wp, wbytes, _stream(dev))
    _check(fn, st)
    return out, last_state


def selective_scan_fwd(u, dt, A, B, C, D=None, z=None, dt_bias=None,
                       out=None, last_state=None, return_last_state=True,
                       h0=None, zoh=False):
    """Selective scan forward on the GPU -> (out, last_state).

    Enqueued on the current CUDA stream of u's device; returns at once.
    Scratch for the inter-chunk carry (when needed) is taken stream-ordered
    by the library.  h0: initial state (batch, d_inner, d_state) fp32, None
    for zero; zoh: zero-order-hold input matrix instead of delta*B.
    """
    if h0 is not None or zoh:
        return _scan_ex("msc_selective_scan_fwd_ex", u, dt, A, B, C, D, z,
                        dt_bias, out, last_state, return_last_state, h0, zoh,
                        None)
    lib = load()
    p, out, last_state, dims, code, dev = _scan_args(
        u, dt, A, B, C, D, z, dt_bias, out, last_state, return_last_state)
    st = lib.msc_selective_scan_fwd(
        p["u"], p["dt"], p["A"], p["B"], p["C"], p["D"], p["z"],
        p["dt_bias"], p["out"], p["last_state"], *dims, code, _stream(dev))
    _check("msc_selective_scan_fwd", st)
    return out, last_state


def scan_workspace_size(batch, L, d_inner, d_state, dtype) -> int:
    """Bytes of workspace selective_scan_fwd_ws needs on the current device."""
    torch = _torch()
    code = MSC_BF16 if dtype == torch.bfloat16 else MSC_F32
    n = ctypes.c_size_t(0)
    _check("msc_selective_scan_workspace_size",
           load().msc_selective_scan_workspace_size(
               batch, L, d_inner, d_state, code, ctypes.byref(n)))
    return int(n.value)


def selective_scan_fwd_ws(u, dt, A, B, C, D=None, z=None, dt_bias=None,
                          out=None, last_state=None, workspace=None,
                          return_last_state=True, h0=None, zoh=False):
    """As selective_scan_fwd with a caller-owned uint8 CUDA workspace."""
    if h0 is not None or zoh:
        if workspace is None and scan_workspace_size(
                u.shape[0], u.shape[1], u.shape[2], B.shape[-1], u.dtype) > 0:
            raise MscError("msc_selective_scan_fwd_ex", 5)
        return _scan_ex("msc_selective_scan_fwd_ex", u, dt, A, B, C, D, z,
                        dt_bias, out, last_state, return_last_state, h0, zoh,
                        workspace)
    lib = load()
    p, out, last_state, dims, code, dev = _scan_args(
        u, dt, A, B, C, D, z, dt_bias, out, last_state, return_last_state)
    wp = _ptr(workspace, "workspace", None, None, dev)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.msc_selective_scan_fwd_ws(
        p["u"], p["dt"], p["A"], p["B"], p["C"], p["D"], p["z"],
        p["dt_bias"], p["out"], p["last_state"], *dims, code, wp, wbytes,
        _stream(dev))
    _check("msc_selective_scan_fwd_ws", st)
    return out, last_state


def selective_state_update(state, u, dt, A, B, C, D=None, z=None,
                           dt_bias=None, out=None, zoh=False):
    """One decode step on the GPU; updates ``state`` in place -> out.
    zoh: zero-order-hold input matrix instead of delta*B."""
    torch = _torch()
    lib = load()
    if state.dim() != 3:
        raise ValueError("state must be (batch, d_inner, d_state)")
    batch, d_inner, d_state = state.shape
    dev = state.device
    code = _dtype_code(u)
    sdt = u.dtype
    f32 = torch.float32
    if out is None:
        out = torch.empty((batch, d_inner), dtype=sdt, device=dev)
    fn = "msc_selective_state_update_ex" if zoh else "msc_selective_state_update"
    extra = (MSC_DISC_ZOH,) if zoh else ()
    st = getattr(lib, fn)(
        _ptr(state, "state", f32, (batch, d_inner, d_state), dev),
        _ptr(u, "u", sdt, (batch, d_inner), dev),
        _ptr(dt, "dt", sdt, (batch, d_inner), dev),
        _ptr(A, "A", f32, (d_inner, d_state), dev),
        _ptr(B, "B", sdt, (batch, d_state), dev),
        _ptr(C, "C", sdt, (batch, d_state), dev),
        _ptr(D, "D", f32, (d_inner,), dev),
        _ptr(z, "z", sdt, (batch, d_inner), dev),
        _ptr(dt_bias, "dt_bias", f32, (d_inner,), dev),
        _ptr(out, "out", sdt, (batch, d_inner), dev),
        batch, d_inner, d_state, code, *extra, _stream(dev))
    _check(fn, st)
    return out


def selective_scan_trap_fwd(u, dt, lam, A, B, C, D=None, z=None, dt_bias=None,
                            h0=None, u_prev=None, B_prev=None, out=None,
                            last_state=None, workspace=None, return_last_state=True):
    """Exponential-trapezoid scan on the GPU -> (out, last_state).

    lam: (batch, L, d_inner) in u's dtype, values in [0, 1]; u_prev
    (batch, d_inner) and B_prev (batch, d_state): the step before t = 0."""
    lib = load()
    p, out, last_state, dims, code, dev = _scan_args(
        u, dt, A, B, C, D, z, dt_bias, out, last_state, return_last_state)
    batch, L, d_inner, d_state = dims
    sdt = u.dtype
    wp = _ptr(workspace, "workspace", None, None, dev)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.msc_selective_scan_trap_fwd(
        p["u"], p["dt"], _ptr(lam, "lam", sdt, (batch, L, d_inner), dev), p["A"], p["B"],
        p["C"], p["D"], p["z"], p["dt_bias"],
        _ptr(h0, "h0", _torch().float32, (batch, d_inner, d_state), dev),
        _ptr(u_prev, "u_prev", sdt, (batch, d_inner), dev),
        _ptr(B_prev, "B_prev", sdt, (batch, d_state), dev),
        p["out"], p["last_state"], *dims, code, wp, wbytes, _stream(dev))
    _check("msc_selective_scan_trap_fwd", st)
    return out, last_state


def selective_state_update_trap(state, u_prev, B_prev, u, dt, lam, A, B, C, D=None,
                                z=None, dt_bias=None, out=None):
    """One exponential-trapezoid decode token; updates ``state`` -> out."""
    torch = _torch()
    batch, d_inner, d_state = state.shape
    dev, sdt, f32 = state.device, u.dtype, torch.float32
    code = _dtype_code(u)
    if out is None:
        out = torch.empty((batch, d_inner), dtype=sdt, device=dev)
    st = load().msc_selective_state_update_trap(
        _ptr(state, "state", f32, (batch, d_inner, d_state), dev),
        _ptr(u_prev, "u_prev", sdt, (batch, d_inner), dev),
        _ptr(B_prev, "B_prev", sdt, (batch, d_state), dev),
        _ptr(u, "u", sdt, (batch, d_inner), dev),
        _ptr(dt, "dt", sdt, (batch, d_inner), dev),
        _ptr(lam, "lam", sdt, (batch, d_inner), dev),
        _ptr(A, "A", f32, (d_inner, d_state), dev),
        _ptr(B, "B", sdt, (batch, d_state), dev),
        _ptr(C, "C", sdt, (batch, d_state), dev),
        _ptr(D, "D", f32, (d_inner,), dev),
        _ptr(z, "z", sdt, (batch, d_inner), dev),
        _ptr(dt_bias, "dt_bias", f32, (d_inner,), dev),
        _ptr(out, "out", sdt, (batch, d_inner), dev),
        batch, d_inner, d_state, code, _stream(dev))
    _check("msc_selective_state_update_trap", st)
    return out


def scan_checkpoint_size(batch, L, d_inner, d_state):
    """(interval, bytes) of the checkpoint array selective_scan_fwd_ckpt
    writes: (batch, ceil(L / interval), d_inner, d_state) fp32."""
    tt, n = ctypes.c_int64(0), ctypes.c_size_t(0)
    _check("msc_scan_checkpoint_size", load().msc_scan_checkpoint_size(
        batch, L, d_inner, d_state, ctypes.byref(tt), ctypes.byref(n)))
    return int(tt.value), int(n.value)


def selective_scan_fwd_ckpt(u, dt, A, B, C, D=None, z=None, dt_bias=None,
                            h0=None, out=None, last_state=None, ckpt=None):
    """Euler selective scan that also writes the backward's checkpoints
    -> (out, last_state, ckpt); ckpt is (batch, rows, d_inner, d_state) fp32,
    row k the state entering step k * interval (scan_checkpoint_size)."""
    lib = load()
    torch = _torch()
    p, out, last_state, dims, code, dev = _scan_args(
        u, dt, A, B, C, D, z, dt_bias, out, last_state, True)
    batch, L, d_inner, d_state = dims
    tt, _ = scan_checkpoint_size(batch, L, d_inner, d_state)
    shape = (batch, (L + tt - 1) // tt, d_inner, d_state)
    if ckpt is None:
        ckpt = torch.empty(shape, dtype=torch.float32, device=dev)
    cp = _ptr(ckpt, "ckpt", torch.float32, shape, dev)
    h0p = _ptr(h0, "h0", torch.float32, (batch, d_inner, d_state), dev)
    st = lib.msc_selective_scan_fwd_ckpt(
        p["u"], p["dt"], p["A"], p["B"], p["C"], p["D"], p["z"],
        p["dt_bias"], h0p, p["out"], p["last_state"], cp, *dims, code, None, 0,
        _stream(dev))
    _check("msc_selective_scan_fwd_ckpt", st)
    return out, last_state, ckpt


def selective_scan_bwd(u, dt, A, B, C, D=None, z=None, dt_bias=None, h0=None,
                       dout=None, dlast_state=None, want_dh0=False, ckpt=None):
    """Backward pass of selective_scan_fwd on the GPU -> dict of gradients:
    du, ddt, dz (u's dtype), dA, dB, dC, dD, ddt_bias, dh0 (fp32; dz, dD,
    ddt_bias None when z, D, dt_bias are None; dh0 only with want_dh0).
    ckpt: the checkpoints selective_scan_fwd_ckpt wrote for these inputs,
    read instead of recomputed (None: recomputed)."""
    torch = _torch()
    batch, L, d_inner = u.shape
    d_state = B.shape[-1]
    dev, sdt, f32 = u.device, u.dtype, torch.float32
    code = _dtype_code(u)
    g = dict(du=torch.empty_like(u), ddt=torch.empty_like(u),
             dz=torch.empty_like(u) if z is not None else None,
             dA=torch.empty(d_inner, d_state, dtype=f32, device=dev),
             dB=torch.empty(batch, L, d_state, dtype=f32, device=dev),
             dC=torch.empty(batch, L, d_state, dtype=f32, device=dev),
             dD=torch.empty(d_inner, dtype=f32, device=dev) if D is not None else None,
             ddt_bias=torch.empty(d_inner, dtype=f32, device=dev) if dt_bias is not None else None,
             dh0=torch.empty(batch, d_inner, d_state, dtype=f32, device=dev) if want_dh0 else None)
    P = lambda t, name, dt_=None, shape=None: _ptr(t, name, dt_, shape, dev)
    head = [
        P(u, "u", sdt, (batch, L, d_inner)), P(dt, "dt", sdt, (batch, L, d_inner)),
        P(A, "A", f32, (d_inner, d_state)), P(B, "B", sdt, (batch, L, d_state)),
        P(C, "C", sdt, (batch, L, d_state)), P(D, "D", f32, (d_inner,)),
        P(z, "z", sdt, (batch, L, d_inner)), P(dt_bias, "dt_bias", f32, (d_inner,)),
        P(h0, "h0", f32, (batch, d_inner, d_state))]
    fn = "msc_selective_scan_bwd"
    if ckpt is not None:
        fn = "msc_selective_scan_bwd_ckpt"
        tt, _ = scan_checkpoint_size(batch, L, d_inner, d_state)
        head.append(P(ckpt, "ckpt", f32, (batch, (L + tt - 1) // tt, d_inner, d_state)))
    st = getattr(load(), fn)(
        *head, P(dout, "dout", sdt, (batch, L, d_inner)),
        P(dlast_state, "dlast_state", f32, (batch, d_inner, d_state)),
        g["du"].data_ptr(), g["ddt"].data_ptr(), g["dA"].data_ptr(), g["dB"].data_ptr(),
        g["dC"].data_ptr(), None if g["dD"] is None else g["dD"].data_ptr(),
        None if g["dz"] is None else g["dz"].data_ptr(),
        None if g["ddt_bias"] is None else g["ddt_bias"].data_ptr(),
        None if g["dh0"] is None else g["dh0"].data_ptr(),
        batch, L, d_inner, d_state, code, _stream(dev))
    _check(fn, st)
    return g


_SCAN_FN = None


def _scan_function():
    """The autograd Function of selective_scan (defined on first use, since
    torch is imported lazily)."""
    global _SCAN_FN
    if _SCAN_FN is not None:
        return _SCAN_FN
    torch = _torch()

    class SelectiveScanFn(torch.autograd.Function):
        @staticmethod
        def forward(ctx, u, dt, A, B, C, D, z, dt_bias, h0):
            ck = None
            try:  # the forward that also writes the backward's checkpoints
                out, last, ck = selective_scan_fwd_ckpt(u, dt, A, B, C, D, z, dt_bias, h0=h0)
            except MscError as e:
                if e.status != 2:  # only unsupported shapes take the plain forward
                    raise
                out, last = selective_scan_fwd(u, dt, A, B, C, D, z, dt_bias, h0=h0)
            ctx.save_for_backward(u, dt, A, B, C, D, z, dt_bias, h0, ck)
            return out, last

        @staticmethod
        def backward(ctx, dout, dlast):
            u, dt, A, B, C, D, z, dt_bias, h0, ck = ctx.saved_tensors
            dout = (torch.zeros_like(u) if dout is None
                    else dout.to(u.dtype).contiguous())
            dlast = None if dlast is None else dlast.float().contiguous()
            want_dh0 = h0 is not None and ctx.needs_input_grad[8]
            try:
                g = selective_scan_bwd(u, dt, A, B, C, D, z, dt_bias, h0=h0, dout=dout,
                                       dlast_state=dlast, want_dh0=want_dh0, ckpt=ck)
            except MscError as e:
                if ck is None or e.status != 2:
                    raise
                g = selective_scan_bwd(u, dt, A, B, C, D, z, dt_bias, h0=h0, dout=dout,
                                       dlast_state=dlast, want_dh0=want_dh0)
            return (g["du"], g["ddt"], g["dA"], g["dB"].to(B.dtype), g["dC"].to(C.dtype),
                    g["dD"], g["dz"], g["ddt_bias"], g["dh0"])

    _SCAN_FN = SelectiveScanFn
    return _SCAN_FN


def selective_scan(u, dt, A, B, C, D=None, z=None, dt_bias=None, h0=None):
    """Differentiable selective scan (the Euler form) -> (out, last_state).

    Forward: selective_scan_fwd_ckpt where the shape allows (the state
    entering every backward tile is kept for the backward), else
    selective_scan_fwd.  Backward: selective_scan_bwd from those
    checkpoints (or recomputing them).  Gradients of B and C are cast to
    their storage dtype; the others keep the dtypes of selective_scan_bwd."""
    return _scan_function().apply(u, dt, A, B, C, D, z, dt_bias, h0)


def causal_conv1d_fwd(x, w, bias=None, state_in=None, out=None, state_out=None,
                      silu=True, return_state=True):
    """Causal depthwise conv1d (+ SiLU) on the GPU -> (out, state_out).

    x: (batch, L, d_inner) bf16/fp32; w: (d_inner, d_conv) fp32; bias:
    (d_inner) fp32; state_in / state_out: (batch, d_inner, d_conv - 1) in
    x's dtype (the inputs before t = 0 / the last d_conv - 1 inputs)."""
    torch = _torch()
    if x.dim() != 3 or w.dim() != 2:
        raise ValueError("x must be (batch, L, d_inner), w (d_inner, d_conv)")
    batch, L, d_inner = x.shape
    d_conv = w.shape[1]
    dev, sdt, f32 = x.device, x.dtype, torch.float32
    code = _dtype_code(x)
    if out is None:
        out = torch.empty_like(x)
    if state_out is None and return_state:
        state_out = torch.empty((batch, d_inner, d_conv - 1), dtype=sdt, device=dev)
    st = load().msc_causal_conv1d_fwd(
        _ptr(x, "x", sdt, (batch, L, d_inner), dev),
        _ptr(w, "w", f32, (d_inner, d_conv), dev),
        _ptr(bias, "bias", f32, (d_inner,), dev),
        _ptr(state_in, "state_in", sdt, (batch, d_inner, d_conv - 1), dev),
        _ptr(out, "out", sdt, (batch, L, d_inner), dev),
        _ptr(state_out, "state_out", sdt, (batch, d_inner, d_conv - 1), dev),
        batch, L, d_inner, d_conv, int(bool(silu)), code, _stream(dev))
    _check("msc_causal_conv1d_fwd", st)
    return out, state_out


def causal_conv1d_update(state, x, w, bias=None, out=None, silu=True):
    """One decode token of the conv; updates ``state`` in place -> out."""
    if x.dim() != 2:
        raise ValueError("x must be (batch, d_inner)")
    batch, d_inner = x.shape
    d_conv = w.shape[1]
    dev, sdt = x.device, x.dtype
    code = _dtype_code(x)
    if out is None:
        out = _torch().empty_like(x)
    st = load().msc_causal_conv1d_update(
        _ptr(state, "state", sdt, (batch, d_inner, d_conv - 1), dev),
        _ptr(x, "x", sdt, (batch, d_inner), dev),
        _ptr(w, "w", _torch().float32, (d_inner, d_conv), dev),
        _ptr(bias, "bias", _torch().float32, (d_inner,), dev),
        _ptr(out, "out", sdt, (batch, d_inner), dev),
        batch, d_inner, d_conv, int(bool(silu)), code, _stream(dev))
    _check("msc_causal_conv1d_update", st)
    return out


def check_device_error(clear: bool = True):
    """Raise MscError(MSC_ERR_TIMEOUT) if a kernel's bounded wait gave up.
    Synchronise the streams used first."""
    _check("msc_check_device_error", load().msc_check_device_error(int(clear)))


def scratch_release():
    """Return the memory the library's scratch pools hold unused to the device."""
    _check("msc_scratch_release", load().msc_scratch_release())


def profile_enable(on: bool = True):
    """Start/stop recording event pairs around each call's main kernel."""
    _check("msc_profile_enable", load().msc_profile_enable(int(on)))


_PROF_KINDS = ("scan", "update", "conv", "conv_update", "scan_bwd")  # MSC_PROF_* order


def profile_read():
    """Since the last read: (kernels launched, {kind: (timed, ms)}) for the
    kinds "scan", "update", "conv", "conv_update" -- main-kernel counts and
    summed device time.  Synchronises the recorded events, then resets."""
    n = ctypes.c_int64(0)
    timed = (ctypes.c_int64 * len(_PROF_KINDS))()
    ms = (ctypes.c_double * len(_PROF_KINDS))()
    _check("msc_profile_read", load().msc_profile_read(ctypes.byref(n), timed, ms))
    return int(n.value), {k: (int(timed[i]), float(ms[i]))
                          for i, k in enumerate(_PROF_KINDS)}


def tuning_set(key: str, value: int):
    """Process-wide plan override (see msc_tuning_set in include/msc.h)."""
    _check("msc_tuning_set", load().msc_tuning_set(key.encode(), int(value)))
