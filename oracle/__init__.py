"""fp64 CPU oracle for the Mamba selective scan and selective state update.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline leg may import this package.  It shares no code
with the CUDA path: ``oracle.c`` is plain C built with gcc (``-O2``, no
fast-math, OpenMP over channels) and loaded here through ctypes.

Every function takes numpy arrays, upcasts them to float64 exactly, and
returns float64 results.  Shapes follow the listings of "Deep dive into
Mamba" section 4.4 and the MambaBlock of "State space models and Mamba":
u, dt_raw, z: (batch, L, d_inner); B, C: (batch, L, d_state);
A: (d_inner, d_state); D, dt_bias: (d_inner,).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile ``src`` (default oracle.c) into the shared library ``out``."""
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-fno-fast-math", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _f64(x):
    if x is None:
        return None
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(x):
    if x is None:
        return ctypes.POINTER(ctypes.c_double)()
    return x.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _dims(u, B):
    batch, L, d_inner = u.shape
    d_state = B.shape[-1]
    return batch, L, d_inner, d_state


class Oracle:
    """ctypes view of one build of oracle.c."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        dp = ctypes.POINTER(ctypes.c_double)
        i64 = ctypes.c_int64
        lib.oracle_softplus.restype = ctypes.c_double
        lib.oracle_softplus.argtypes = [ctypes.c_double]
        lib.oracle_silu.restype = ctypes.c_double
        lib.oracle_silu.argtypes = [ctypes.c_double]
        lib.oracle_threads.restype = ctypes.c_int
        lib.oracle_threads.argtypes = [ctypes.c_int]
        lib.oracle_scan_fwd.restype = ctypes.c_int
        lib.oracle_scan_fwd.argtypes = [dp] * 11 + [i64] * 4 + [ctypes.c_int] * 2
        lib.oracle_state_update.restype = ctypes.c_int
        lib.oracle_state_update.argtypes = [dp] * 10 + [i64] * 3 + [ctypes.c_int] * 2
        lib.oracle_scan_fwd_segmented.restype = ctypes.c_int
        lib.oracle_scan_fwd_segmented.argtypes = ([dp] * 10 + [i64] * 5
                                                  + [ctypes.c_int])
        lib.oracle_scan_fwd_trap.restype = ctypes.c_int
        lib.oracle_scan_fwd_trap.argtypes = [dp] * 14 + [i64] * 4 + [ctypes.c_int]
        lib.oracle_state_update_trap.restype = ctypes.c_int
        lib.oracle_state_update_trap.argtypes = [dp] * 13 + [i64] * 3 + [ctypes.c_int]
        lib.oracle_scan_bwd.restype = ctypes.c_int
        lib.oracle_scan_bwd.argtypes = [dp] * 20 + [i64] * 4
        lib.oracle_causal_conv1d.restype = ctypes.c_int
        lib.oracle_causal_conv1d.argtypes = [dp] * 6 + [i64] * 4 + [ctypes.c_int] * 2
        lib.oracle_conv1d_update.restype = ctypes.c_int
        lib.oracle_conv1d_update.argtypes = [dp] * 5 + [i64] * 3 + [ctypes.c_int] * 2
        self.lib = lib
        self.path = lib_path

    def threads(self, nthreads: int = 0) -> int:
        """Number of OpenMP threads a call with ``nthreads`` uses (0 = all)."""
        return int(self.lib.oracle_threads(int(nthreads)))

    def softplus(self, x: float) -> float:
        """log(1 + e^x), evaluated without overflow (scalar)."""
        return float(self.lib.oracle_softplus(float(x)))

    def silu(self, z: float) -> float:
        """z * sigmoid(z) (scalar)."""
        return float(self.lib.oracle_silu(float(z)))

    def scan_fwd(self, u, dt_raw, A, B, C, D=None, z=None, dt_bias=None,
                 h0=None, zoh: bool = False, nthreads: int = 0):
        """Selective scan forward in fp64.  Returns (out, last_state).

        h0: initial state (batch, d_inner, d_state), None for zero.
        zoh: zero-order-hold input matrix instead of delta*B."""
        u, dt_raw, A, B, C = map(_f64, (u, dt_raw, A, B, C))
        D, z, dt_bias, h0 = map(_f64, (D, z, dt_bias, h0))
        batch, L, d_inner, d_state = _dims(u, B)
        out = np.zeros((batch, L, d_inner), dtype=np.float64)
        last = np.zeros((batch, d_inner, d_state), dtype=np.float64)
        rc = self.lib.oracle_scan_fwd(
            _ptr(u), _ptr(dt_raw), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
            _ptr(z), _ptr(dt_bias), _ptr(h0), _ptr(out), _ptr(last), batch,
            L, d_inner, d_state, int(bool(zoh)), int(nthreads))
        if rc != 0:
            raise ValueError("oracle_scan_fwd rejected its sizes")
        return out, last

    def scan_fwd_segmented(self, u, dt_raw, A, B, C, D=None, z=None,
                           dt_bias=None, seg: int = 64, nthreads: int = 0):
        """Segmented scan with the associative merge -> (out, last_state)."""
        u, dt_raw, A, B, C = map(_f64, (u, dt_raw, A, B, C))
        D, z, dt_bias = map(_f64, (D, z, dt_bias))
        batch, L, d_inner, d_state = _dims(u, B)
        out = np.zeros((batch, L, d_inner), dtype=np.float64)
        last = np.zeros((batch, d_inner, d_state), dtype=np.float64)
        rc = self.lib.oracle_scan_fwd_segmented(
            _ptr(u), _ptr(dt_raw), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
            _ptr(z), _ptr(dt_bias), _ptr(out), _ptr(last), batch, L,
            d_inner, d_state, int(seg), int(nthreads))
        if rc != 0:
            raise ValueError("oracle_scan_fwd_segmented rejected its sizes")
        return out, last

    def state_update(self, state, u, dt_raw, A, B, C, D=None, z=None,
                     dt_bias=None, zoh: bool = False, nthreads: int = 0):
        """One decode step in fp64 -> (new_state, out); inputs untouched.

        state: (batch, d_inner, d_state); u, dt_raw, z: (batch, d_inner);
        B, C: (batch, d_state).
        """
        st = np.array(state, dtype=np.float64, copy=True, order="C")
        u, dt_raw, A, B, C = map(_f64, (u, dt_raw, A, B, C))
        D, z, dt_bias = map(_f64, (D, z, dt_bias))
        batch, d_inner, d_state = st.shape
        out = np.zeros((batch, d_inner), dtype=np.float64)
        rc = self.lib.oracle_state_update(
            _ptr(st), _ptr(u), _ptr(dt_raw), _ptr(A), _ptr(B), _ptr(C),
            _ptr(D), _ptr(z), _ptr(dt_bias), _ptr(out), batch, d_inner,
            d_state, int(bool(zoh)), int(nthreads))
        if rc != 0:
            raise ValueError("oracle_state_update rejected its sizes")
        return st, out

    def scan_fwd_trap(self, u, dt_raw, lam, A, B, C, D=None, z=None, dt_bias=None,
                      h0=None, u_prev=None, B_prev=None, nthreads: int = 0):
        """Exponential-trapezoid scan in fp64 -> (out, last_state).

        lam: (batch, L, d_inner); u_prev: (batch, d_inner) and B_prev:
        (batch, d_state) are the step before t = 0 (None: zero)."""
        u, dt_raw, lam, A, B, C = map(_f64, (u, dt_raw, lam, A, B, C))
        D, z, dt_bias, h0, u_prev, B_prev = map(_f64, (D, z, dt_bias, h0, u_prev, B_prev))
        batch, L, d_inner, d_state = _dims(u, B)
        out = np.zeros((batch, L, d_inner), dtype=np.float64)
        last = np.zeros((batch, d_inner, d_state), dtype=np.float64)
        rc = self.lib.oracle_scan_fwd_trap(
            _ptr(u), _ptr(dt_raw), _ptr(lam), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
            _ptr(z), _ptr(dt_bias), _ptr(h0), _ptr(u_prev), _ptr(B_prev), _ptr(out),
            _ptr(last), batch, L, d_inner, d_state, int(nthreads))
        if rc != 0:
            raise ValueError("oracle_scan_fwd_trap rejected its sizes")
        return out, last

    def state_update_trap(self, state, u_prev, B_prev, u, dt_raw, lam, A, B, C,
                          D=None, z=None, dt_bias=None, nthreads: int = 0):
        """One trapezoid decode token in fp64 -> (new_state, out)."""
        st = np.array(state, dtype=np.float64, copy=True, order="C")
        u_prev, B_prev, u, dt_raw, lam, A, B, C = map(
            _f64, (u_prev, B_prev, u, dt_raw, lam, A, B, C))
        D, z, dt_bias = map(_f64, (D, z, dt_bias))
        batch, d_inner, d_state = st.shape
        out = np.zeros((batch, d_inner), dtype=np.float64)
        rc = self.lib.oracle_state_update_trap(
            _ptr(st), _ptr(u_prev), _ptr(B_prev), _ptr(u), _ptr(dt_raw), _ptr(lam),
            _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(dt_bias), _ptr(out),
            batch, d_inner, d_state, int(nthreads))
        if rc != 0:
            raise ValueError("oracle_state_update_trap rejected its sizes")
        return st, out

    def scan_bwd(self, u, dt_raw, A, B, C, D=None, z=None, dt_bias=None, h0=None,
                 dout=None, dlast=None):
        """Gradients of the scan in fp64 -> dict du, ddt, dA, dB, dC, dD, dz,
        ddt_bias, dh0 (dz None without z)."""
        u, dt_raw, A, B, C, dout = map(_f64, (u, dt_raw, A, B, C, dout))
        D, z, dt_bias, h0, dlast = map(_f64, (D, z, dt_bias, h0, dlast))
        batch, L, d_inner, d_state = _dims(u, B)
        g = dict(du=np.zeros((batch, L, d_inner)), ddt=np.zeros((batch, L, d_inner)),
                 dA=np.zeros((d_inner, d_state)), dB=np.zeros((batch, L, d_state)),
                 dC=np.zeros((batch, L, d_state)), dD=np.zeros(d_inner),
                 dz=np.zeros((batch, L, d_inner)), ddt_bias=np.zeros(d_inner),
                 dh0=np.zeros((batch, d_inner, d_state)))
        rc = self.lib.oracle_scan_bwd(
            _ptr(u), _ptr(dt_raw), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
            _ptr(dt_bias), _ptr(h0), _ptr(dout), _ptr(dlast), _ptr(g["du"]),
            _ptr(g["ddt"]), _ptr(g["dA"]), _ptr(g["dB"]), _ptr(g["dC"]), _ptr(g["dD"]),
            _ptr(g["dz"]), _ptr(g["ddt_bias"]), _ptr(g["dh0"]), batch, L, d_inner,
            d_state)
        if rc != 0:
            raise ValueError("oracle_scan_bwd rejected its sizes")
        if z is None:
            g["dz"] = None
        return g

    def causal_conv1d(self, x, w, bias=None, state_in=None, silu: bool = True,
                      nthreads: int = 0):
        """Causal depthwise conv1d (+ SiLU) in fp64 -> (out, state_out).

        x: (batch, L, d_inner); w: (d_inner, d_conv); bias: (d_inner);
        state_in / state_out: (batch, d_inner, d_conv - 1), oldest first."""
        x, w = _f64(x), _f64(w)
        bias, state_in = _f64(bias), _f64(state_in)
        batch, L, d_inner = x.shape
        d_conv = w.shape[1]
        out = np.zeros((batch, L, d_inner), dtype=np.float64)
        st = np.zeros((batch, d_inner, d_conv - 1), dtype=np.float64)
        rc = self.lib.oracle_causal_conv1d(
            _ptr(x), _ptr(w), _ptr(bias), _ptr(state_in), _ptr(out), _ptr(st),
            batch, L, d_inner, d_conv, int(bool(silu)), int(nthreads))
        if rc != 0:
            raise ValueError("oracle_causal_conv1d rejected its sizes")
        return out, st

    def conv1d_update(self, state, x, w, bias=None, silu: bool = True,
                      nthreads: int = 0):
        """One decode step of the conv -> (new_state, out); inputs untouched."""
        st = np.array(state, dtype=np.float64, copy=True, order="C")
        x, w, bias = _f64(x), _f64(w), _f64(bias)
        batch, d_inner = x.shape
        d_conv = w.shape[1]
        out = np.zeros((batch, d_inner), dtype=np.float64)
        rc = self.lib.oracle_conv1d_update(
            _ptr(st), _ptr(x), _ptr(w), _ptr(bias), _ptr(out), batch, d_inner,
            d_conv, int(bool(silu)), int(nthreads))
        if rc != 0:
            raise ValueError("oracle_conv1d_update rejected its sizes")
        return st, out


_default = None


def default() -> Oracle:
    """The oracle built from oracle.c (compiled on first use)."""
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default


def threads(nthreads: int = 0) -> int:
    return default().threads(nthreads)


def softplus(x: float) -> float:
    return default().softplus(x)


def silu(z: float) -> float:
    return default().silu(z)


def scan_fwd(*args, **kwargs):
    return default().scan_fwd(*args, **kwargs)


def scan_fwd_segmented(*args, **kwargs):
    return default().scan_fwd_segmented(*args, **kwargs)


def state_update(*args, **kwargs):
    return default().state_update(*args, **kwargs)


def causal_conv1d(*args, **kwargs):
    return default().causal_conv1d(*args, **kwargs)


def conv1d_update(*args, **kwargs):
    return default().conv1d_update(*args, **kwargs)


def scan_fwd_trap(*args, **kwargs):
    return default().scan_fwd_trap(*args, **kwargs)


def state_update_trap(*args, **kwargs):
    return default().state_update_trap(*args, **kwargs)


def scan_bwd(*args, **kwargs):
    return default().scan_bwd(*args, **kwargs)
