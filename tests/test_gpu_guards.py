"""Out-of-bounds and missed writes, without a sanitizer: every buffer an
entry point writes is a view inside a larger allocation whose margins (64 KB
before and after) hold a NaN sentinel.  After the call the margins must be
bit for bit unchanged (no write outside the buffer), and a buffer the call
must fill whole must hold no sentinel (no element left unwritten).  The
shapes are ragged: partial channel tiles, lengths off every tile and octet
size, odd batch counts, time chunks, d_state 8 to 64."""
import numpy as np
import pytest

import selective_state_space_144_b300 as msc
from selective_state_space_144_b300 import synth
from tests.helpers import scan_device_args, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

GUARD_BYTES = 64 * 1024
# NaN payloads no kernel produces (an arithmetic NaN is the canonical one)
SENTINEL = {torch.float32: 0x7FA1B2C3, torch.bfloat16: 0x7FA1}
INT_VIEW = {torch.float32: torch.int32, torch.bfloat16: torch.int16}


class Guarded:
    """A tensor of `shape` and `dtype` inside a sentinel-filled allocation;
    `init` (a tensor) gives it starting contents (in/out buffers)."""

    def __init__(self, shape, dtype, init=None):
        es = torch.empty((), dtype=dtype).element_size()
        self.g = GUARD_BYTES // es
        self.n = int(np.prod(shape))
        self.dtype = dtype
        self.flat = torch.empty(self.n + 2 * self.g, dtype=dtype, device="cuda")
        self.flat.view(INT_VIEW[dtype]).fill_(self._sentinel())
        self.t = self.flat[self.g:self.g + self.n].view(shape)
        if init is not None:
            self.t.copy_(init)

    def _sentinel(self):
        s = SENTINEL[self.dtype]
        return s if self.dtype == torch.float32 else s - (1 << 16) if s >= 1 << 15 else s

    def check(self, name, full=True):
        torch.cuda.synchronize()
        bits = self.flat.view(INT_VIEW[self.dtype])
        s = self._sentinel()
        head, tail = bits[:self.g], bits[self.g + self.n:]
        assert bool((head == s).all()), f"{name}: write before the buffer"
        assert bool((tail == s).all()), f"{name}: write past the buffer"
        if full:
            inner = bits[self.g:self.g + self.n]
            left = int((inner == s).sum())
            assert left == 0, f"{name}: {left} of {self.n} elements not written"


SCAN_SHAPES = [  # (batch, L, d_inner, d_state, dtype, chunks)
    (2, 77, 40, 16, "bf16", 0),    # TMA path: 5 channel tiles, partial last tile
    (3, 45, 33, 16, "f32", 0),     # element-load path (d_inner not a multiple of 8)
    (2, 100, 48, 32, "bf16", 0),
    (1, 130, 16, 8, "f32", 0),
    (2, 201, 64, 16, "bf16", 3),   # time chunks: summary, carry prefix, outputs
    (1, 70, 24, 64, "f32", 2),
]


@pytest.mark.parametrize("batch,L,d_inner,N,dtype,chunks", SCAN_SHAPES)
@pytest.mark.parametrize("variant", ["euler", "zoh_h0", "trapezoid"])
def test_scan_writes_stay_inside(batch, L, d_inner, N, dtype, chunks, variant):
    x = synth.scan_inputs(batch, L, d_inner, N, dtype=dtype, seed=2000 + L, D="normal")
    a = scan_device_args(x)
    sdt = a["u"].dtype
    out = Guarded((batch, L, d_inner), sdt)
    last = Guarded((batch, d_inner, N), torch.float32)
    msc.tuning_set("scan_chunks", chunks)
    try:
        if variant == "euler":
            msc.selective_scan_fwd(**a, out=out.t, last_state=last.t)
        elif variant == "zoh_h0":
            h0 = torch.randn(batch, d_inner, N, device="cuda")
            msc.selective_scan_fwd(**a, out=out.t, last_state=last.t, h0=h0, zoh=True)
        else:
            lam = to_device(synth.round_bf16(np.random.default_rng(L).uniform(
                0, 1, (batch, L, d_inner)).astype(np.float32)), dtype)
            up = to_device(x.u[:, 0], dtype)
            Bp = to_device(x.B[:, 0], dtype)
            msc.selective_scan_trap_fwd(a["u"], a["dt"], lam, a["A"], a["B"], a["C"], a["D"],
                                        a["z"], a["dt_bias"], u_prev=up, B_prev=Bp,
                                        out=out.t, last_state=last.t)
    finally:
        msc.tuning_set("scan_chunks", 0)
    out.check("out")
    last.check("last_state")
    msc.check_device_error()


@pytest.mark.parametrize("batch,L,d_inner,N,dtype", [
    (2, 77, 40, 16, "bf16"), (3, 45, 32, 8, "f32"), (1, 70, 24, 64, "bf16"),
    (2, 33, 16, 32, "f32")])
def test_checkpointing_forward_and_backward_writes_stay_inside(batch, L, d_inner, N, dtype):
    """The checkpointing forward (out, last_state, checkpoints) and both
    backward entry points (every gradient, dh0 included), through the C ABI
    with guarded buffers."""
    x = synth.scan_inputs(batch, L, d_inner, N, dtype=dtype, seed=2100 + L, D="normal")
    a = scan_device_args(x)
    sdt, f32 = a["u"].dtype, torch.float32
    h0 = torch.randn(batch, d_inner, N, device="cuda")
    tt, _ = msc.scan_checkpoint_size(batch, L, d_inner, N)
    out = Guarded((batch, L, d_inner), sdt)
    last = Guarded((batch, d_inner, N), f32)
    ck = Guarded((batch, (L + tt - 1) // tt, d_inner, N), f32)
    msc.selective_scan_fwd_ckpt(**a, h0=h0, out=out.t, last_state=last.t, ckpt=ck.t)
    for name, g in (("out", out), ("last_state", last), ("ckpt", ck)):
        g.check(name)

    dout = torch.randn(batch, L, d_inner, device="cuda").to(sdt)
    dlast = torch.randn(batch, d_inner, N, device="cuda")
    lib = msc.load()
    P = lambda t: None if t is None else t.data_ptr()
    for use_ckpt in (False, True):
        g = dict(du=Guarded((batch, L, d_inner), sdt), ddt=Guarded((batch, L, d_inner), sdt),
                 dA=Guarded((d_inner, N), f32), dB=Guarded((batch, L, N), f32),
                 dC=Guarded((batch, L, N), f32), dD=Guarded((d_inner,), f32),
                 dz=Guarded((batch, L, d_inner), sdt), ddt_bias=Guarded((d_inner,), f32),
                 dh0=Guarded((batch, d_inner, N), f32))
        head = [P(a["u"]), P(a["dt"]), P(a["A"]), P(a["B"]), P(a["C"]), P(a["D"]),
                P(a["z"]), P(a["dt_bias"]), P(h0)]
        fn = lib.msc_selective_scan_bwd
        if use_ckpt:
            fn = lib.msc_selective_scan_bwd_ckpt
            head.append(P(ck.t))
        st = fn(*head, P(dout), P(dlast), *[P(g[k].t) for k in (
            "du", "ddt", "dA", "dB", "dC", "dD", "dz", "ddt_bias", "dh0")],
            batch, L, d_inner, N, 1 if dtype == "bf16" else 0,
            torch.cuda.current_stream().cuda_stream)
        assert st == 0, msc.load().msc_status_string(st)
        for k, v in g.items():
            v.check(f"{k} (from checkpoints: {use_ckpt})")
    msc.check_device_error()


DECODE_SHAPES = [  # (batch, d_inner, d_state): stream, row and general kernels
    (3, 136, 16), (5, 50, 16), (4, 72, 64), (9, 264, 8), (6, 200, 32), (2, 30, 5)]


@pytest.mark.parametrize("batch,d_inner,N", DECODE_SHAPES)
@pytest.mark.parametrize("variant", ["euler", "zoh", "trapezoid"])
@pytest.mark.parametrize("path", [0, 1])
def test_decode_writes_stay_inside(batch, d_inner, N, variant, path):
    """The state updated in place and the token's output, on both decode
    kernel choices; two tokens so that the trapezoid's second one reads the
    previous token's u and B."""
    p = synth.decode_params(batch, d_inner, N, seed=2200 + d_inner, dtype="bf16")
    A, D, bias = to_device(p.A, "f32"), to_device(p.D, "f32"), to_device(p.dt_bias, "f32")
    state = Guarded((batch, d_inner, N), torch.float32,
                    init=torch.from_numpy(p.state0).cuda())
    msc.tuning_set("update_path", path)
    try:
        prev = None
        for k in range(2):
            s = synth.decode_step(batch, d_inner, N, k, seed=2200 + d_inner, dtype="bf16")
            dv = {n: to_device(getattr(s, f), "bf16") for n, f in
                  (("u", "u"), ("dt", "dt_raw"), ("B", "B"), ("C", "C"), ("z", "z"))}
            out = Guarded((batch, d_inner), torch.bfloat16)
            if variant == "trapezoid":
                lam = to_device(np.full((batch, d_inner), 0.25, np.float32), "bf16")
                msc.selective_state_update_trap(
                    state.t, None if prev is None else prev[0], None if prev is None else prev[1],
                    dv["u"], dv["dt"], lam, A, dv["B"], dv["C"], D, dv["z"], bias, out=out.t)
            else:
                msc.selective_state_update(state.t, dv["u"], dv["dt"], A, dv["B"], dv["C"], D,
                                           dv["z"], bias, out=out.t, zoh=variant == "zoh")
            out.check(f"out, token {k}")
            state.check(f"state, token {k}")
            prev = (dv["u"], dv["B"])
    finally:
        msc.tuning_set("update_path", 0)
    msc.check_device_error()


@pytest.mark.parametrize("batch,L,d_inner,dtype", [
    (2, 77, 40, "bf16"), (3, 33, 33, "f32"), (1, 5, 1000, "bf16"), (9, 64, 96, "bf16")])
def test_conv_writes_stay_inside(batch, L, d_inner, dtype):
    """Conv prefill (output and final window) and the decode-token update
    (window in place, output)."""
    rng = np.random.default_rng(2300 + L)
    sdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    x = to_device(synth.round_bf16(rng.standard_normal((batch, L, d_inner)).astype(np.float32)),
                  dtype)
    w = torch.randn(d_inner, 4, device="cuda") / 2
    b = torch.randn(d_inner, device="cuda") / 10
    s_in = torch.randn(batch, d_inner, 3, device="cuda").to(sdt)
    out = Guarded((batch, L, d_inner), sdt)
    s_out = Guarded((batch, d_inner, 3), sdt)
    msc.causal_conv1d_fwd(x, w, b, state_in=s_in, out=out.t, state_out=s_out.t)
    out.check("conv out")
    s_out.check("conv state_out")
    win = Guarded((batch, d_inner, 3), sdt, init=s_in)
    tok = Guarded((batch, d_inner), sdt)
    msc.causal_conv1d_update(win.t, x[:, 0].contiguous(), w, b, out=tok.t)
    tok.check("conv update out")
    win.check("conv update window")
    msc.check_device_error()
