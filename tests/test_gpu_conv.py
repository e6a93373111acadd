"""GPU parity of the causal depthwise conv1d (+ SiLU) before the scan and of
its decode update against the fp64 oracle ("Deep dive into Mamba" sections
3.2 and 5.2; the MambaBlock of "State space models and Mamba").  Outputs:
rel-L2 <= 1e-5 for fp32 storage, <= 2e-3 for bf16 storage against the
oracle rounded to bf16; conv states hold input values and must match bit
for bit."""
import numpy as np
import pytest

import oracle
import selective_state_space_144_b300 as msc
from selective_state_space_144_b300 import synth
from tests.helpers import TOL, as_stored, from_device, rel_l2, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def conv_case(batch, L, d_inner, d_conv, dtype, seed, with_state=False):
    """x in storage precision (u-like N(0,1)), w ~ N(0, 1/d_conv), bias ~ N(0, 0.1)."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((batch, L, d_inner)).astype(np.float32)
    st = rng.standard_normal((batch, d_inner, d_conv - 1)).astype(np.float32)
    if dtype == "bf16":
        x, st = synth.round_bf16(x), synth.round_bf16(st)
    w = (rng.standard_normal((d_inner, d_conv)) / np.sqrt(d_conv)).astype(np.float32)
    bias = (0.1 * rng.standard_normal(d_inner)).astype(np.float32)
    return x, w, bias, (st if with_state else None)


def run_conv(x, w, bias, st, dtype, silu=True, offset=0):
    xd = to_device(x, dtype)
    if offset:   # shift x by one element: misaligned for 8-byte vectors
        buf = torch.empty(x.size + offset, dtype=xd.dtype, device="cuda")
        xd = buf[offset:].view(x.shape).copy_(xd)
    std = None if st is None else to_device(st, dtype)
    out, st_out = msc.causal_conv1d_fwd(xd, to_device(w, "f32"),
                                        None if bias is None else to_device(bias, "f32"),
                                        state_in=std, silu=silu)
    torch.cuda.synchronize()
    return from_device(out), from_device(st_out)


def check(x, w, bias, st, dtype, silu=True, offset=0):
    y, st_out = run_conv(x, w, bias, st, dtype, silu, offset)
    y_ref, st_ref = oracle.causal_conv1d(x, w, bias, state_in=st, silu=silu)
    assert np.all(np.isfinite(y))
    if y.size:
        assert rel_l2(y, as_stored(y_ref, dtype)) <= TOL[dtype]
    assert np.array_equal(st_out, st_ref.astype(np.float32))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d_conv", [1, 2, 3, 4, 5, 8])
@pytest.mark.parametrize("d_inner", [45, 1024])
def test_conv_shapes(dtype, d_conv, d_inner):
    x, w, bias, st = conv_case(2, 150, d_inner, d_conv, dtype, seed=d_conv * 7 + d_inner)
    check(x, w, bias, None, dtype)
    check(x, w, bias, st if st is not None else
          conv_case(2, 1, d_inner, d_conv, dtype, 1, with_state=True)[3], dtype)


@pytest.mark.parametrize("L", [0, 1, 2, 3, 4, 31, 32, 33, 63, 64, 65, 129])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_conv_lengths(L, dtype):
    """Sequences shorter than the window, exactly one tile, ragged tiles; the
    conv state then mixes state_in and x."""
    x, w, bias, st = conv_case(3, L, 64, 4, dtype, seed=100 + L, with_state=True)
    check(x, w, bias, st, dtype)
    check(x, w, bias, None, dtype)


@pytest.mark.parametrize("silu", [False, True])
@pytest.mark.parametrize("with_bias", [False, True])
def test_conv_options(silu, with_bias):
    x, w, bias, _ = conv_case(2, 90, 128, 4, "f32", seed=5)
    check(x, w, bias if with_bias else None, None, "f32", silu=silu)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_conv_misaligned_input(dtype):
    """x one element off an 8-byte boundary: element-wise path, same result."""
    x, w, bias, st = conv_case(2, 70, 128, 4, dtype, seed=6, with_state=True)
    check(x, w, bias, st, dtype, offset=1)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_conv_split_prefill(dtype):
    """Prefill in pieces, each continuing from the previous piece's conv
    state, equals one prefill."""
    x, w, bias, _ = conv_case(2, 300, 256, 4, dtype, seed=7)
    y0, s0 = run_conv(x, w, bias, None, dtype)
    ys, st = [], None
    for lo, hi in ((0, 1), (1, 130), (130, 300)):
        y, st = run_conv(x[:, lo:hi], w, bias, st, dtype)
        ys.append(y)
    assert np.array_equal(np.concatenate(ys, axis=1), y0)
    assert np.array_equal(st, s0)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d_conv", [1, 2, 4, 6])
@pytest.mark.parametrize("batch,d_inner", [(3, 96), (13, 300), (16, 64)])
def test_conv_update(dtype, d_conv, batch, d_inner):
    """Decode tokens against the oracle, and decode == prefill (batch 3: a
    thread per (row, channel); 13 and 16: 8 batch rows per thread, the last
    group partial for 13, a ragged channel block for 300)."""
    L = 9
    x, w, bias, st = conv_case(batch, L, d_inner, d_conv, dtype, seed=200 + d_conv,
                               with_state=True)
    y_pre, st_pre = run_conv(x, w, bias, st, dtype)
    state = to_device(st, dtype)
    wd, bd = to_device(w, "f32"), to_device(bias, "f32")
    ref_st = st.astype(np.float64)
    outs = []
    for t in range(L):
        o = msc.causal_conv1d_update(state, to_device(x[:, t].copy(), dtype), wd, bd)
        ref_st, ref_o = oracle.conv1d_update(ref_st, x[:, t], w, bias)
        outs.append(from_device(o))
        assert rel_l2(outs[-1], as_stored(ref_o, dtype)) <= TOL[dtype], t
    torch.cuda.synchronize()
    assert np.array_equal(from_device(state), ref_st.astype(np.float32))
    assert np.array_equal(np.stack(outs, axis=1), y_pre)
    assert np.array_equal(from_device(state), st_pre)


def test_conv_layer_size():
    """The 8 x 2048 x 1536 layer with d_conv 4 in bf16, every element."""
    x, w, bias, _ = conv_case(8, 2048, 1536, 4, "bf16", seed=11)
    check(x, w, bias, None, "bf16")
