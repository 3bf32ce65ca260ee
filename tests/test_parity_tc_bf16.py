"""conv2d_fwd_tc_bf16 (tcgen05 kind::f16: bf16 activations in and out, bf16
operands, fp32 accumulation) vs the fp64 oracle on the same bf16-exact
inputs.  Tolerance |y - y_ref| <= 5e-3 * (sum |x * w| + |b|) for the
computation (the filters are rounded to bf16 inside: at most 2^-8 relative
per product, bf16's unit roundoff), plus, for a bf16 output, its own storage
rounding of at most 2^-8 * |y_ref|."""
import numpy as np
import pytest
import torch

import synthetic as S
import stencil_conv2d_fwd_gb300 as sc
from bf16_util import bf16_bits_to_f32, round_to_bf16, to_bf16_bits
from parity_util import assert_conv_close, nchw_to_nhwc, nhwc_to_nchw

pytestmark = pytest.mark.gpu
BF16_RTOL = 5e-3
CANARY = 4096
CANARY_BITS = 0x7BAD


def tol_scale(y_ref, a, y_dtype):
    """The per-element bound divided by BF16_RTOL: A, plus the bf16 storage
    rounding of the result when y is bf16."""
    if y_dtype == sc.SC_BF16:
        return a + (2.0 ** -8 / BF16_RTOL) * np.abs(y_ref)
    return a


def conv_bf16(x_nchw, w, b, act, y_dtype, dev):
    """x_nchw must hold bf16-exact values; returns y as NCHW float32."""
    N, Cin, H, W = x_nchw.shape
    Cout, _, R, S_ = w.shape
    xb = to_bf16_bits(nchw_to_nhwc(x_nchw))
    assert (bf16_bits_to_f32(xb).reshape(xb.shape) == nchw_to_nhwc(x_nchw)).all()
    xd = torch.from_numpy(xb.view(np.int16)).to(dev)
    wd = torch.from_numpy(np.ascontiguousarray(w)).to(dev)
    bd = None if b is None else torch.from_numpy(b).to(dev)
    n = N * H * W * Cout
    if y_dtype == sc.SC_BF16:
        buf = torch.full((n + 2 * CANARY,), CANARY_BITS, dtype=torch.int16, device=dev)
    else:
        buf = torch.full((n + 2 * CANARY,), -7.75e30, dtype=torch.float32, device=dev)
    yd = buf[CANARY:CANARY + n]
    sc.check(sc.conv2d_fwd_tc_bf16(xd, wd, bd, yd, N, H, W, Cin, Cout, R, S_, act, y_dtype), "conv2d_fwd_tc_bf16")
    st = sc.sc_last_device_status()
    assert st == sc.SC_OK, sc.sc_status_string(st)
    torch.cuda.synchronize()
    h = buf.cpu().numpy()
    assert (h[:CANARY] == h[0]).all() and (h[CANARY + n:] == h[0]).all(), "write outside the output buffer"
    y = h[CANARY:CANARY + n]
    if y_dtype == sc.SC_BF16:
        y = bf16_bits_to_f32(y.view(np.uint16))
    return nhwc_to_nchw(np.asarray(y, dtype=np.float32).reshape(N, H, W, Cout))


SHAPES = [
    # (N, Cin, Cout, H, W, R, S)
    (1, 8, 16, 9, 13, 3, 3),
    (1, 8, 4, 1, 1, 3, 3),
    (2, 16, 32, 33, 70, 3, 3),
    (1, 24, 12, 17, 130, 3, 3),
    (1, 64, 128, 10, 40, 3, 3),
    (1, 32, 4, 20, 300, 3, 3),
    (1, 16, 48, 11, 257, 3, 3),
    (1, 8, 16, 12, 17, 1, 1),
    (1, 8, 12, 12, 17, 3, 1),
    (1, 128, 32, 9, 40, 3, 3),
    (1, 256, 8, 6, 33, 3, 3),
]


@pytest.mark.parametrize("y_dtype", [1, 0], ids=["y_bf16", "y_f32"])
@pytest.mark.parametrize("shape", SHAPES, ids=[str(s) for s in SHAPES])
def test_bf16_shapes(oracle_mod, cuda_dev, sc, shape, y_dtype):
    N, Cin, Cout, H, W, R, S_ = shape
    c = S.conv_case(700 + Cin + Cout + W, N, Cin, Cout, H, W, R, S_, act=1)
    L = c.layers[0]
    x = round_to_bf16(c.x)
    y = conv_bf16(x, L.w, L.b, L.act, y_dtype, cuda_dev)
    yr, a = oracle_mod.conv2d_nchw(x, L.w, L.b, L.act)
    assert_conv_close(y, yr, tol_scale(yr, a, y_dtype), rtol=BF16_RTOL, what=f"bf16 {shape} y_dtype={y_dtype}")


@pytest.mark.parametrize("y_dtype", [1, 0], ids=["y_bf16", "y_f32"])
@pytest.mark.parametrize("cid,li", [(4, 0), (3, 1), (3, 2)])
def test_bf16_workloads_full_size(oracle_mod, cuda_dev, sc, cid, li, y_dtype):
    """Full workload sizes.  With y_f32 the bound is the plain 5e-3 * A of the
    tensor-core variants (no storage term): the computation alone."""
    wl = S.config(cid)
    L = wl.layers[li]
    x = wl.x if li == 0 else np.maximum(S.uniform(77, 0, (wl.n, L.cin, wl.h, wl.w), -1, 1), 0).astype(np.float32)
    x = round_to_bf16(x)
    y = conv_bf16(x, L.w, L.b, L.act, y_dtype, cuda_dev)
    yr, a = oracle_mod.conv2d_nchw(x, L.w, L.b, L.act)
    worst = assert_conv_close(y, yr, tol_scale(yr, a, y_dtype), rtol=BF16_RTOL,
                              what=f"bf16 workload {cid} layer {li} y_dtype={y_dtype}")
    assert worst < 1.0


def test_bf16_rejects_what_it_does_not_run(cuda_dev, sc):
    x = torch.zeros(8 * 8 * 32, dtype=torch.int16, device=cuda_dev)
    w = torch.zeros(32 * 32 * 9, device=cuda_dev)
    y = torch.zeros(8 * 8 * 32, device=cuda_dev)
    # bf16 pixel rows must be a multiple of 16 bytes: Cin % 8
    assert sc.conv2d_fwd_tc_bf16(x, w, None, y, 1, 8, 8, 4, 4, 3, 3, 0, sc.SC_F32) == sc.SC_ERR_UNSUPPORTED
    # bf16 output rows through the TMA store: Cout % 8 once Cout > 16
    assert sc.conv2d_fwd_tc_bf16(x, w, None, y, 1, 8, 8, 8, 20, 3, 3, 0, sc.SC_BF16) == sc.SC_ERR_UNSUPPORTED
    assert sc.conv2d_fwd_tc_bf16(x, w, None, y, 1, 8, 8, 8, 20, 3, 3, 0, 7) == sc.SC_ERR_UNSUPPORTED
    assert sc.conv2d_fwd_tc_bf16(x, w, None, y, 1, 8, 8, 8, 8, 5, 5, 0, sc.SC_F32) == sc.SC_ERR_UNSUPPORTED
    assert sc.conv2d_fwd_tc_bf16(x[1:], w, None, y, 1, 8, 8, 8, 8, 3, 3, 0, sc.SC_F32) == sc.SC_ERR_ALIGN
    torch.cuda.synchronize()
    assert sc.sc_last_device_status() == sc.SC_OK
