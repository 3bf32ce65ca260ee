"""conv2d_fwd on the GPU vs the fp64 oracle, element by element.

Tolerance: |y_gpu - y_ref| <= 1e-5 * (sum |x * w| + |b|) per element (the
fp32 bound of the direct-convolution path).  Covers the five workloads at
full size (layer by layer for the 3-layer net, each layer fed the GPU's own
input), ragged tiles, every supported filter size, both layouts, and edge
cases (images smaller than the filter, one pixel, N > 1, no bias).
"""
import numpy as np
import pytest
import torch

import synthetic as S
import stencil_conv2d_fwd_gb300 as sc
from parity_util import assert_conv_close, conv_gpu, nchw_to_nhwc, nhwc_to_nchw

pytestmark = pytest.mark.gpu


def _one(oracle_mod, dev, x, L, layout=sc.SC_NHWC, rows=None):
    y = conv_gpu(x, L.w, L.b, L.act, dev, layout=layout)
    yr, a = oracle_mod.conv2d_nchw(x, L.w, L.b, L.act)
    return y, yr, a


@pytest.mark.parametrize("cid", [1, 2, 4])
def test_workload_full_size(oracle_mod, cuda_dev, sc, cid):
    c = S.config(cid)
    L = c.layers[0]
    y, yr, a = _one(oracle_mod, cuda_dev, c.x, L)
    assert_conv_close(y, yr, a, what=f"workload {cid}")


def test_upscaling_net_layer_by_layer_and_end_to_end(oracle_mod, cuda_dev, sc):
    """Each layer is checked against the oracle fed the GPU's own input to it;
    the final output is also checked against the all-fp64 chain with the
    propagated bound E_L = 1e-5 A_L + conv(|w_L|, E_{L-1} + u |y_{L-1}|)."""
    c = S.config(3)
    x = c.x
    x64 = c.x.astype(np.float64)
    E = np.zeros_like(x64)
    u = 2.0 ** -24
    for li, L in enumerate(c.layers):
        y = conv_gpu(x, L.w, L.b, L.act, cuda_dev)
        yr, a = oracle_mod.conv2d_nchw(x, L.w, L.b, L.act)
        assert_conv_close(y, yr, a, what=f"layer {li + 1}")
        # all-fp64 chain: the oracle takes fp32 inputs, so the chain's own
        # rounding to fp32 between layers enters the bound as u*|y|
        y64, a64 = oracle_mod.conv2d_nchw(x64.astype(np.float32), L.w, L.b, L.act)
        Ein = E + u * np.abs(x64) + np.abs(x64 - x64.astype(np.float32).astype(np.float64))
        prop = torch.nn.functional.conv2d(torch.from_numpy(Ein), torch.from_numpy(np.abs(L.w).astype(np.float64)),
                                          padding=(L.r // 2, L.s // 2)).numpy()
        E = 1e-5 * a + prop   # a: scale of this layer at the GPU's own input
        x, x64 = y, y64
    err = np.abs(x.astype(np.float64) - x64)
    assert (err <= E).all(), f"end-to-end error {err.max()} exceeds the propagated bound"


def test_upscaling_net_with_split_tf32_layers_end_to_end(oracle_mod, cuda_dev, sc):
    """The net with its 32 -> 32 and 32 -> 4 layers on conv2d_fwd_tc_x3 (layer
    1 on conv2d_fwd): each layer within 1e-5 * A of the oracle fed the GPU's
    own input, and the final output within the bound propagated through the
    all-fp64 chain, as for the FFMA net above."""
    c = S.config(3)
    x = c.x
    x64 = c.x.astype(np.float64)
    E = np.zeros_like(x64)
    u = 2.0 ** -24
    for li, L in enumerate(c.layers):
        if li >= 1:
            N, Cin, H, W = x.shape
            xd = torch.from_numpy(nchw_to_nhwc(x)).to(cuda_dev)
            wd, bd = torch.from_numpy(L.w).to(cuda_dev), torch.from_numpy(L.b).to(cuda_dev)
            yd = torch.empty(N * H * W * L.cout, device=cuda_dev)
            sc.check(sc.conv2d_fwd_tc_x3(xd, wd, bd, yd, N, H, W, Cin, L.cout, L.r, L.s, L.act), "conv2d_fwd_tc_x3")
            torch.cuda.synchronize()
            y = nhwc_to_nchw(yd.cpu().numpy().reshape(N, H, W, L.cout))
        else:
            y = conv_gpu(x, L.w, L.b, L.act, cuda_dev)
        yr, a = oracle_mod.conv2d_nchw(x, L.w, L.b, L.act)
        assert_conv_close(y, yr, a, what=f"layer {li + 1}")
        y64, a64 = oracle_mod.conv2d_nchw(x64.astype(np.float32), L.w, L.b, L.act)
        Ein = E + u * np.abs(x64) + np.abs(x64 - x64.astype(np.float32).astype(np.float64))
        prop = torch.nn.functional.conv2d(torch.from_numpy(Ein), torch.from_numpy(np.abs(L.w).astype(np.float64)),
                                          padding=(L.r // 2, L.s // 2)).numpy()
        E = 1e-5 * a + prop
        x, x64 = y, y64
    err = np.abs(x.astype(np.float64) - x64)
    assert (err <= E).all(), f"end-to-end error {err.max()} exceeds the propagated bound"


SHAPES = [
    # (N, Cin, Cout, H, W, R, S)
    (1, 4, 4, 1, 1, 3, 3),
    (1, 4, 4, 2, 3, 5, 5),
    (2, 8, 8, 9, 13, 3, 3),
    (1, 12, 20, 17, 70, 3, 3),
    (3, 16, 16, 33, 65, 3, 3),
    (2, 32, 12, 10, 101, 3, 3),   # 9-16 channels on a small image: 48-pixel tiles
    (1, 32, 32, 19, 131, 3, 3),
    (1, 32, 4, 11, 300, 3, 3),
    (2, 64, 64, 15, 57, 3, 3),
    (1, 36, 68, 10, 40, 3, 3),
    (1, 64, 128, 9, 33, 3, 3),
    (1, 68, 48, 7, 29, 3, 3),
    (1, 20, 12, 21, 22, 1, 1),
    (1, 16, 32, 13, 70, 5, 5),
    (1, 8, 16, 12, 40, 7, 7),
    (1, 8, 8, 12, 17, 3, 5),
    (1, 8, 8, 12, 17, 7, 1),
    # TMA-staged 5x5 and 1x1: wide, narrow with Cin % 8 != 0, 16-channel
    # groups, a filter bank above the TMA kernel's limit (cp.async fallback)
    (1, 32, 32, 21, 90, 5, 5),
    (2, 12, 4, 9, 170, 5, 5),
    (1, 16, 16, 7, 33, 5, 5),
    (1, 64, 40, 8, 30, 5, 5),
    (1, 32, 64, 9, 50, 1, 1),
    (2, 8, 4, 5, 7, 1, 1),
    (2, 4, 36, 5, 9, 5, 3),
    # 32 -> 4 with enough 8 x 160 tiles for the narrow-output kernel: ragged
    # tiles at the right and bottom edges, several images, a 1 x 3 filter
    (12, 32, 4, 75, 330, 3, 3),
    (8, 32, 4, 77, 490, 1, 3),
    # small images, at most 16 channels in and out (whole-tile kernel):
    # ragged 4 x 32 tiles, several images, fewer channels than 16, 1 x 3 and
    # 3 x 1 filters, and the largest image it takes (64 K pixels)
    (4, 12, 8, 30, 50, 3, 3),
    (1, 16, 12, 7, 97, 1, 3),
    (1, 4, 16, 5, 33, 3, 1),
    (2, 16, 4, 100, 40, 3, 3),
    (1, 16, 16, 256, 256, 3, 3),
    (1, 16, 16, 257, 256, 3, 3),
]


@pytest.mark.parametrize("shape", SHAPES, ids=[str(s) for s in SHAPES])
@pytest.mark.parametrize("act", [0, 1])
def test_general_shapes(oracle_mod, cuda_dev, sc, shape, act):
    N, Cin, Cout, H, W, R, S_ = shape
    c = S.conv_case(100 + Cin + Cout + H, N, Cin, Cout, H, W, R, S_, act=act)
    L = c.layers[0]
    y, yr, a = _one(oracle_mod, cuda_dev, c.x, L)
    assert_conv_close(y, yr, a, what=str(shape))


C1_SHAPES = [
    (1, 1, 1, 1, 3, 3), (1, 1, 2, 3, 5, 5), (1, 1, 64, 64, 3, 3), (2, 1, 37, 45, 3, 3),
    (1, 4, 20, 33, 5, 5), (1, 8, 31, 130, 5, 5), (1, 12, 9, 17, 3, 3), (1, 16, 40, 70, 7, 7),
    (1, 24, 16, 100, 5, 5), (1, 32, 50, 260, 5, 5), (2, 32, 23, 41, 3, 3), (1, 64, 12, 66, 5, 5),
    (1, 32, 10, 35, 1, 1), (1, 8, 15, 21, 3, 7), (1, 1, 64, 1030, 7, 7), (1, 32, 6, 1300, 5, 5),
    # W % 4 == 0 (the register-ring kernel): every filter size, bands that are
    # not a multiple of K rows, a 2-pixel-wide strip per lane group
    (1, 32, 17, 96, 7, 7), (1, 8, 9, 44, 1, 1), (2, 16, 13, 52, 3, 3), (1, 4, 7, 8, 3, 5), (1, 1, 23, 36, 5, 5),
    # more than 16 channels, W % 4 == 0 (two output rows per pass): odd band
    # ends, channel groups past Cout, 3x3 and 5x5
    (1, 32, 13, 44, 3, 3), (2, 24, 9, 40, 5, 5), (1, 32, 7, 8, 5, 5), (1, 64, 11, 36, 3, 3),
    # the tiled kernel (17-32 channels per group, W % 4 == 0): a tile past the
    # image's right edge, channel groups past Cout, every filter size incl.
    # 7 x 7 and non-square, one-row images, N > 1
    (2, 32, 37, 300, 5, 5), (1, 40, 9, 516, 7, 7), (1, 32, 1, 4, 3, 3), (1, 36, 13, 260, 1, 1),
    (1, 32, 11, 128, 3, 5), (3, 48, 5, 68, 5, 5),
]


@pytest.mark.parametrize("shape", C1_SHAPES, ids=[str(s) for s in C1_SHAPES])
def test_single_input_channel_shapes(oracle_mod, cuda_dev, sc, shape):
    N, Cout, H, W, R, S_ = shape
    c = S.conv_case(200 + Cout + H + W, N, 1, Cout, H, W, R, S_, act=1)
    L = c.layers[0]
    y, yr, a = _one(oracle_mod, cuda_dev, c.x, L)
    assert_conv_close(y, yr, a, what=str(shape))


@pytest.mark.parametrize("shape", [(2, 8, 12, 9, 20, 3, 3), (1, 1, 16, 13, 37, 5, 5), (1, 16, 4, 17, 9, 3, 3),
                                   (1, 1, 1, 10, 11, 3, 3), (2, 1, 32, 9, 68, 5, 5)])
def test_nchw_layout(oracle_mod, cuda_dev, sc, shape):
    N, Cin, Cout, H, W, R, S_ = shape
    c = S.conv_case(300 + Cin + Cout, N, Cin, Cout, H, W, R, S_, act=1)
    L = c.layers[0]
    y, yr, a = _one(oracle_mod, cuda_dev, c.x, L, layout=sc.SC_NCHW)
    assert_conv_close(y, yr, a, what="nchw " + str(shape))


def test_no_bias(oracle_mod, cuda_dev, sc):
    c = S.conv_case(400, 1, 16, 16, 20, 30, 3, 3, act=0)
    L = c.layers[0]
    y = conv_gpu(c.x, L.w, None, 0, cuda_dev)
    yr, a = oracle_mod.conv2d_nchw(c.x, L.w, None, 0)
    assert_conv_close(y, yr, a, what="no bias")


def test_delta_filter_is_exact(cuda_dev, sc):
    """A centre delta filter returns x + b exactly (one nonzero product)."""
    c = S.conv_case(401, 1, 8, 8, 17, 23, 3, 3, act=0)
    w = np.zeros((8, 8, 3, 3), np.float32)
    for i in range(8):
        w[i, i, 1, 1] = 1.0
    b = np.linspace(-1, 1, 8).astype(np.float32)
    y = conv_gpu(c.x, w, b, 0, cuda_dev)
    np.testing.assert_array_equal(y, c.x + b[None, :, None, None])


def test_side_stream(oracle_mod, cuda_dev, sc):
    c = S.conv_case(402, 1, 8, 8, 16, 16, 3, 3, act=1)
    L = c.layers[0]
    s = torch.cuda.Stream()
    y = conv_gpu(c.x, L.w, L.b, 1, cuda_dev, stream=s)
    yr, a = oracle_mod.conv2d_nchw(c.x, L.w, L.b, 1)
    assert_conv_close(y, yr, a, what="side stream")


def test_misaligned_pointer_rejected_without_launch(cuda_dev, sc):
    x = torch.zeros(4 * 8 * 8 + 1, device=cuda_dev)
    w = torch.zeros(4 * 4 * 9, device=cuda_dev)
    y = torch.full((4 * 8 * 8,), 3.0, device=cuda_dev)
    rc = sc.conv2d_fwd(x.data_ptr() + 4, w, None, y, 1, 8, 8, 4, 4, 3, 3, sc.SC_NHWC, 0)
    assert rc == sc.SC_ERR_ALIGN
    torch.cuda.synchronize()
    assert (y == 3.0).all()


@pytest.mark.parametrize("Cout", [4, 32])
def test_tma_kernel_bounded_wait_expiry(oracle_mod, cuda_dev, sc, Cout):
    """Failure detection without a fault: copy 1 of every CTA of the
    TMA-staged convolution is never issued; the waits for it expire (2 ms),
    the kernel records SC_ERR_DEVICE_TIMEOUT and returns; the next call on
    the same context is correct."""
    from parity_util import nchw_to_nhwc
    N, Cin, H, W = 1, 32, 24, 200
    c = S.conv_case(990 + Cout, N, Cin, Cout, H, W, 3, 3, act=0)
    L = c.layers[0]
    xd = torch.from_numpy(nchw_to_nhwc(c.x)).to(cuda_dev)
    wd = torch.from_numpy(np.ascontiguousarray(L.w)).to(cuda_dev)
    bd = torch.from_numpy(L.b).to(cuda_dev)
    yd = torch.empty(N * H * W * Cout, device=cuda_dev)
    assert sc.sc_last_device_status() == sc.SC_OK
    rc = sc.sc_test_conv_wait_expiry(xd, wd, bd, yd, N, H, W, Cin, Cout, 1, 2000)
    assert rc == sc.SC_OK, sc.sc_status_string(rc)
    assert sc.sc_last_device_status() == sc.SC_ERR_DEVICE_TIMEOUT
    assert sc.sc_last_device_status() == sc.SC_OK          # read clears it
    y, yr, a = _one(oracle_mod, cuda_dev, c.x, L)           # context still usable
    assert_conv_close(y, yr, a, what=f"after the expiry test, Cout={Cout}")
