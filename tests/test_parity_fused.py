"""conv2d_fwd_tc_fused2 (two 3x3 layers on the tensor cores, the 32-channel
intermediate kept on chip) vs the fp64 oracle run layer by layer.  Bound per
element of y: layer 2's own TF32 error, 5e-3 * A3 (A3 = sum |t * w2| + |b2|
from the oracle), plus layer 1's error (at most 5e-3 * A2 per element of t;
ReLU is 1-Lipschitz) carried through |w2|: conv(5e-3 * A2, |w2|), computed by
the oracle with a bias-free, activation-free convolution."""
import numpy as np
import pytest
import torch

import synthetic as S
from parity_util import assert_conv_close, nchw_to_nhwc, nhwc_to_nchw

pytestmark = pytest.mark.gpu
TC_RTOL = 5e-3


def fused_gpu(x, w1, b1, w2, b2, act1, act2, dev, sc):
    N, C0, H, W = x.shape
    C1, C2 = w1.shape[0], w2.shape[0]
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    xd, w1d, b1d, w2d, b2d = t(nchw_to_nhwc(x)), t(w1), t(b1), t(w2), t(b2)
    n = N * H * W * C2
    buf = torch.full((n + 8192,), -7.75e30, device=dev)
    yd = buf[4096:4096 + n]
    sc.check(sc.conv2d_fwd_tc_fused2(xd, w1d, b1d, w2d, b2d, yd, N, H, W, C0, C1, C2, act1, act2),
             "conv2d_fwd_tc_fused2")
    st = sc.sc_last_device_status()
    assert st == sc.SC_OK, sc.sc_status_string(st)
    torch.cuda.synchronize()
    h = buf.cpu().numpy()
    assert (h[:4096] == -7.75e30).all() and (h[4096 + n:] == -7.75e30).all(), "write outside the output buffer"
    return nhwc_to_nchw(h[4096:4096 + n].reshape(N, H, W, C2))


def fused_bound(oracle_mod, x, w1, b1, w2, b2, act1, act2):
    t_ref, a2 = oracle_mod.conv2d_nchw(x, w1, b1, act1)
    y_ref, a3 = oracle_mod.conv2d_nchw(t_ref.astype(np.float32), w2, b2, act2)
    carried, _ = oracle_mod.conv2d_nchw((TC_RTOL * a2).astype(np.float32), np.abs(w2), None, 0)
    return y_ref, a3 + 1.01 * carried / TC_RTOL


SHAPES = [
    # (N, C0, C2, H, W, act1, act2)
    (1, 32, 4, 13, 61, 1, 0),
    (2, 16, 8, 7, 30, 1, 1),
    (1, 8, 4, 20, 57, 0, 0),
    (1, 32, 8, 1, 1, 1, 0),
    (1, 32, 4, 3, 2, 1, 0),
    (1, 32, 4, 40, 200, 1, 0),
]


@pytest.mark.parametrize("shape", SHAPES, ids=[str(s) for s in SHAPES])
def test_fused_shapes(oracle_mod, cuda_dev, sc, shape):
    N, C0, C2, H, W, act1, act2 = shape
    c1 = S.conv_case(1100 + C0 + W, N, C0, 32, H, W, 3, 3, act=act1)
    c2 = S.conv_case(1200 + C2 + W, N, 32, C2, H, W, 3, 3, act=act2)
    x, L1, L2 = c1.x, c1.layers[0], c2.layers[0]
    y = fused_gpu(x, L1.w, L1.b, L2.w, L2.b, act1, act2, cuda_dev, sc)
    y_ref, scale = fused_bound(oracle_mod, x, L1.w, L1.b, L2.w, L2.b, act1, act2)
    assert_conv_close(y, y_ref, scale, rtol=TC_RTOL, what=f"fused {shape}")


def test_fused_layers_2_and_3_of_the_net_full_size(oracle_mod, cuda_dev, sc):
    wl = S.config(3)
    L2, L3 = wl.layers[1], wl.layers[2]
    x = np.maximum(S.uniform(77, 0, (wl.n, L2.cin, wl.h, wl.w), -1, 1), 0).astype(np.float32)
    y = fused_gpu(x, L2.w, L2.b, L3.w, L3.b, L2.act, L3.act, cuda_dev, sc)
    y_ref, scale = fused_bound(oracle_mod, x, L2.w, L2.b, L3.w, L3.b, L2.act, L3.act)
    worst = assert_conv_close(y, y_ref, scale, rtol=TC_RTOL, what="fused 3-L2 + 3-L3")
    assert worst < 1.0


def test_fused_rejects_what_it_does_not_run(cuda_dev, sc):
    x = torch.zeros(8 * 8 * 32, device=cuda_dev)
    w1 = torch.zeros(32 * 32 * 9, device=cuda_dev)
    w2 = torch.zeros(16 * 32 * 9, device=cuda_dev)
    y = torch.zeros(8 * 8 * 16, device=cuda_dev)
    f = sc.conv2d_fwd_tc_fused2
    assert f(x, w1, None, w2, None, y, 1, 8, 8, 32, 16, 4, 1, 0) == sc.SC_ERR_UNSUPPORTED   # C1 != 32
    assert f(x, w1, None, w2, None, y, 1, 8, 8, 32, 32, 16, 1, 0) == sc.SC_ERR_UNSUPPORTED  # C2 > 8
    assert f(x, w1, None, w2, None, y, 1, 8, 8, 6, 32, 4, 1, 0) == sc.SC_ERR_UNSUPPORTED    # C0 % 4
    assert f(x[1:], w1, None, w2, None, y, 1, 8, 8, 32, 32, 4, 1, 0) == sc.SC_ERR_ALIGN
    torch.cuda.synchronize()
    assert sc.sc_last_device_status() == sc.SC_OK
