"""Seeded random shapes against the fp64 oracle, element by element, for the
paths whose tiling has the most edges: the tiled single-channel kernel
(20-64 output channels, W % 4 == 0, every filter size up to 7 x 7,
non-square filters, bands that end mid-tile) and the split-TF32 tensor-core
variant (channel groups of 4-32, 1 x 1 to 3 x 3 filters, ragged tiles), the
latter at the fp32 bound 1e-5 * A like conv2d_fwd itself.  The shapes come
from a fixed generator, so a failure names a reproducible case."""
import numpy as np
import pytest
import torch

import synthetic as S
import stencil_conv2d_fwd_gb300 as sc
from parity_util import assert_conv_close, conv_gpu, nchw_to_nhwc, nhwc_to_nchw

pytestmark = pytest.mark.gpu


def _c1_shapes(n=16, seed=2026):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        K = int(rng.choice([1, 3, 5, 7]))
        R = K
        S_ = int(rng.choice([k for k in (1, 3, 5, 7) if k <= K])) if rng.random() < 0.3 else K
        out.append((int(rng.integers(1, 3)), 4 * int(rng.integers(5, 17)), int(rng.integers(1, 40)),
                    4 * int(rng.integers(1, 130)), R, S_))
    return out


def _x3_shapes(n=16, seed=2027):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        R, S_ = (int(rng.choice([1, 3])), int(rng.choice([1, 3])))
        out.append((int(rng.integers(1, 3)), 4 * int(rng.integers(1, 17)), 4 * int(rng.integers(1, 17)),
                    int(rng.integers(1, 30)), int(rng.integers(1, 200)), R, S_))
    return out


C1 = _c1_shapes()
X3 = _x3_shapes()


@pytest.mark.parametrize("shape", C1, ids=[str(s) for s in C1])
def test_single_channel_sweep(oracle_mod, cuda_dev, sc, shape):
    N, Cout, H, W, R, S_ = shape
    c = S.conv_case(400 + Cout + H + W, N, 1, Cout, H, W, R, S_, act=int((H + W) % 2))
    L = c.layers[0]
    y = conv_gpu(c.x, L.w, L.b, L.act, cuda_dev)
    yr, a = oracle_mod.conv2d_nchw(c.x, L.w, L.b, L.act)
    assert_conv_close(y, yr, a, what=str(shape))


@pytest.mark.parametrize("shape", X3, ids=[str(s) for s in X3])
def test_split_tf32_sweep(oracle_mod, cuda_dev, sc, shape):
    N, Cin, Cout, H, W, R, S_ = shape
    c = S.conv_case(500 + Cin + Cout + W, N, Cin, Cout, H, W, R, S_, act=int(W % 2))
    L = c.layers[0]
    xd = torch.from_numpy(nchw_to_nhwc(c.x)).to(cuda_dev)
    wd, bd = torch.from_numpy(L.w).to(cuda_dev), torch.from_numpy(L.b).to(cuda_dev)
    yd = torch.empty(N * H * W * Cout, device=cuda_dev)
    sc.check(sc.conv2d_fwd_tc_x3(xd, wd, bd, yd, N, H, W, Cin, Cout, R, S_, L.act), "conv2d_fwd_tc_x3")
    torch.cuda.synchronize()
    assert sc.sc_last_device_status() == sc.SC_OK
    y = nhwc_to_nchw(yd.cpu().numpy().reshape(N, H, W, Cout))
    yr, a = oracle_mod.conv2d_nchw(c.x, L.w, L.b, L.act)
    assert_conv_close(y, yr, a, what=f"tc_x3 {shape}")
