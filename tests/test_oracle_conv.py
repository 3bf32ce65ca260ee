"""Pins of the convolution oracle against facts fixed by the definition.

The definition (page "Optimizing convolution kernels - CNNs in Vulkan Part
2/3", sections "Where we left off" and "Vectorization"): centred taps
``x + kx - S/2, y + ky - R/2`` with unflipped weights (cross-correlation),
bias added after the sum, ReLU on the result; zero outside the image.

Each check below is computed independently of the oracle (numpy slicing, a
dense matrix built from the definition, closed forms, torch's fp64 conv2d as
a library special case) so that a flipped kernel, a wrong anchor, a wrong
padding value, a swapped weight index or a misplaced bias fails one of them.
"""
import math

import numpy as np
import pytest
import torch

import synthetic as S


def _grid(seed, shape, step=2.0 ** -8, lim=64):
    """Values k * step with |k| <= lim: sums of a few stay exact in fp32."""
    rng = np.random.default_rng(seed)
    return (rng.integers(-lim, lim + 1, size=shape) * step).astype(np.float32)


@pytest.mark.parametrize("R,S_", [(1, 1), (3, 3), (5, 5), (7, 7), (3, 5), (5, 3)])
def test_centre_delta_returns_input_plus_bias(oracle_mod, R, S_):
    x = S.uniform(7, 0, (2, 3, 9, 11), -1, 1)
    w = np.zeros((3, 3, R, S_), np.float32)
    for c in range(3):
        w[c, c, R // 2, S_ // 2] = 1.0
    b = np.array([0.25, -0.5, 0.125], np.float32)
    y, a = oracle_mod.conv2d_nchw(x, w, b, act=0)
    np.testing.assert_array_equal(y, x.astype(np.float64) + b[None, :, None, None])
    np.testing.assert_array_equal(a, np.abs(x.astype(np.float64)) + np.abs(b)[None, :, None, None])


@pytest.mark.parametrize("R,S_", [(3, 3), (5, 5), (3, 5)])
def test_shifted_delta_shifts_with_zero_fill(oracle_mod, R, S_):
    """Tap (r, s) alone gives y[h][w] = x[h + r - R/2][w + s - S/2], 0 outside."""
    H, W = 7, 10
    x = S.uniform(8, 0, (1, 1, H, W), -1, 1)
    for r in range(R):
        for s in range(S_):
            w = np.zeros((1, 1, R, S_), np.float32)
            w[0, 0, r, s] = 1.0
            y, _ = oracle_mod.conv2d_nchw(x, w, None, act=0)
            dy, dx = r - R // 2, s - S_ // 2
            exp = np.zeros((H, W))
            for h in range(H):
                for ww in range(W):
                    hh, xx = h + dy, ww + dx
                    if 0 <= hh < H and 0 <= xx < W:
                        exp[h, ww] = x[0, 0, hh, xx]
            np.testing.assert_array_equal(y[0, 0], exp)


def test_linearity_in_x_and_w(oracle_mod):
    x1, x2 = _grid(1, (2, 4, 8, 9)), _grid(2, (2, 4, 8, 9))
    w1, w2 = _grid(3, (5, 4, 3, 3)), _grid(4, (5, 4, 3, 3))
    conv = lambda x, w: oracle_mod.conv2d_nchw(x, w, None, act=0)[0]
    lhs = conv(x1 + 2 * x2, w1)  # fp32 inputs exact on this grid
    rhs = conv(x1, w1) + 2 * conv(x2, w1)
    np.testing.assert_allclose(lhs, rhs, rtol=0, atol=1e-12)
    lhs = conv(x1, w1 - 3 * w2)
    rhs = conv(x1, w1) - 3 * conv(x1, w2)
    np.testing.assert_allclose(lhs, rhs, rtol=0, atol=1e-12)


@pytest.mark.parametrize("R", [3, 5])
def test_constant_image_box_filter_closed_form(oracle_mod, R):
    """Constant c, box weights v: value = Cin * c * v * (#in-image taps) + b."""
    N, Cin, Cout, H, W = 1, 3, 2, 9, 12
    c, v = 0.75, 0.5
    x = np.full((N, Cin, H, W), c, np.float32)
    w = np.full((Cout, Cin, R, R), v, np.float32)
    b = np.array([0.125, -2.0], np.float32)
    y, _ = oracle_mod.conv2d_nchw(x, w, b, act=0)
    p = R // 2
    for h in range(H):
        nr = min(h + p, H - 1) - max(h - p, 0) + 1
        for ww in range(W):
            nc = min(ww + p, W - 1) - max(ww - p, 0) + 1
            for co in range(Cout):
                assert y[0, co, h, ww] == Cin * c * v * nr * nc + b[co]
    # interior value, the plain closed form
    assert y[0, 0, H // 2, W // 2] == Cin * c * v * R * R + b[0]


def _pass1d_rows(img, k):
    """Zero-padded 1-D correlation along x of every row (independent of the oracle)."""
    H, W = img.shape
    p = len(k) // 2
    pad = np.zeros((H, W + 2 * p))
    pad[:, p:p + W] = img
    return sum(k[j] * pad[:, j:j + W] for j in range(len(k)))


def test_separable_filter_equals_two_1d_passes(oracle_mod):
    x = S.uniform(9, 0, (1, 1, 13, 17), -1, 1)
    u = np.array([0.25, -1.0, 0.5, 2.0, 0.125])     # column factor (R)
    v = np.array([1.0, 0.5, -0.25])                  # row factor (S)
    w = np.outer(u, v).astype(np.float32)[None, None]
    y, _ = oracle_mod.conv2d_nchw(x, w, None, act=0)
    rows = _pass1d_rows(x[0, 0].astype(np.float64), v)
    cols = _pass1d_rows(rows.T, u).T
    np.testing.assert_allclose(y[0, 0], cols, rtol=0, atol=1e-13)


def _toeplitz(w, H, W):
    """Dense operator of the definition: y_flat = M @ x_flat (NCHW order)."""
    Cout, Cin, R, S_ = w.shape
    M = np.zeros((Cout * H * W, Cin * H * W))
    for co in range(Cout):
        for h in range(H):
            for ww in range(W):
                row = (co * H + h) * W + ww
                for ci in range(Cin):
                    for hh in range(H):
                        for xx in range(W):
                            r, s = hh - h + R // 2, xx - ww + S_ // 2
                            if 0 <= r < R and 0 <= s < S_:
                                M[row, (ci * H + hh) * W + xx] = w[co, ci, r, s]
    return M


@pytest.mark.parametrize("R,act", [(3, 1), (5, 0)])
def test_brute_force_8x8_dense_operator(oracle_mod, R, act):
    H = W = 8
    Cin, Cout = 3, 2
    x = S.uniform(10, 0, (1, Cin, H, W), -1, 1)
    w = S.normal(10, 1, (Cout, Cin, R, R), 0.3)
    b = S.uniform(10, 2, (Cout,), -0.5, 0.5)
    M = _toeplitz(w.astype(np.float64), H, W)
    exp = M @ x.reshape(-1).astype(np.float64) + np.repeat(b.astype(np.float64), H * W)
    if act:
        exp = np.maximum(exp, 0.0)
    y, _ = oracle_mod.conv2d_nchw(x, w, b, act=act)
    np.testing.assert_allclose(y.reshape(-1), exp, rtol=0, atol=1e-13)


def test_bias_then_relu_order(oracle_mod):
    """act(sum + b): a positive sum pulled below zero by the bias reads 0."""
    x = np.full((1, 1, 3, 3), 1.0, np.float32)
    w = np.zeros((1, 1, 1, 1), np.float32)
    w[0, 0, 0, 0] = 0.5
    y, _ = oracle_mod.conv2d_nchw(x, w, np.array([-0.75], np.float32), act=1)
    assert (y == 0.0).all()
    y, _ = oracle_mod.conv2d_nchw(x, w, np.array([-0.25], np.float32), act=1)
    assert (y == 0.25).all()


def test_points_match_full(oracle_mod):
    c = S.conv_case(11, 2, 4, 8, 9, 10, 3, 3, act=1)
    L = c.layers[0]
    y, a = oracle_mod.conv2d_nchw(c.x, L.w, L.b, L.act)
    rng = np.random.default_rng(0)
    pts = np.stack([rng.integers(0, m, 50) for m in (2, 8, 9, 10)], 1).astype(np.int32)
    yp, ap = oracle_mod.conv2d_points(c.x, L.w, L.b, L.act, pts)
    np.testing.assert_array_equal(yp, y[pts[:, 0], pts[:, 1], pts[:, 2], pts[:, 3]])
    np.testing.assert_array_equal(ap, a[pts[:, 0], pts[:, 1], pts[:, 2], pts[:, 3]])


def test_row_band_matches_full(oracle_mod):
    c = S.conv_case(12, 1, 4, 4, 11, 7, 5, 5, act=0)
    L = c.layers[0]
    y, _ = oracle_mod.conv2d_nchw(c.x, L.w, L.b, L.act)
    yb, _ = oracle_mod.conv2d_nchw(c.x, L.w, L.b, L.act, rows=(3, 8))
    np.testing.assert_array_equal(yb, y[:, :, 3:8])


def _torch_ref(x, w, b, act):
    y = torch.nn.functional.conv2d(torch.from_numpy(x).double(), torch.from_numpy(w).double(),
                                   None if b is None else torch.from_numpy(b).double(),
                                   padding=(w.shape[2] // 2, w.shape[3] // 2))
    return (y.relu() if act else y).numpy()


@pytest.mark.parametrize("cid", [1, 2])
def test_library_special_case_small_configs(oracle_mod, cid):
    c = S.config(cid)
    L = c.layers[0]
    y, _ = oracle_mod.conv2d_nchw(c.x, L.w, L.b, L.act)
    np.testing.assert_allclose(y, _torch_ref(c.x, L.w, L.b, L.act), rtol=0, atol=1e-12)


@pytest.mark.slow
@pytest.mark.parametrize("cid", [3, 4])
def test_library_special_case_full_configs(oracle_mod, cid):
    """torch fp64 conv2d on the CPU agrees with the oracle at full workload size
    (config 4 on 4 of its 32 images; every layer of the 3-layer net)."""
    c = S.config(cid)
    x = c.x if cid == 3 else c.x[:4]
    for L in c.layers:
        y, _ = oracle_mod.conv2d_nchw(x, L.w, L.b, L.act)
        np.testing.assert_allclose(y, _torch_ref(x, L.w, L.b, L.act), rtol=0, atol=1e-11)
        x = y.astype(np.float32)


def test_repack_is_the_layout_definition(oracle_mod):
    x = S.uniform(13, 0, (2, 5, 3, 4), -1, 1)
    nhwc = oracle_mod.repack(x, 2, 5, 3, 4, to_nhwc=True)
    np.testing.assert_array_equal(nhwc, x.transpose(0, 2, 3, 1))
    back = oracle_mod.repack(nhwc, 2, 5, 3, 4, to_nhwc=False)
    np.testing.assert_array_equal(back, x)
    assert nhwc[1, 2, 3, 4] == x[1, 4, 2, 3]
