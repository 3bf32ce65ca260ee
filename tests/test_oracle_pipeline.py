"""Pins of the stencil-pipeline oracle.

Stages (the fused pipeline of page "Model-Based Warp Overlapped Tiling for
Image Processing Programs on GPUs", Abstract, a chain of stencils over one
image): horizontal binomial [1,4,6,4,1]/16, vertical binomial, unsharp mask
out = clamp(in + 1.5 (in - blur), 0, 1), clamp-to-edge borders.
"""
import numpy as np
import pytest
import torch

import synthetic as S

C5 = np.array([1, 4, 6, 4, 1], dtype=np.float64) / 16.0


def test_constant_image_is_fixed(oracle_mod):
    for c in (0.0, 0.3, 1.0):
        img = np.full((9, 13), c, np.float32)
        out = oracle_mod.stencil_pipeline(img)
        np.testing.assert_allclose(out, np.float64(np.float32(c)), rtol=0, atol=1e-15)


def test_linear_ramp_is_fixed_in_the_interior(oracle_mod):
    """The symmetric binomial preserves affine functions away from borders,
    so blur = in and the unsharp step returns in."""
    H, W = 16, 20
    yy, xx = np.mgrid[0:H, 0:W]
    img = ((100 + 2 * xx + 3 * yy) / 1024.0).astype(np.float32)  # exact in fp32
    out, t2 = oracle_mod.stencil_pipeline(img, with_t2=True)
    inner = (slice(2, H - 2), slice(2, W - 2))
    np.testing.assert_allclose(t2[inner], img[inner], rtol=0, atol=1e-14)
    np.testing.assert_allclose(out[inner], img[inner], rtol=0, atol=1e-14)


def test_impulse_gives_outer_product_stencil(oracle_mod):
    H, W, a = 11, 12, 0.5
    img = np.zeros((H, W), np.float32)
    img[5, 6] = a
    out, t2 = oracle_mod.stencil_pipeline(img, with_t2=True)
    exp_t2 = np.zeros((H, W))
    exp_t2[3:8, 4:9] = a * np.outer(C5, C5)
    np.testing.assert_allclose(t2, exp_t2, rtol=0, atol=1e-16)
    exp = np.clip(img + 1.5 * (img - exp_t2), 0, 1)
    np.testing.assert_allclose(out, exp, rtol=0, atol=1e-16)
    assert out[5, 6] == pytest.approx(min(1.0, a + 1.5 * (a - a * 36 / 256)))


def _replicate_ref(img):
    t = torch.from_numpy(img.astype(np.float64))[None, None]
    k = torch.from_numpy(np.outer(C5, C5))[None, None]
    blur = torch.nn.functional.conv2d(torch.nn.functional.pad(t, (2, 2, 2, 2), mode="replicate"), k)
    blur = blur[0, 0].numpy()
    return np.clip(img + 1.5 * (img - blur), 0, 1), blur


@pytest.mark.parametrize("shape", [(8, 8), (5, 7), (1, 9), (6, 1), (2, 2), (33, 70)])
def test_clamp_to_edge_matches_replicate_pad(oracle_mod, shape):
    img = S.uniform(21, 0, shape, 0, 1)
    out, t2 = oracle_mod.stencil_pipeline(img, with_t2=True)
    ref, blur = _replicate_ref(img)
    np.testing.assert_allclose(t2, blur, rtol=0, atol=1e-14)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-14)


def _blur_matrix(n):
    """1-D clamp-to-edge binomial as an n x n matrix, from the stage definition."""
    B = np.zeros((n, n))
    for i in range(n):
        for k in range(-2, 3):
            B[i, min(max(i + k, 0), n - 1)] += C5[k + 2]
    return B


def test_brute_force_8x8(oracle_mod):
    img = S.uniform(22, 0, (8, 8), 0, 1).astype(np.float32)
    B = _blur_matrix(8)
    blur = B @ img.astype(np.float64) @ B.T
    exp = np.clip(img + 1.5 * (img - blur), 0, 1)
    out, t2 = oracle_mod.stencil_pipeline(img, with_t2=True)
    np.testing.assert_allclose(t2, blur, rtol=0, atol=1e-15)
    np.testing.assert_allclose(out, exp, rtol=0, atol=1e-15)


def test_row_band_matches_full(oracle_mod):
    img = S.uniform(23, 0, (30, 17), 0, 1)
    full = oracle_mod.stencil_pipeline(img)
    np.testing.assert_array_equal(oracle_mod.stencil_pipeline(img, rows=(0, 4)), full[0:4])
    np.testing.assert_array_equal(oracle_mod.stencil_pipeline(img, rows=(13, 30)), full[13:30])


def test_output_clamped_to_unit_interval(oracle_mod):
    img = S.uniform(24, 0, (40, 40), 0, 1)
    out = oracle_mod.stencil_pipeline(img)
    assert out.min() >= 0.0 and out.max() <= 1.0
    assert (out == 0.0).any() and (out == 1.0).any()  # the clamp is active on noise
