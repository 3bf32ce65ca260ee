"""conv2d_fwd_tc_x3 (tcgen05, split-TF32 operands: three TF32 products per product,
head and correction accumulators) vs the fp64 oracle, at conv2d_fwd's own
fp32 bound |y - y_ref| <= 1e-5 * (sum |x * w| + |b|) per element.  One test
also runs plain TF32 (conv2d_fwd_tc) on the same data to show that bound is
out of its reach, so a split that silently dropped its correction products
would fail here."""
import numpy as np
import pytest
import torch

import synthetic as S
import stencil_conv2d_fwd_gb300 as sc
from parity_util import CONV_RTOL, assert_conv_close, check_canaries, guarded_empty, nchw_to_nhwc, nhwc_to_nchw

pytestmark = pytest.mark.gpu


def conv_tc(entry, x_nchw, w, b, act, dev):
    N, Cin, H, W = x_nchw.shape
    Cout, _, R, S_ = w.shape
    xd = torch.from_numpy(nchw_to_nhwc(x_nchw)).to(dev)
    wd = torch.from_numpy(np.ascontiguousarray(w)).to(dev)
    bd = None if b is None else torch.from_numpy(b).to(dev)
    n_out = N * H * W * Cout
    buf, yd = guarded_empty(n_out, dev)
    sc.check(entry(xd, wd, bd, yd, N, H, W, Cin, Cout, R, S_, act), entry.__name__)
    st = sc.sc_last_device_status()
    assert st == sc.SC_OK, sc.sc_status_string(st)
    torch.cuda.synchronize()
    check_canaries(buf, n_out)
    return nhwc_to_nchw(yd.cpu().numpy().reshape(N, H, W, Cout))


SHAPES = [
    # (N, Cin, Cout, H, W, R, S)
    (1, 8, 16, 9, 13, 3, 3),
    (1, 4, 4, 1, 1, 3, 3),
    (2, 16, 32, 33, 70, 3, 3),
    (1, 12, 20, 17, 130, 3, 3),
    (1, 64, 128, 10, 40, 3, 3),
    (1, 32, 4, 20, 300, 3, 3),
    (1, 16, 48, 11, 257, 3, 3),
    (1, 8, 16, 12, 17, 1, 1),
    (1, 8, 12, 12, 17, 3, 1),
    (1, 40, 8, 7, 61, 1, 3),
    # 4 output channels, 3 x 3: all nine taps in N
    (2, 8, 4, 7, 29, 3, 3),
    (1, 12, 4, 5, 200, 3, 3),
    (1, 64, 4, 37, 95, 3, 3),
    (3, 16, 4, 50, 31, 3, 3),
    # filters too large for 32-channel groups: 16-, 8- and 4-channel groups
    (1, 64, 64, 9, 40, 3, 3),
    (1, 128, 32, 9, 40, 3, 3),
    (1, 256, 12, 6, 33, 3, 3),
]


@pytest.mark.parametrize("shape", SHAPES, ids=[str(s) for s in SHAPES])
@pytest.mark.parametrize("act", [0, 1])
def test_x3_shapes(oracle_mod, cuda_dev, sc, shape, act):
    N, Cin, Cout, H, W, R, S_ = shape
    c = S.conv_case(900 + Cin + Cout + W, N, Cin, Cout, H, W, R, S_, act=act)
    L = c.layers[0]
    y = conv_tc(sc.conv2d_fwd_tc_x3, c.x, L.w, L.b, L.act, cuda_dev)
    yr, a = oracle_mod.conv2d_nchw(c.x, L.w, L.b, L.act)
    assert_conv_close(y, yr, a, what=f"tc_x3 {shape}")


@pytest.mark.parametrize("cid,li", [(4, 0), (3, 1), (3, 2)])
def test_x3_workloads_full_size(oracle_mod, cuda_dev, sc, cid, li):
    wl = S.config(cid)
    L = wl.layers[li]
    x = wl.x if li == 0 else np.maximum(S.uniform(77, 0, (wl.n, L.cin, wl.h, wl.w), -1, 1), 0).astype(np.float32)
    y = conv_tc(sc.conv2d_fwd_tc_x3, x, L.w, L.b, L.act, cuda_dev)
    yr, a = oracle_mod.conv2d_nchw(x, L.w, L.b, L.act)
    assert_conv_close(y, yr, a, what=f"tc_x3 workload {cid} layer {li}")


def test_x3_meets_the_fp32_bound_that_tf32_misses(oracle_mod, cuda_dev, sc):
    c = S.conv_case(931, 1, 32, 32, 24, 90, 3, 3, act=0)
    L = c.layers[0]
    yr, a = oracle_mod.conv2d_nchw(c.x, L.w, L.b, L.act)
    y3 = conv_tc(sc.conv2d_fwd_tc_x3, c.x, L.w, L.b, L.act, cuda_dev)
    worst3 = assert_conv_close(y3, yr, a, what="tc_x3")
    y1 = conv_tc(sc.conv2d_fwd_tc, c.x, L.w, L.b, L.act, cuda_dev)
    worst1 = float((np.abs(y1 - yr) / (CONV_RTOL * a)).max())
    assert worst1 > 1.0, f"plain TF32 stayed within the fp32 bound ({worst1}): the check cannot tell the split apart"
    assert worst3 < worst1 / 20, (worst3, worst1)


def test_x3_same_sign_sums(oracle_mod, cuda_dev, sc):
    """Non-negative inputs and filters: every partial sum grows towards
    sum |x * w|, the case where rounding in the accumulators is largest
    relative to the bound."""
    N, Cin, Cout, H, W = 1, 64, 32, 16, 64
    x = S.uniform(932, 0, (N, Cin, H, W), 0.0, 1.0).astype(np.float32)
    w = S.uniform(932, 1, (Cout, Cin, 3, 3), 0.0, 2.0 / (9 * Cin)).astype(np.float32)
    b = np.zeros(Cout, dtype=np.float32)
    y = conv_tc(sc.conv2d_fwd_tc_x3, x, w, b, 0, cuda_dev)
    yr, a = oracle_mod.conv2d_nchw(x, w, b, 0)
    assert_conv_close(y, yr, a, what="tc_x3 same-sign")


def test_x3_without_bias_and_several_images(oracle_mod, cuda_dev, sc):
    c = S.conv_case(933, 3, 24, 28, 11, 47, 3, 3, act=1)
    L = c.layers[0]
    y = conv_tc(sc.conv2d_fwd_tc_x3, c.x, L.w, None, L.act, cuda_dev)
    yr, a = oracle_mod.conv2d_nchw(c.x, L.w, np.zeros(L.cout, dtype=np.float32), L.act)
    assert_conv_close(y, yr, a, what="tc_x3 no bias")


def test_x3_rejects_what_it_does_not_run(cuda_dev, sc):
    x = torch.zeros(4 * 8 * 8 * 6, device=cuda_dev)
    w = torch.zeros(4 * 6 * 25, device=cuda_dev)
    y = torch.zeros(4 * 8 * 8 * 4, device=cuda_dev)
    assert sc.conv2d_fwd_tc_x3(x, w, None, y, 1, 8, 8, 6, 4, 3, 3, 0) == sc.SC_ERR_UNSUPPORTED
    assert sc.conv2d_fwd_tc_x3(x, w, None, y, 1, 8, 8, 4, 4, 5, 5, 0) == sc.SC_ERR_UNSUPPORTED
    # heads and remainders of the filters do not fit in shared memory (plain
    # TF32 still runs this shape; with 4 output channels the nine-taps-in-N
    # layout's smaller stages leave room, so 8 are used here)
    xb = torch.zeros(8 * 8 * 320, device=cuda_dev)
    wb = torch.zeros(8 * 320 * 9, device=cuda_dev)
    y8 = torch.zeros(8 * 8 * 8, device=cuda_dev)
    assert sc.conv2d_fwd_tc_x3(xb, wb, None, y8, 1, 8, 8, 320, 8, 3, 3, 0) == sc.SC_ERR_UNSUPPORTED
    assert sc.conv2d_fwd_tc(xb, wb, None, y8, 1, 8, 8, 320, 8, 3, 3, 0) == sc.SC_OK
    assert sc.conv2d_fwd_tc_x3(xb, wb, None, y8, 1, 8, 8, 320, 4, 3, 3, 0) == sc.SC_OK
    wu = torch.zeros(4 * 4 * 9 + 1, device=cuda_dev)[1:]
    assert sc.conv2d_fwd_tc_x3(x, wu, None, y, 1, 8, 8, 4, 4, 3, 3, 0) == sc.SC_ERR_ALIGN
    torch.cuda.synchronize()
    assert sc.sc_last_device_status() == sc.SC_OK
