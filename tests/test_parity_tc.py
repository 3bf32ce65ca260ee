"""conv2d_fwd_tc (tcgen05, TF32 operands, fp32 accumulation) vs the fp64
oracle.  Its own tolerance: |y - y_ref| <= 5e-3 * (sum |x * w| + |b|) per
element (TF32 keeps 10 explicit mantissa bits of x and w)."""
import numpy as np
import pytest
import torch

import synthetic as S
import stencil_conv2d_fwd_gb300 as sc
from parity_util import assert_conv_close, check_canaries, guarded_empty, nchw_to_nhwc, nhwc_to_nchw

pytestmark = pytest.mark.gpu
TC_RTOL = 5e-3


def conv_tc(x_nchw, w, b, act, dev):
    N, Cin, H, W = x_nchw.shape
    Cout, _, R, S_ = w.shape
    xd = torch.from_numpy(nchw_to_nhwc(x_nchw)).to(dev)
    wd = torch.from_numpy(np.ascontiguousarray(w)).to(dev)
    bd = None if b is None else torch.from_numpy(b).to(dev)
    n_out = N * H * W * Cout
    buf, yd = guarded_empty(n_out, dev)
    sc.check(sc.conv2d_fwd_tc(xd, wd, bd, yd, N, H, W, Cin, Cout, R, S_, act), "conv2d_fwd_tc")
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
    # 4 output channels, 3 x 3: all nine taps in N (an image shorter than a
    # tile, Cin not a multiple of 8, two 32-channel stages, N > 1)
    (2, 8, 4, 7, 29, 3, 3),
    (1, 12, 4, 5, 200, 3, 3),
    (1, 64, 4, 37, 95, 3, 3),
    (3, 16, 4, 50, 31, 3, 3),
    # filters too large for 32-channel groups: 16- and 8-channel groups
    (1, 128, 32, 9, 40, 3, 3),
    (1, 256, 12, 6, 33, 3, 3),
]


@pytest.mark.parametrize("shape", SHAPES, ids=[str(s) for s in SHAPES])
def test_tc_shapes(oracle_mod, cuda_dev, sc, shape):
    N, Cin, Cout, H, W, R, S_ = shape
    c = S.conv_case(600 + Cin + Cout + W, N, Cin, Cout, H, W, R, S_, act=1)
    L = c.layers[0]
    y = conv_tc(c.x, L.w, L.b, L.act, cuda_dev)
    yr, a = oracle_mod.conv2d_nchw(c.x, L.w, L.b, L.act)
    assert_conv_close(y, yr, a, rtol=TC_RTOL, what=f"tc {shape}")


@pytest.mark.parametrize("cid,li", [(4, 0), (3, 1), (3, 2)])
def test_tc_workloads_full_size(oracle_mod, cuda_dev, sc, cid, li):
    wl = S.config(cid)
    L = wl.layers[li]
    x = wl.x if li == 0 else np.maximum(S.uniform(77, 0, (wl.n, L.cin, wl.h, wl.w), -1, 1), 0).astype(np.float32)
    y = conv_tc(x, L.w, L.b, L.act, cuda_dev)
    yr, a = oracle_mod.conv2d_nchw(x, L.w, L.b, L.act)
    worst = assert_conv_close(y, yr, a, rtol=TC_RTOL, what=f"tc workload {cid} layer {li}")
    assert worst < 1.0


def test_tc_rejects_what_it_does_not_run(cuda_dev, sc):
    x = torch.zeros(4 * 8 * 8 * 6, device=cuda_dev)
    w = torch.zeros(4 * 6 * 25, device=cuda_dev)
    y = torch.zeros(4 * 8 * 8 * 4, device=cuda_dev)
    assert sc.conv2d_fwd_tc(x, w, None, y, 1, 8, 8, 6, 4, 3, 3, 0) == sc.SC_ERR_UNSUPPORTED
    assert sc.conv2d_fwd_tc(x, w, None, y, 1, 8, 8, 4, 4, 5, 5, 0) == sc.SC_ERR_UNSUPPORTED
    # filters that stay too large even in 4-channel groups
    xb = torch.zeros(8 * 8 * 600, device=cuda_dev)
    wb = torch.zeros(4 * 600 * 9, device=cuda_dev)
    assert sc.conv2d_fwd_tc(xb, wb, None, y, 1, 8, 8, 600, 4, 3, 3, 0) == sc.SC_ERR_UNSUPPORTED
    # the filters are bulk-copied: w must be 16-byte aligned like x and y
    wu = torch.zeros(4 * 4 * 9 + 1, device=cuda_dev)[1:]
    assert sc.conv2d_fwd_tc(x, wu, None, y, 1, 8, 8, 4, 4, 3, 3, 0) == sc.SC_ERR_ALIGN
    torch.cuda.synchronize()
    assert sc.sc_last_device_status() == sc.SC_OK


def test_tf32_operands_are_truncated(cuda_dev, sc):
    """The TF32 MMA reads an fp32 operand as its upper 19 bits (the 13 low
    mantissa bits dropped, rounding toward zero).  conv2d_fwd_tc_x3 relies on
    this: it feeds the copied activations to the MMA as their TF32 heads.  A
    1 x 1 convolution with a unit weight (or a unit input) returns each
    operand as the MMA saw it."""
    vals = np.array([1 + 2 ** -11 + 2 ** -12, 1 + 2 ** -11, 1 + 2 ** -12, 1 + 2 ** -10 + 2 ** -11,
                     -(1 + 2 ** -11 + 2 ** -12), 1 + 2 ** -11 + 2 ** -23, 3.0e-5 * (1 + 2 ** -11)], dtype=np.float32)
    head = (vals.view(np.uint32) & np.uint32(0xFFFFE000)).view(np.float32)
    n = len(vals)
    for side in ("x", "w"):
        got = []
        for v in vals:
            x = np.zeros((1, 1, 32, 4), np.float32)
            w = np.zeros((4, 4, 1, 1), np.float32)
            x[0, 0, 0, 0] = v if side == "x" else 1.0
            w[0, 0, 0, 0] = 1.0 if side == "x" else v
            yd = torch.zeros(32 * 4, device=cuda_dev)
            sc.check(sc.conv2d_fwd_tc(torch.from_numpy(x).to(cuda_dev), torch.from_numpy(w).to(cuda_dev), None, yd,
                                      1, 1, 32, 4, 4, 1, 1, 0), "conv2d_fwd_tc")
            torch.cuda.synchronize()
            got.append(yd.cpu().numpy()[0])
        assert np.array_equal(np.array(got, np.float32), head), (side, got, head)
    assert n == len(head)
