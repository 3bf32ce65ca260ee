"""conv2d_fwd_nchw_noalloc: the NCHW convolution for callers that must not
allocate device memory during the call (a process that reserved the GPU's
memory up front, a real-time frame loop that cannot risk an allocation).

It must match the fp64 oracle within the fp32 parity tolerance
|y - y_ref| <= 1e-5 * (sum |x * w| + |b|) on two calls in a row (the second
call starts with the first call's data still in the shared scratch array),
take no buffer from the library's memory pool, and accept a problem that
needs exactly the whole scratch array.  This file is collected last on
purpose.
"""
import numpy as np
import pytest
import torch

import synthetic as S
import stencil_conv2d_fwd_gb300 as sc
from parity_util import CONV_RTOL, check_canaries, guarded_empty

pytestmark = pytest.mark.gpu


def _run(fn, c, dev, with_layout):
    L = c.layers[0]
    N, Cin, H, W = c.x.shape
    xd = torch.from_numpy(c.x).to(dev)
    wd = torch.from_numpy(L.w).to(dev)
    bd = torch.from_numpy(L.b).to(dev)
    n = N * H * W * L.cout
    buf, yd = guarded_empty(n, dev)
    if with_layout:
        rc = fn(xd, wd, bd, yd, N, H, W, Cin, L.cout, L.r, L.s, sc.SC_NCHW, L.act)
    else:
        rc = fn(xd, wd, bd, yd, N, H, W, Cin, L.cout, L.r, L.s, L.act)
    sc.check(rc)
    torch.cuda.synchronize()
    check_canaries(buf, n)
    return yd.cpu().numpy().reshape(N, L.cout, H, W)


def _scratch_floats(N, H, W, Cin, Cout):
    """Scratch a call needs: NHWC x rounded up to 64 floats, then NHWC y."""
    nx = N * H * W * Cin if Cin > 1 else 0
    return (nx + 63) // 64 * 64 + (N * H * W * Cout if Cout > 1 else 0)


CASES = [
    (901, 2, 16, 32, 37, 53, 3, 1),   # larger: fills more scratch
    (902, 1, 8, 12, 19, 23, 5, 0),    # smaller: stale data beyond its end
    (903, 1, 1, 16, 21, 33, 5, 1),    # Cin = 1: only the output repack
    (904, 1, 4, 4, 1024, 1024, 3, 1),  # needs exactly the whole scratch array
]


def test_exact_limit_case_fills_the_scratch():
    _, N, Cin, Cout, H, W, _, _ = CASES[3]
    assert _scratch_floats(N, H, W, Cin, Cout) == sc.SC_NOALLOC_SCRATCH_FLOATS


@pytest.mark.parametrize("case", CASES, ids=[str(c[0]) for c in CASES])
def test_noalloc_matches_the_oracle_on_two_calls_in_a_row(oracle_mod, cuda_dev, sc, case):
    seed, N, Cin, Cout, H, W, K, act = case
    c = S.conv_case(seed, N, Cin, Cout, H, W, K, K, act=act)
    L = c.layers[0]
    y_ref, a = oracle_mod.conv2d_nchw(c.x, L.w, L.b, L.act)
    ref = _run(sc.conv2d_fwd, c, cuda_dev, True)
    allocs = sc.sc_test_workspace_allocs()
    for _ in range(2):
        got = _run(sc.conv2d_fwd_nchw_noalloc, c, cuda_dev, False).astype(np.float64)
        assert (np.abs(got - y_ref) <= CONV_RTOL * a).all()
        # and the same as the allocating entry point, which runs the same kernels
        assert (np.abs(got - ref) <= CONV_RTOL * a).all()
    assert sc.sc_test_workspace_allocs() == allocs, "the no-allocation entry point took a pool buffer"


def test_noalloc_rejects_problems_beyond_its_scratch(cuda_dev, sc):
    N, C, H, W = 1, 4, 1024, 1025        # one column more than the exact-limit case
    assert _scratch_floats(N, H, W, C, C) > sc.SC_NOALLOC_SCRATCH_FLOATS
    x = torch.zeros(N * C * H * W, device=cuda_dev)
    w = torch.zeros(C * C * 9, device=cuda_dev)
    y = torch.full((N * C * H * W,), 5.0, device=cuda_dev)
    rc = sc.conv2d_fwd_nchw_noalloc(x, w, None, y, N, H, W, C, C, 3, 3, 0)
    assert rc == sc.SC_ERR_SHAPE
    torch.cuda.synchronize()
    assert (y == 5.0).all()
