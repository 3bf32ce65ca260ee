"""Helpers for GPU-vs-oracle parity tests (tests only).

Conv tolerance (fp32 path): |y_gpu - y_ref| <= 1e-5 * A per element, with
A = sum |x * w| + |b| from the oracle.  Pipeline tolerance: 1e-5 absolute.
Outputs are surrounded by guard canaries that must survive the call.
"""
import numpy as np
import torch

import stencil_conv2d_fwd_gb300 as sc

CONV_RTOL = 1e-5
PIPE_ATOL = 1e-5
CANARY = 4096            # floats of guard before and after each output
CANARY_VALUE = -7.75e30


def guarded_empty(n: int, dev) -> tuple:
    """A device buffer with n usable floats (16-byte aligned) between canaries."""
    buf = torch.full((n + 2 * CANARY,), CANARY_VALUE, dtype=torch.float32, device=dev)
    return buf, buf[CANARY:CANARY + n]


def check_canaries(buf: torch.Tensor, n: int):
    h = buf.cpu().numpy()
    assert (h[:CANARY] == CANARY_VALUE).all(), "write before the output buffer"
    assert (h[CANARY + n:] == CANARY_VALUE).all(), "write after the output buffer"


def nchw_to_nhwc(a):
    return np.ascontiguousarray(a.transpose(0, 2, 3, 1))


def nhwc_to_nchw(a):
    return np.ascontiguousarray(a.transpose(0, 3, 1, 2))


def conv_gpu(x_nchw, w, b, act, dev, layout=sc.SC_NHWC, stream=None):
    """Run conv2d_fwd through the C-ABI; returns the output as NCHW float32."""
    N, Cin, H, W = x_nchw.shape
    Cout, _, R, S = w.shape
    xin = x_nchw if layout == sc.SC_NCHW else nchw_to_nhwc(x_nchw)
    xd = torch.from_numpy(np.ascontiguousarray(xin)).to(dev)
    wd = torch.from_numpy(np.ascontiguousarray(w)).to(dev)
    bd = None if b is None else torch.from_numpy(np.ascontiguousarray(b)).to(dev)
    n_out = N * H * W * Cout
    buf, yd = guarded_empty(n_out, dev)
    rc = sc.conv2d_fwd(xd, wd, bd, yd, N, H, W, Cin, Cout, R, S, layout, act, stream=stream)
    sc.check(rc, "conv2d_fwd")
    st = sc.sc_last_device_status(stream)
    assert st == sc.SC_OK, sc.sc_status_string(st)
    torch.cuda.synchronize()
    check_canaries(buf, n_out)
    y = yd.cpu().numpy()
    if layout == sc.SC_NCHW:
        return y.reshape(N, Cout, H, W)
    return nhwc_to_nchw(y.reshape(N, H, W, Cout))


def assert_conv_close(y_gpu, y_ref, scale, rtol=CONV_RTOL, what=""):
    y_gpu = np.asarray(y_gpu, dtype=np.float64)
    err = np.abs(y_gpu - y_ref)
    bound = rtol * scale
    bad = err > bound
    assert np.isfinite(y_gpu).all(), f"{what}: non-finite output"
    if bad.any():
        idx = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {err.size} elements outside {rtol}*A; worst at {idx}: "
            f"gpu={y_gpu[idx]!r} ref={y_ref[idx]!r} A={scale[idx]!r}")
    return float((err / np.maximum(bound, 1e-300)).max())
