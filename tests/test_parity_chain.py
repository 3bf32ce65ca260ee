"""conv2d_chain_fwd_host on the GPU: a chain of layers from a host input to a
host output.

The chain runs conv2d_fwd's kernels on the same data, so its output must
equal, bit for bit, the same layers run one conv2d_fwd call at a time on
device buffers; each of those layers is held to the fp64 oracle fed the
GPU's own input to it, at the fp32 bound 1e-5 * A.  Covered: the 3-layer
net of workload 3 at a reduced and at its full size, pinned and pageable
host buffers, chains of one layer, and batches of images.
"""
import numpy as np
import pytest
import torch

import synthetic as S
import stencil_conv2d_fwd_gb300 as sc
from parity_util import assert_conv_close, nchw_to_nhwc, nhwc_to_nchw

pytestmark = pytest.mark.gpu


def _layers_on_device(layers, dev):
    keep, spec = [], []
    for L in layers:
        wd = torch.from_numpy(np.ascontiguousarray(L.w)).to(dev)
        bd = torch.from_numpy(np.ascontiguousarray(L.b)).to(dev)
        keep += [wd, bd]
        spec.append((wd, bd, L.cout, L.r, L.s, L.act))
    return keep, spec


def _chain_host(x_nchw, spec, dev, pinned=True):
    N, Cin, H, W = x_nchw.shape
    cout = spec[-1][2]
    x_nhwc = torch.from_numpy(nchw_to_nhwc(x_nchw))
    y = torch.full((N * H * W * cout,), np.nan, dtype=torch.float32)
    if pinned:
        x_nhwc, y = x_nhwc.pin_memory(), y.pin_memory()
    sc.check(sc.conv2d_chain_fwd_host(x_nhwc, y, N, H, W, Cin, spec), "conv2d_chain_fwd_host")
    torch.cuda.synchronize()
    assert sc.sc_last_device_status() == sc.SC_OK
    return nhwc_to_nchw(y.numpy().reshape(N, H, W, cout))


def _chain_layer_by_layer(oracle_mod, x_nchw, layers, spec, dev):
    """conv2d_fwd one layer at a time on device buffers; every layer checked
    against the oracle on the GPU's own input.  Returns the last output."""
    N, Cin, H, W = x_nchw.shape
    cur = torch.from_numpy(nchw_to_nhwc(x_nchw)).to(dev)
    cin = Cin
    for li, (L, (wd, bd, cout, r, s, act)) in enumerate(zip(layers, spec)):
        y = torch.empty(N * H * W * cout, device=dev)
        sc.check(sc.conv2d_fwd(cur, wd, bd, y, N, H, W, cin, cout, r, s, sc.SC_NHWC, act), "conv2d_fwd")
        torch.cuda.synchronize()
        x_in = nhwc_to_nchw(cur.cpu().numpy().reshape(N, H, W, cin))
        yr, a = oracle_mod.conv2d_nchw(x_in, L.w, L.b, L.act)
        assert_conv_close(nhwc_to_nchw(y.cpu().numpy().reshape(N, H, W, cout)), yr, a, what=f"layer {li + 1}")
        cur, cin = y, cout
    return nhwc_to_nchw(cur.cpu().numpy().reshape(N, H, W, cin))


@pytest.mark.parametrize("size", ["reduced", "full"])
def test_upscaling_net_chain_from_host(oracle_mod, cuda_dev, sc, size):
    scale = {"h": 45, "w": 77} if size == "reduced" else None
    c = S.config(3, scale=scale)
    keep, spec = _layers_on_device(c.layers, cuda_dev)
    if size == "full":
        # the full-size layers are held to the oracle by test_parity_conv; here
        # the chain must reproduce the layer-by-layer device path exactly
        N, Cin, H, W = c.x.shape
        cur = torch.from_numpy(nchw_to_nhwc(c.x)).to(cuda_dev)
        cin = Cin
        for wd, bd, cout, r, s, act in spec:
            y = torch.empty(N * H * W * cout, device=cuda_dev)
            sc.check(sc.conv2d_fwd(cur, wd, bd, y, N, H, W, cin, cout, r, s, sc.SC_NHWC, act), "conv2d_fwd")
            cur, cin = y, cout
        torch.cuda.synchronize()
        ref = nhwc_to_nchw(cur.cpu().numpy().reshape(N, H, W, cin))
    else:
        ref = _chain_layer_by_layer(oracle_mod, c.x, c.layers, spec, cuda_dev)
    got = _chain_host(c.x, spec, cuda_dev, pinned=True)
    assert np.array_equal(got, ref), "the chain differs from the same layers run one call at a time"


def test_chain_with_pageable_buffers_one_layer_and_a_batch(oracle_mod, cuda_dev, sc):
    c = S.conv_case(1200, 3, 8, 12, 19, 41, 3, 3, act=1)
    keep, spec = _layers_on_device(c.layers, cuda_dev)
    ref = _chain_layer_by_layer(oracle_mod, c.x, c.layers, spec, cuda_dev)
    assert np.array_equal(_chain_host(c.x, spec, cuda_dev, pinned=False), ref)
    assert np.array_equal(_chain_host(c.x, spec, cuda_dev, pinned=True), ref)


def test_chain_of_mixed_filters(oracle_mod, cuda_dev, sc):
    """1 -> 4 (3x3, ReLU) -> 16 (5x5, ReLU) -> 4 (1x1) -> 8 (3x3): every kernel
    family in one chain, ragged sizes, two images."""
    rng_layers = []
    shapes = [(1, 4, 3, 1), (4, 16, 5, 1), (16, 4, 1, 0), (4, 8, 3, 1)]
    for i, (cin, cout, k, act) in enumerate(shapes):
        L = S.conv_case(1300 + i, 1, cin, cout, 4, 4, k, k, act=act).layers[0]
        rng_layers.append(L)
    x = S.conv_case(1310, 2, 1, 4, 23, 58, 3, 3).x
    keep, spec = _layers_on_device(rng_layers, cuda_dev)
    ref = _chain_layer_by_layer(oracle_mod, x, rng_layers, spec, cuda_dev)
    assert np.array_equal(_chain_host(x, spec, cuda_dev), ref)


@pytest.mark.parametrize("pinned", [True, False])
def test_chain_of_one_single_channel_layer(oracle_mod, cuda_dev, sc, pinned):
    """A chain of one layer with one input channel (the tiled single-channel
    kernel, whose stores go through shared memory and the TMA), pinned and
    pageable host buffers."""
    c = S.conv_case(1320, 2, 1, 32, 29, 140, 5, 5, act=1)
    keep, spec = _layers_on_device(c.layers, cuda_dev)
    ref = _chain_layer_by_layer(oracle_mod, c.x, c.layers, spec, cuda_dev)
    assert np.array_equal(_chain_host(c.x, spec, cuda_dev, pinned=pinned), ref)


def test_chain_captured_in_a_cuda_graph(oracle_mod, cuda_dev, sc):
    """The call is stream-ordered throughout (pool buffers, copies, launches),
    so it can be captured into a CUDA graph; two replays on new host data
    give the results of direct calls."""
    c = S.config(3, scale={"h": 37, "w": 161})
    keep, spec = _layers_on_device(c.layers, cuda_dev)
    N, Cin, H, W = c.x.shape
    cout = spec[-1][2]
    x_host = torch.from_numpy(nchw_to_nhwc(c.x)).pin_memory()
    y_host = torch.full((N * H * W * cout,), np.nan, dtype=torch.float32).pin_memory()
    ref = _chain_host(c.x, spec, cuda_dev, pinned=True)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            rc = sc.conv2d_chain_fwd_host(x_host, y_host, N, H, W, Cin, spec, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    assert rc == sc.SC_OK, sc.sc_status_string(rc)
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(nhwc_to_nchw(y_host.numpy().reshape(N, H, W, cout)), ref)
    # new input in the same pinned buffer: the replay reads it
    x2 = (c.x * 0.5).astype(np.float32)
    x_host.copy_(torch.from_numpy(nchw_to_nhwc(x2)))
    y_host.fill_(np.nan)
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(nhwc_to_nchw(y_host.numpy().reshape(N, H, W, cout)), _chain_host(x2, spec, cuda_dev))
