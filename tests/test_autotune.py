"""First-call autotuning of conv2d_fwd's tile configuration: every candidate
configuration matches the oracle; a tuned call caches its choice and gives
the same result again; a call captured into a CUDA graph is not timed and
caches nothing."""
import numpy as np
import pytest
import torch

import synthetic as S
import stencil_conv2d_fwd_gb300 as sc_mod
from parity_util import assert_conv_close, conv_gpu, nchw_to_nhwc, nhwc_to_nchw

CLASSES = [
    # (N, Cin, Cout, H, W): one shape per output-channel class, tiles ragged
    (1, 32, 64, 21, 70),
    (1, 32, 32, 19, 133),
    (1, 16, 16, 18, 150),
    (1, 8, 8, 9, 300),
    (1, 32, 4, 13, 517),
    (1, 12, 40, 9, 35),     # Cin % 16 != 0: only the default configuration
]


def test_candidates_are_listed_on_the_host():
    # host-side calls only: no GPU needed
    sc = sc_mod
    names = sc.sc_autotune_candidates(32, 32, 3, 3)
    assert len(names) >= 2 and names[0] == "heuristic"
    assert sc.sc_autotune_candidates(32, 4, 3, 3)[0] == "heuristic"
    assert sc.sc_autotune_candidates(12, 40, 3, 3) == ["heuristic"]
    assert sc.sc_autotune_candidates(1, 32, 5, 5) == []
    assert sc.sc_autotune_candidates(32, 32, 5, 5) == []


def test_switch_returns_the_previous_setting():
    sc = sc_mod
    prev = sc.sc_set_autotune(1)
    try:
        assert sc.sc_set_autotune(0) == 1
        assert sc.sc_set_autotune(0) == 0
    finally:
        sc.sc_set_autotune(prev)


def _run_candidate(x_nchw, w, b, act, cand, dev):
    N, Cin, H, W = x_nchw.shape
    Cout = w.shape[0]
    xd = torch.from_numpy(nchw_to_nhwc(x_nchw)).to(dev)
    wd = torch.from_numpy(np.ascontiguousarray(w)).to(dev)
    bd = torch.from_numpy(b).to(dev)
    yd = torch.full((N * H * W * Cout,), float("nan"), device=dev)
    rc = sc_mod.sc_test_conv_candidate(xd, wd, bd, yd, N, H, W, Cin, Cout, 3, 3, act, cand)
    torch.cuda.synchronize()
    return rc, nhwc_to_nchw(yd.cpu().numpy().reshape(N, H, W, Cout))


@pytest.mark.gpu
@pytest.mark.parametrize("shape", CLASSES, ids=[str(s) for s in CLASSES])
def test_every_candidate_matches_the_oracle(oracle_mod, cuda_dev, sc, shape):
    N, Cin, Cout, H, W = shape
    c = S.conv_case(900 + Cin + Cout + W, N, Cin, Cout, H, W, 3, 3, act=1)
    L = c.layers[0]
    yr, a = oracle_mod.conv2d_nchw(c.x, L.w, L.b, L.act)
    names = sc.sc_autotune_candidates(Cin, Cout, 3, 3)
    ran = 0
    for i, name in enumerate(names):
        rc, y = _run_candidate(c.x, L.w, L.b, L.act, i, cuda_dev)
        if rc == sc.SC_ERR_UNSUPPORTED:
            continue
        assert rc == sc.SC_OK, (name, sc.sc_status_string(rc))
        assert_conv_close(y, yr, a, what=f"candidate {i} ({name}) {shape}")
        ran += 1
    assert ran >= 1
    assert sc.sc_last_device_status() == sc.SC_OK
    # out-of-range candidates are refused
    rc, _ = _run_candidate(c.x, L.w, L.b, L.act, len(names), cuda_dev)
    assert rc == sc.SC_ERR_UNSUPPORTED


TMA_EDGES = [
    # (N, Cin, Cout, H, W): TMA-staged candidates at their edges
    (2, 12, 4, 7, 165),     # Cin % 8 != 0 (zero-filled channels), batch of 2, ragged tiles
    (1, 4, 8, 5, 9),        # a single 4-channel step, image narrower than one tile
    (1, 64, 16, 6, 81),     # 8 steps per tile, two output-channel lanes per pixel
    (3, 20, 4, 3, 161),     # image shorter than one tile
]


@pytest.mark.gpu
@pytest.mark.parametrize("shape", TMA_EDGES, ids=[str(s) for s in TMA_EDGES])
def test_tma_candidates_at_their_edges(oracle_mod, cuda_dev, sc, shape):
    N, Cin, Cout, H, W = shape
    c = S.conv_case(970 + Cin + Cout + W, N, Cin, Cout, H, W, 3, 3, act=0)
    L = c.layers[0]
    yr, a = oracle_mod.conv2d_nchw(c.x, L.w, L.b, L.act)
    names = sc.sc_autotune_candidates(Cin, Cout, 3, 3)
    ran = 0
    for i, name in enumerate(names):
        if not name.startswith("TMA"):
            continue
        rc, y = _run_candidate(c.x, L.w, L.b, L.act, i, cuda_dev)
        assert rc == sc.SC_OK, (name, sc.sc_status_string(rc))
        assert_conv_close(y, yr, a, what=f"candidate {i} ({name}) {shape}")
        ran += 1
    assert ran >= 1
    assert sc.sc_last_device_status() == sc.SC_OK


N4_MANY_TILES = [
    # (N, Cin, Cout, H, W): 32 -> 4 with more 8 x 160 tiles than CTAs, so the
    # narrow-output kernels' CTAs take several tiles (the cross-step prefetch
    # runs across tile boundaries); ragged right and bottom edges, several
    # images
    (12, 32, 4, 75, 330),
    (5, 32, 4, 41, 1281),
]


@pytest.mark.gpu
@pytest.mark.parametrize("shape", N4_MANY_TILES, ids=[str(s) for s in N4_MANY_TILES])
@pytest.mark.parametrize("act", [0, 1])
def test_narrow_output_candidates_with_many_tiles(oracle_mod, cuda_dev, sc, shape, act):
    N, Cin, Cout, H, W = shape
    c = S.conv_case(980 + W + act, N, Cin, Cout, H, W, 3, 3, act=act)
    L = c.layers[0]
    yr, a = oracle_mod.conv2d_nchw(c.x, L.w, L.b, L.act)
    names = sc.sc_autotune_candidates(Cin, Cout, 3, 3)
    ran = 0
    for i, name in enumerate(names):
        if not name.startswith("N4"):
            continue
        rc, y = _run_candidate(c.x, L.w, L.b, L.act, i, cuda_dev)
        assert rc == sc.SC_OK, (name, sc.sc_status_string(rc))
        assert_conv_close(y, yr, a, what=f"candidate {i} ({name}) {shape}")
        ran += 1
    assert ran >= 2
    assert sc.sc_last_device_status() == sc.SC_OK


@pytest.mark.gpu
def test_tuned_call_caches_its_choice_and_repeats(oracle_mod, cuda_dev, sc):
    N, Cin, Cout, H, W = 1, 32, 32, 23, 97
    c = S.conv_case(950, N, Cin, Cout, H, W, 3, 3, act=1)
    L = c.layers[0]
    yr, a = oracle_mod.conv2d_nchw(c.x, L.w, L.b, L.act)
    sc.sc_autotune_clear()
    prev = sc.sc_set_autotune(1)
    try:
        assert sc.sc_autotune_lookup(N, H, W, Cin, Cout, 3, 3, L.act, True) == -1
        y1 = conv_gpu(c.x, L.w, L.b, L.act, cuda_dev)
        choice = sc.sc_autotune_lookup(N, H, W, Cin, Cout, 3, 3, L.act, True)
        assert 0 <= choice < len(sc.sc_autotune_candidates(Cin, Cout, 3, 3))
        y2 = conv_gpu(c.x, L.w, L.b, L.act, cuda_dev)
        assert_conv_close(y1, yr, a, what="tuned first call")
        assert np.array_equal(y1, y2), "the cached choice must reproduce the first call's output"
        # NCHW callers go through the same tuned path
        y3 = conv_gpu(c.x, L.w, L.b, L.act, cuda_dev, layout=sc.SC_NCHW)
        assert_conv_close(y3, yr, a, what="tuned NCHW call")
    finally:
        sc.sc_set_autotune(prev)
        sc.sc_autotune_clear()
    assert sc.sc_autotune_lookup(N, H, W, Cin, Cout, 3, 3, L.act, True) == -1


@pytest.mark.gpu
def test_captured_call_is_not_timed(oracle_mod, cuda_dev, sc):
    N, Cin, Cout, H, W = 1, 32, 4, 17, 211
    c = S.conv_case(960, N, Cin, Cout, H, W, 3, 3, act=1)
    L = c.layers[0]
    yr, a = oracle_mod.conv2d_nchw(c.x, L.w, L.b, L.act)
    xd = torch.from_numpy(nchw_to_nhwc(c.x)).to(cuda_dev)
    wd = torch.from_numpy(L.w).to(cuda_dev)
    bd = torch.from_numpy(L.b).to(cuda_dev)
    yd = torch.zeros(N * H * W * Cout, device=cuda_dev)
    sc.sc_autotune_clear()
    prev = sc.sc_set_autotune(1)
    try:
        s = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                rc = sc.conv2d_fwd(xd, wd, bd, yd, N, H, W, Cin, Cout, 3, 3, sc.SC_NHWC, L.act, s)
        assert rc == sc.SC_OK
        assert sc.sc_autotune_lookup(N, H, W, Cin, Cout, 3, 3, L.act, True) == -1
        g.replay()
        torch.cuda.synchronize()
    finally:
        sc.sc_set_autotune(prev)
        sc.sc_autotune_clear()
    y = nhwc_to_nchw(yd.cpu().numpy().reshape(N, H, W, Cout))
    assert_conv_close(y, yr, a, what="captured tuned call")
