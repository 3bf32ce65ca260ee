"""stencil_pipeline_fwd on the GPU vs the fp64 oracle, 1e-5 absolute."""
import numpy as np
import pytest
import torch

import synthetic as S
import stencil_conv2d_fwd_gb300 as sc
from parity_util import PIPE_ATOL, check_canaries, guarded_empty

pytestmark = pytest.mark.gpu


def pipe_gpu(img, dev, offset=0):
    H, W = img.shape
    src = torch.zeros(H * W + 8, device=dev)
    src[offset:offset + H * W] = torch.from_numpy(img.reshape(-1)).to(dev)
    buf, out = guarded_empty(H * W + 8, dev)
    rc = sc.stencil_pipeline_fwd(src[offset:].data_ptr(), out[offset:].data_ptr(), H, W)
    sc.check(rc, "stencil_pipeline_fwd")
    assert sc.sc_last_device_status() == sc.SC_OK
    torch.cuda.synchronize()
    check_canaries(buf, H * W + 8)
    return out[offset:offset + H * W].cpu().numpy().reshape(H, W)


def test_workload_full_size(oracle_mod, cuda_dev, sc):
    c = S.config(5)
    out = pipe_gpu(c.img, cuda_dev)
    ref = oracle_mod.stencil_pipeline(c.img)
    err = np.abs(out - ref)
    assert err.max() <= PIPE_ATOL, err.max()


@pytest.mark.parametrize("shape", [(1, 1), (1, 9), (6, 1), (2, 2), (5, 7), (33, 70), (130, 1030),
                                   (64, 4096), (300, 129), (257, 2052), (40, 1023)])
def test_shapes(oracle_mod, cuda_dev, sc, shape):
    img = S.uniform(31 + shape[0], 0, shape, 0, 1)
    out = pipe_gpu(img, cuda_dev)
    ref = oracle_mod.stencil_pipeline(img)
    assert np.abs(out - ref).max() <= PIPE_ATOL


@pytest.mark.parametrize("offset", [1, 2, 3])
def test_unaligned_pointers_take_the_scalar_path(oracle_mod, cuda_dev, sc, offset):
    img = S.uniform(41, 0, (37, 260), 0, 1)
    out = pipe_gpu(img, cuda_dev, offset=offset)
    assert np.abs(out - oracle_mod.stencil_pipeline(img)).max() <= PIPE_ATOL


def test_constant_and_impulse(oracle_mod, cuda_dev, sc):
    img = np.full((50, 300), 0.375, np.float32)
    assert np.abs(pipe_gpu(img, cuda_dev) - 0.375).max() <= PIPE_ATOL
    img = np.zeros((50, 300), np.float32)
    img[20, 150] = 0.5
    assert np.abs(pipe_gpu(img, cuda_dev) - oracle_mod.stencil_pipeline(img)).max() <= PIPE_ATOL


def test_bounded_wait_expiry_reports_status_and_context_survives(oracle_mod, cuda_dev, sc):
    """Failure detection without a fault: one TMA copy is never issued, the
    kernel's time-bounded wait for it expires (10 ms), it records
    SC_ERR_DEVICE_TIMEOUT and returns; the next call works normally."""
    img = S.uniform(51, 0, (64, 512), 0, 1)
    ind = torch.from_numpy(img).to(cuda_dev)
    outd = torch.empty_like(ind)
    assert sc.sc_last_device_status() == sc.SC_OK
    rc = sc.sc_test_stencil_wait_expiry(ind, outd, 64, 512, 1, 10000)
    assert rc == sc.SC_OK, sc.sc_status_string(rc)
    assert sc.sc_last_device_status() == sc.SC_ERR_DEVICE_TIMEOUT
    assert sc.sc_last_device_status() == sc.SC_OK          # read clears it
    out = pipe_gpu(img, cuda_dev)                            # context still usable
    assert np.abs(out - oracle_mod.stencil_pipeline(img)).max() <= PIPE_ATOL


def test_wait_expiry_hook_needs_the_tma_path(cuda_dev, sc):
    ind = torch.zeros(8 * 100, device=cuda_dev)
    outd = torch.empty_like(ind)
    assert sc.sc_test_stencil_wait_expiry(ind, outd, 8, 100, 0, 1000) == sc.SC_ERR_UNSUPPORTED
