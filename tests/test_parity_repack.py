"""sc_repack (NCHW <-> NHWC) on the GPU vs the oracle's index definition: bit-exact."""
import numpy as np
import pytest
import torch

import synthetic as S
import stencil_conv2d_fwd_gb300 as sc
from parity_util import check_canaries, guarded_empty

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shape", [(1, 1, 1, 1), (1, 4, 3, 5), (2, 16, 7, 9), (1, 32, 40, 33),
                                   (3, 64, 5, 70), (1, 5, 31, 33), (1, 100, 3, 3), (2, 4, 128, 128),
                                   # 16-byte kernel (C % 4 == 0, H * W % 4 == 0): full and ragged
                                   # 32 x 128 tiles, fewer than 32 channels
                                   (1, 64, 56, 56), (2, 8, 3, 44), (1, 12, 20, 36), (1, 36, 9, 60)])
@pytest.mark.parametrize("to_nhwc", [True, False])
def test_repack(oracle_mod, cuda_dev, sc, shape, to_nhwc):
    N, C, H, W = shape
    src = S.uniform(50 + C, 0, (N * C * H * W,), -1, 1)
    ref = oracle_mod.repack(src, N, C, H, W, to_nhwc).reshape(-1)
    sd = torch.from_numpy(src).to(cuda_dev)
    buf, dd = guarded_empty(src.size, cuda_dev)
    srcl, dstl = (sc.SC_NCHW, sc.SC_NHWC) if to_nhwc else (sc.SC_NHWC, sc.SC_NCHW)
    sc.check(sc.sc_repack(sd, dd, N, C, H, W, srcl, dstl))
    torch.cuda.synchronize()
    check_canaries(buf, src.size)
    np.testing.assert_array_equal(dd.cpu().numpy(), ref)
