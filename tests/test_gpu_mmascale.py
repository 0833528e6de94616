"""Block scales in the 128 x 4 block layout of block-scaled MMA, against
the oracle byte for byte: random scale arrays (ragged rows and columns, a
leading dimension wider than the scale count), and the scales the library's
own MX and NVFP4 quantizers write."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import Guarded, dev, host, require_cuda

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("rows,scale_cols,s_ld", [(128, 4, 4), (300, 7, 7), (1, 1, 3), (257, 256, 260),
                                                  (8192, 256, 256)])
def test_random_scales(rows, scale_cols, s_ld):
    fq = require_cuda()
    s = np.random.default_rng(91).integers(0, 256, size=(rows, s_ld), dtype=np.uint64).astype(np.uint8)
    want = oracle.mma_scale_layout(s, scale_cols)
    out = Guarded((want.size,))
    fq.mx_scales_to_mma_layout(dev(s), scale_cols, out=out.t)
    torch.cuda.synchronize()
    out.check()
    np.testing.assert_array_equal(host(out.t), want)


def test_library_scales():
    """The rowwise and grouped columnwise MX scales and NVFP4's block
    scales of one activation, rearranged on the GPU."""
    fq = require_cuda()
    x = synth.config2(384, 1024, seed=92)
    xd = dev(x)
    offs = [0, 100, 100, 250, 384]
    r = fq.mxfp8_quantize(xd, fq.E4M3, fq.BOTH, group_offsets=offs)
    T = fq.mxfp8_col_blocks(384, offs)
    nv = fq.fp8q_quantize_nvfp4(xd)
    for s, sc in ((r["s_row"], 32), (r["s_col"], T), (nv["s"], 64)):
        got = host(fq.mx_scales_to_mma_layout(s, sc))
        want = oracle.mma_scale_layout(host(s), sc)
        np.testing.assert_array_equal(got, want)
