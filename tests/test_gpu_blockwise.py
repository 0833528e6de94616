"""Blockwise FP8 (1x128 / 128x1 groups and 128x128 blocks, FP32 scales)
against the oracle, bit for bit: codes and scale_inv of both copies."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import dev, host, require_cuda

pytestmark = pytest.mark.gpu


def _check(fq, x, fmt, block, pow2):
    r = fq.fp8q_quantize_blockwise(dev(x), fmt, block, pow2, fq.BOTH)
    if block == fq.BLOCK_1X128:
        q, si = oracle.blockwise(x, fmt, (1, 128), pow2)
        qt, sit = oracle.blockwise(x, fmt, (128, 1), pow2)
        qt, sit = qt.T, sit.T
    else:
        q, si = oracle.blockwise(x, fmt, (128, 128), pow2)
        qt, sit = q.T, si.T
    np.testing.assert_array_equal(host(r["q"]), q)
    np.testing.assert_array_equal(host(r["scale_inv"]).view(np.uint32), si.view(np.uint32))
    np.testing.assert_array_equal(host(r["q_t"]), qt)
    np.testing.assert_array_equal(host(r["scale_inv_t"]).view(np.uint32), np.ascontiguousarray(sit).view(np.uint32))


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("block", [1, 128])
@pytest.mark.parametrize("pow2", [False, True])
@pytest.mark.parametrize("shape", [(256, 384), (144, 208), (16, 16)])
def test_blockwise_matches_oracle(fmt, block, pow2, shape):
    """Several tiles, and tiles cut short in both directions."""
    fq = require_cuda()
    x = synth.config2(*shape, seed=21 + shape[0])
    _check(fq, x, fmt, block, pow2)


@pytest.mark.parametrize("block", [1, 128])
def test_blockwise_activation_4096(block):
    fq = require_cuda()
    x = synth.config2(4096, 4096, seed=2)
    _check(fq, x, 0, block, False)


def test_blockwise_special_values():
    """A group holding NaN takes scale 1 (its NaN encodes as 0x7F, the rest
    as scale 1 casts); Inf saturates; an all-zero group gets scale 1."""
    fq = require_cuda()
    rng = np.random.default_rng(22)
    x = rng.standard_normal((128, 256)).astype(np.float32)
    x[3, 5] = np.nan
    x[7, 200] = np.inf
    x[9, :128] = 0.0
    _check(fq, synth.to_bf16_bits(x), 0, 1, False)
    _check(fq, synth.to_bf16_bits(x), 0, 128, True)


def test_blockwise_single_direction_leaves_other_copy_alone():
    fq = require_cuda()
    x = synth.config2(128, 256, seed=23)
    r = fq.fp8q_quantize_blockwise(dev(x), 0, fq.BLOCK_1X128, False, fq.ROW)
    assert r["q_t"] is None and r["scale_inv_t"] is None
    q, si = oracle.blockwise(x, 0, (1, 128))
    np.testing.assert_array_equal(host(r["q"]), q)
    r = fq.fp8q_quantize_blockwise(dev(x), 0, fq.BLOCK_1X128, False, fq.COL)
    qt, sit = oracle.blockwise(x, 0, (128, 1))
    np.testing.assert_array_equal(host(r["q_t"]), qt.T)
    fq.check_device()
