"""NVFP4 quantization against the oracle, bit for bit: packed E2M1 codes,
E4M3 block scales, the tensor amax and the tensor scale."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import dev, host, require_cuda

pytestmark = pytest.mark.gpu


def _check(fq, x):
    r = fq.fp8q_quantize_nvfp4(dev(x))
    ref = oracle.nvfp4(x)
    np.testing.assert_array_equal(host(r["s"]), ref["s"])
    np.testing.assert_array_equal(host(r["q"]), ref["q"])
    assert host(r["scale"]).view(np.uint32)[0] == ref["S"].view(np.uint32)
    assert host(r["amax"]).view(np.uint32)[0] == oracle.amax_bits(x)
    return ref


@pytest.mark.parametrize("shape", [(256, 512), (3, 48), (1, 16)])
def test_nvfp4_bf16(shape):
    fq = require_cuda()
    _check(fq, synth.config2(*shape, seed=61 + shape[0]))


def test_nvfp4_fp32():
    fq = require_cuda()
    rng = np.random.default_rng(62)
    _check(fq, (rng.standard_normal((64, 256)) * np.exp(rng.standard_normal((64, 1)) * 5)).astype(np.float32))


def test_nvfp4_e2m1_rounding_at_unit_scale():
    """Tensor amax 2688 makes S = 1, and a block with amax 6 gets scale 1, so
    its elements are rounded to E2M1 as they are: a grid over [-8, 8] with
    every midpoint."""
    fq = require_cuda()
    mags = [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    vals = sorted(set(np.linspace(-8, 8, 161).tolist() + [(a + b) / 2 for a, b in zip(mags, mags[1:])]
                      + [-(a + b) / 2 for a, b in zip(mags, mags[1:])]))
    n = -(-len(vals) // 15)
    x = np.zeros((n + 1, 16), np.float32)
    for i in range(n):
        chunk = vals[15 * i:15 * i + 15]
        x[i, :len(chunk)] = chunk
        x[i, 15] = 6.0
    x[n, 0] = 2688.0
    ref = _check(fq, x)
    assert ref["S"] == 1.0


def test_nvfp4_special_blocks():
    """Zero blocks, a NaN block (scale code NaN, zero codes), an Inf block
    (saturates), and blocks far below the tensor amax (scale underflows)."""
    fq = require_cuda()
    rng = np.random.default_rng(63)
    x = rng.standard_normal((16, 64)).astype(np.float32)
    x[0, :16] = 0.0
    x[1, 20] = np.nan
    x[2, 40] = np.inf
    x[3, :16] *= 1e-30
    x[4, 0] = 1e30
    _check(fq, x)
    _check(fq, synth.to_bf16_bits(np.where(np.isinf(x), 3e38, x).astype(np.float32)))


def test_nvfp4_activation_4096():
    fq = require_cuda()
    _check(fq, synth.config2(4096, 4096, seed=2))
    fq.check_device()
