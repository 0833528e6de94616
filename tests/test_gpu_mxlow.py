"""MXFP4 (E2M1) and MXFP6 (E2M3, E3M2) against the oracle, bit for bit:
codes, scale bytes and saturation counts of both copies, under both scale
rules."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import Guarded, dev, host, require_cuda

pytestmark = pytest.mark.gpu

ELEMS = {"e2m1": oracle.E2M1, "e2m3": oracle.E2M3, "e3m2": oracle.E3M2}


def _check(fq, x, elem, rule, direction=3):
    rows, cols = x.shape
    fp4 = elem == oracle.E2M1
    shapes = {"q_row": (rows, cols // 2 if fp4 else cols), "s_row": (rows, cols // 32),
              "q_col": (cols, rows // 2 if fp4 else rows), "s_col": (cols, (rows + 31) // 32)}
    g = {k: Guarded(v) for k, v in shapes.items()}
    out = {k: v.t for k, v in g.items()}
    r = fq.mx_quantize_fp4_fp6(dev(x), elem, direction, rule, count_saturation=True, out=out)
    torch.cuda.synchronize()
    for v in g.values():
        v.check()
    ref = oracle.mxlp_quantize(x, elem, direction, rule)
    keys = ([("q_row", "s_row")] if direction & 1 else []) + ([("q_col", "s_col")] if direction & 2 else [])
    for qk, sk in keys:
        np.testing.assert_array_equal(host(r[sk]), ref[sk], err_msg=sk)
        np.testing.assert_array_equal(host(r[qk]), ref[qk], err_msg=qk)
    assert host(r["sat"]).tolist() == ref["sat"]
    return ref["sat"]


@pytest.mark.parametrize("elem", ["e2m1", "e2m3", "e3m2"])
@pytest.mark.parametrize("rule", [0, 1])
def test_bf16_activation(elem, rule):
    fq = require_cuda()
    sat = _check(fq, synth.config2(256, 1024, seed=41), ELEMS[elem], rule)
    if rule == 0:
        assert sat == [0, 0]


@pytest.mark.parametrize("elem", ["e2m1", "e2m3", "e3m2"])
@pytest.mark.parametrize("shape", [(40, 96), (300, 544), (2, 32), (64, 32)])
def test_ragged_shapes(elem, shape):
    """rows % 32 != 0 (a short last column block), column tiles that end
    inside a warp (cols % 64 == 32), and tiny tensors."""
    fq = require_cuda()
    _check(fq, synth.student_t(*shape, 3.0, seed=42), ELEMS[elem], 1)


@pytest.mark.parametrize("elem", ["e2m1", "e2m3", "e3m2"])
def test_fp32_wide_range_and_specials(elem):
    """FP32 rows over 2^-140 .. 2^120 (subnormal inputs, clamped scales),
    zero, -0, Inf and NaN blocks, values on every rounding midpoint."""
    fq = require_cuda()
    rng = np.random.default_rng(43)
    fmt = ELEMS[elem]
    x = (rng.standard_normal((96, 256)) * 2.0 ** rng.integers(-140, 120, size=(96, 1))).astype(np.float32)
    x[3, :] = 0.0
    x[4, 32:64] = -0.0
    x[5, 7] = np.inf
    x[6, 40] = -np.inf
    x[7, 100] = np.nan
    x[40:48, 9] = np.nan
    n = 8 if fmt == oracle.E2M1 else 32
    mags = [oracle.lp_value(fmt, c) for c in range(n)]
    mids = np.array([(a + b) / 2 for a, b in zip(mags, mags[1:])], np.float32)
    x[10, :mids.size] = mids
    x[10, 31] = mags[-1]            # the block's scale is 2^0: midpoints land exactly
    x[11, :mids.size] = -mids
    x[11, 31] = -mags[-1]
    for d in (1, 2, 3):
        _check(fq, x, fmt, 0, d)
        _check(fq, x, fmt, 1, d)


def test_saturation_under_ocp():
    """Blocks whose amax sits just under 2^k * 2 (above destmax * 2^X under
    the OCP rule): saturated counts match the oracle and are nonzero."""
    fq = require_cuda()
    rng = np.random.default_rng(44)
    x = rng.standard_normal((64, 128)).astype(np.float32)
    x[:, ::32] = 7.9 * 2.0 ** rng.integers(-10, 10, size=(64, 4))
    for elem in ELEMS.values():
        assert _check(fq, x, elem, 1)[0] > 0


def test_activation_8192_both_copies():
    """The 8192 x 8192 BF16 activation, MXFP4 and MXFP6 (E2M3), both copies
    in one call, round-up rule: every code and scale byte."""
    fq = require_cuda()
    x = synth.config2(8192, 8192, seed=0)
    for elem in (oracle.E2M1, oracle.E2M3):
        _check(fq, x, elem, 0)


@pytest.mark.parametrize("elem", ["e2m1", "e2m3", "e3m2"])
def test_bf16_specials_each_direction(elem):
    """BF16 input (the TMA kernel): rows over 2^-133 .. 2^120 (subnormal
    BF16 inputs, clamped scales), zero, -0, Inf and NaN blocks, values near
    every rounding midpoint; each direction alone and both, both rules."""
    fq = require_cuda()
    rng = np.random.default_rng(45)
    fmt = ELEMS[elem]
    x = (rng.standard_normal((96, 320)) * 2.0 ** rng.integers(-133, 120, size=(96, 1))).astype(np.float32)
    x[3, :] = 0.0
    x[4, 32:64] = -0.0
    x[5, 7] = np.inf
    x[6, 40] = -np.inf
    x[7, 100] = np.nan
    x[40:48, 9] = np.nan
    n = 8 if fmt == oracle.E2M1 else 32
    mags = [oracle.lp_value(fmt, c) for c in range(n)]
    mids = np.array([(a + b) / 2 for a, b in zip(mags, mags[1:])], np.float32)
    x[10, :mids.size] = mids
    x[10, 31] = mags[-1]
    x[11, :mids.size] = -mids
    x[11, 31] = -mags[-1]
    xb = synth.to_bf16_bits(x)
    for d in (1, 2, 3):
        _check(fq, xb, fmt, 0, d)
        _check(fq, xb, fmt, 1, d)
