"""MXFP8 under both scale rules, with saturation counts, against the oracle
(codes, scale bytes and the counts of both copies, bit for bit)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import dev, host, require_cuda

pytestmark = pytest.mark.gpu

RULES = {"up": (0, oracle.MX_RULE_UP), "ocp": (1, oracle.MX_RULE_OCP)}


def _check(fq, x, fmt, rule, offsets=None):
    lib_rule, orc_rule = RULES[rule]
    rows, cols = x.shape
    off = None if offsets is None else list(offsets)
    T = oracle.mx_col_blocks(rows, None if offsets is None else np.array(offsets))
    ld = (T + 15) // 16 * 16 if offsets is not None else T
    r = fq.mxfp8_quantize(dev(x), fmt, fq.BOTH, group_offsets=off, s_col_ld=ld, rule=lib_rule,
                          count_saturation=True)
    ref = oracle.mx_quantize_rule(x, fmt, 3, orc_rule, offsets=None if offsets is None else np.array(offsets),
                                  s_col_ld=ld)
    for k in ("q_row", "s_row", "q_col"):
        np.testing.assert_array_equal(host(r[k]), ref[k], err_msg=k)
    np.testing.assert_array_equal(host(r["s_col"])[:, :T], ref["s_col"][:, :T])
    assert host(r["sat"]).tolist() == ref["sat"]
    return ref["sat"]


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("rule", ["up", "ocp"])
def test_bf16_activation_rules(fmt, rule):
    fq = require_cuda()
    x = synth.config2(256, 512, seed=12)
    sat = _check(fq, x, fmt, rule)
    if rule == "up":
        assert sat == [0, 0]


@pytest.mark.parametrize("rule", ["up", "ocp"])
def test_grouped_ragged_rules(rule):
    fq = require_cuda()
    x = synth.student_t(300, 256, 4.0, seed=13)
    _check(fq, x, 0, rule, offsets=[0, 0, 45, 46, 130, 300])


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("rule", ["up", "ocp"])
def test_grouped_band_rules(fmt, rule):
    """rows % 32 == 0 (512-row bands): groups straddling and ending on band
    edges; saturated elements of a block loaded by two bands count once."""
    fq = require_cuda()
    x = synth.config2(1600, 256, seed=16)
    _check(fq, x, fmt, rule, offsets=[0, 0, 45, 46, 130, 500, 511, 512, 530, 1024, 1025, 1599, 1600])


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("rule", ["up", "ocp"])
def test_fp32_input_rules(fmt, rule):
    fq = require_cuda()
    rng = np.random.default_rng(14)
    x = (rng.standard_normal((96, 256)) * np.exp(rng.standard_normal((96, 1)) * 4)).astype(np.float32)
    _check(fq, x, fmt, rule)


def test_blocks_built_to_saturate():
    """Blocks whose amax sits just above the maximum times a power of two:
    the OCP rule clamps them, the round-up rule does not."""
    fq = require_cuda()
    rng = np.random.default_rng(15)
    x = rng.standard_normal((64, 128)).astype(np.float32)
    x[:, ::32] = 480.0 * 2.0 ** rng.integers(-10, 10, size=(64, 4))
    x[:, 1::32] = -470.0 * 2.0 ** rng.integers(-10, 10, size=(64, 4))
    xb = synth.to_bf16_bits(x)
    assert _check(fq, xb, 0, "ocp")[0] > 0
    assert _check(fq, xb, 0, "up") == [0, 0]


def test_activation_4096_ocp_counts():
    """The 4096x4096 activation: codes and both saturation counts under the
    OCP rule."""
    fq = require_cuda()
    x = synth.config2(4096, 4096, seed=2)
    sat = _check(fq, x, 0, "ocp")
    assert sat[0] > 0 and sat[1] > 0
