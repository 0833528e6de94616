"""Dequantization kernels against the oracle, bit for bit.

Codes and scale bytes are drawn on the host (or enumerated), so neither
side's input comes from the other.  Outputs sit in guarded buffers that
catch stray writes.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import Guarded, dev, host, require_cuda

pytestmark = pytest.mark.gpu

OUT = {0: torch.bfloat16, 1: torch.float32}
RAW = {0: torch.int16, 1: torch.int32}
NPU = {0: np.uint16, 1: np.uint32}


def _bits(t: torch.Tensor, out_dt: int) -> np.ndarray:
    return host(t.view(RAW[out_dt])).view(NPU[out_dt])


def _mx(fq, q, s, rows, cols, fmt, direction, out_dt, offsets=None):
    y = Guarded(q.shape, OUT[out_dt])
    off = None if offsets is None else list(offsets)
    fq.mxfp8_dequantize(dev(q), dev(s), rows, cols, fmt, direction, group_offsets=off, out_dtype=OUT[out_dt],
                        out=y.t)
    torch.cuda.synchronize()
    y.check()
    return _bits(y.t, out_dt)


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("out_dt", [0, 1])
def test_mx_every_code_under_every_scale_byte(fmt, out_dt):
    """All 256 codes x all 256 scale bytes (0xFF included), rowwise layout."""
    fq = require_cuda()
    q = np.tile(np.arange(256, dtype=np.uint8).reshape(8, 32), (256, 1))      # [2048, 32]
    s = np.repeat(np.arange(256, dtype=np.uint8), 8).reshape(2048, 1)
    got = _mx(fq, q, s, 2048, 32, fmt, 1, out_dt)
    want = oracle.mx_dequantize(q, s, fmt, 1, 2048, 32, out_dt=out_dt)
    np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("out_dt", [0, 1])
@pytest.mark.parametrize("rows", [150, 4096])
def test_mx_columnwise_ragged_groups(fmt, out_dt, rows):
    """Columnwise copy with ragged group offsets (empty, 1-row and odd
    groups); rows = 150 puts vectors across column ends."""
    fq = require_cuda()
    rng = np.random.default_rng(31 + rows)
    cols = 96
    cuts = np.sort(rng.integers(0, rows + 1, size=6))
    offs = np.concatenate([[0], cuts[:2], [cuts[1]], [cuts[1] + 1 if cuts[1] < rows else rows], cuts[2:], [rows]])
    offs = np.maximum.accumulate(np.minimum(offs, rows)).astype(np.int64)
    T = oracle.mx_col_blocks(rows, offs)
    s_ld = T + 3
    q = rng.integers(0, 256, size=(cols, rows), dtype=np.uint64).astype(np.uint8)
    s = rng.integers(90, 160, size=(cols, s_ld), dtype=np.uint64).astype(np.uint8)
    s[:, ::17] = 0xFF
    got = _mx(fq, q, s, rows, cols, fmt, 2, out_dt, offsets=offs)
    want = oracle.mx_dequantize(q, s, fmt, 2, rows, cols, out_dt=out_dt, offsets=offs)
    np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("fmt", [0, 1])
def test_mx_rowwise_large(fmt):
    """Several grid-stride rounds: 4096 x 4096 random codes and bytes."""
    fq = require_cuda()
    rng = np.random.default_rng(41)
    q = rng.integers(0, 256, size=(4096, 4096), dtype=np.uint64).astype(np.uint8)
    s = rng.integers(60, 200, size=(4096, 128), dtype=np.uint64).astype(np.uint8)
    got = _mx(fq, q, s, 4096, 4096, fmt, 1, 0)
    want = oracle.mx_dequantize(q, s, fmt, 1, 4096, 4096, out_dt=0)
    np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("out_dt", [0, 1])
@pytest.mark.parametrize("shape", [(333, 100), (64, 256), (1, 7), (4096, 2048)])
def test_per_tensor_groups(fmt, out_dt, shape):
    """Per-group scale_inv (including 0, tiny, huge and Inf), ragged tails
    (n % 16 != 0) and empty groups."""
    fq = require_cuda()
    rows, cols = shape
    rng = np.random.default_rng(rows * 7 + cols)
    q = rng.integers(0, 256, size=shape, dtype=np.uint64).astype(np.uint8)
    offs = np.unique(np.concatenate([[0, rows], rng.integers(0, rows + 1, size=4)])).astype(np.int64)
    offs = np.concatenate([offs[:1], offs]) if rows > 1 else offs  # an empty first group
    G = len(offs) - 1
    si = np.array([1.0 / 448, 3.1e-5, 0.0, 2.0 ** 120, np.inf, 1.0][:G] + [0.75] * max(0, G - 6), np.float32)
    y = Guarded(shape, OUT[out_dt])
    fq.fp8q_dequantize_per_tensor(dev(q), dev(si), fmt, group_offsets=list(offs), out_dtype=OUT[out_dt], out=y.t)
    torch.cuda.synchronize()
    y.check()
    want = oracle.dequant_per_tensor(q, fmt, si, out_dt=out_dt, offsets=offs)
    np.testing.assert_array_equal(_bits(y.t, out_dt), want)


def test_mx_quantize_then_dequantize_host_codes():
    """The oracle's own MX codes of a config-2-like tensor, dequantized on the
    GPU in both layouts, equal the oracle's dequantization."""
    fq = require_cuda()
    import synth
    x = synth.config2(256, 512, seed=9)
    r = oracle.mx_quantize(x, 0, 3)
    for direction, qk, sk in ((1, "q_row", "s_row"), (2, "q_col", "s_col")):
        got = _mx(fq, r[qk], r[sk], 256, 512, 0, direction, 0)
        want = oracle.mx_dequantize(r[qk], r[sk], 0, direction, 256, 512, out_dt=0)
        np.testing.assert_array_equal(got, want)
