"""Quantization-error statistics (SQNR, zero-rate) against the oracle.

The quantized copies are made by the oracle, or drawn on the host (random
codes and scale bytes, NaN and overflow included), so neither side's input
comes from the other.  Counts must match exactly.  The two sums must match
to RTOL: the kernel sums each chunk of 32 elements in FP32 with fused
multiply-adds, which is within 33 units of 2^-24 of the exact chunk sum
(32 roundings of a sum of non-negative terms, plus the rounding of e = x -
xh when it is inexact, which doubles in e^2: 35 * 2^-24 ~ 2.1e-6), then adds
chunk sums in FP64; the oracle sums in FP64 throughout (error ~1e-16 * n).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import dev, require_cuda

pytestmark = pytest.mark.gpu

RTOL = 2.5e-6


def _gpu(fq, t):
    torch.cuda.synchronize()
    return fq.qstats_dict(t)


# SQNR: relative errors of RTOL in the two sums move 10 log10(signal/noise)
# by at most 10 / ln(10) * 2 * RTOL dB.
SQNR_TOL_DB = 10.0 / np.log(10.0) * 2 * RTOL


def _same(got, want):
    for k in ("n", "n_zero", "n_flushed", "n_nonfinite"):
        assert got[k] == want[k], (k, got, want)
    for k in ("signal", "noise"):
        assert got[k] == pytest.approx(want[k], rel=RTOL, abs=0.0), (k, got, want)
    # the SQNR and zero-rate the library computes on the device
    w_db = oracle.sqnr_db(want)
    if np.isfinite(w_db):
        assert abs(got["sqnr_db"] - w_db) <= SQNR_TOL_DB, (got["sqnr_db"], w_db)
    else:
        assert got["sqnr_db"] == w_db or (np.isnan(w_db) and np.isnan(got["sqnr_db"])), (got["sqnr_db"], w_db)
    assert got["zero_rate"] == oracle.zero_rate(want), (got["zero_rate"], oracle.zero_rate(want))


def _mx_case(fq, x, fmt, offsets=None):
    off = None if offsets is None else np.asarray(offsets, np.int64)
    T = oracle.mx_col_blocks(x.shape[0], off)
    ld = (T + 15) // 16 * 16 if off is not None else T
    r = oracle.mx_quantize(x, fmt, 3, offsets=off, s_col_ld=ld)
    xd = dev(x)
    for d, (qq, ss) in ((1, ("q_row", "s_row")), (2, ("q_col", "s_col"))):
        want = oracle.qstats_mx(x, r[qq], r[ss], fmt, d, offsets=off)
        got = _gpu(fq, fq.mxfp8_qstats(xd, dev(r[qq]), dev(r[ss]), fmt, d,
                                       group_offsets=None if off is None else list(off)))
        _same(got, want)


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("shape", [(256, 512), (300, 256), (37, 96)])
def test_mx_bf16(fmt, shape):
    fq = require_cuda()
    _mx_case(fq, synth.config2(*shape, seed=21), fmt)


@pytest.mark.parametrize("fmt", [0, 1])
def test_mx_bf16_columnwise_edges(fmt):
    """BF16 without groups and rows % 32 == 0 (the TMA-fed columnwise
    kernel): a partial last 256-column strip (800 columns), a last unit of
    two blocks (320 rows), rows over 2^-80 .. 2^40 (tiny chunks take the
    FP64 path), and zero, -0, Inf and NaN chunks."""
    fq = require_cuda()
    rng = np.random.default_rng(31)
    x = (rng.standard_normal((320, 800)) * 2.0 ** rng.integers(-80, 40, size=(320, 1))).astype(np.float32)
    x[0:32, 5] = 0.0
    x[32:64, 7] = -0.0
    x[70, 9] = np.inf
    x[100, 11] = np.nan
    _mx_case(fq, synth.to_bf16_bits(x), fmt)


@pytest.mark.parametrize("fmt", [0, 1])
def test_mx_fp32_wide_range(fmt):
    """FP32 rows spread over 2^-40 .. 2^40 (tiny rows take the FP64 path)."""
    fq = require_cuda()
    rng = np.random.default_rng(22)
    x = (rng.standard_normal((160, 256)) * 2.0 ** rng.integers(-80, 40, size=(160, 1))).astype(np.float32)
    _mx_case(fq, x, fmt)


@pytest.mark.parametrize("offsets", [[0, 0, 45, 46, 130, 300], [0, 300], [0, 32, 64, 64, 300]])
def test_mx_grouped_columnwise(offsets):
    fq = require_cuda()
    _mx_case(fq, synth.student_t(300, 256, 4.0, seed=23), 0, offsets)


def _pt_case(fq, x, fmt, offsets=None):
    off = None if offsets is None else np.asarray(offsets, np.int64)
    c = oracle.current_scaling(x, fmt, offsets=off)
    want = oracle.qstats_per_tensor(x, c["q"].reshape(x.shape), fmt, c["scale_inv"], offsets=off)
    got = _gpu(fq, fq.fp8q_qstats_per_tensor(dev(x), dev(c["q"].reshape(x.shape)), torch.from_numpy(c["scale_inv"]),
                                             fmt, group_offsets=None if off is None else list(off)))
    _same(got, want)
    return got


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("shape", [(256, 512), (77, 45), (1, 31), (5, 1000)])
def test_per_tensor(fmt, shape):
    """Whole chunks, chunks across rows (cols % 32 != 0) and a ragged end."""
    fq = require_cuda()
    _pt_case(fq, synth.config2(*shape, seed=24), fmt)


@pytest.mark.parametrize("shape", [(300, 256), (301, 45)])
def test_per_tensor_grouped(shape):
    fq = require_cuda()
    x = synth.student_t(*shape, 4.0, seed=25)
    got = _pt_case(fq, x, 0, [0, 0, 45, 46, 130, shape[0]])
    assert got["n"] == x.size


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("direction", [1, 2])
def test_random_codes_and_scale_bytes(fmt, direction):
    """Arbitrary codes (NaN and Inf codes) under arbitrary scale bytes (0,
    254, 0xFF): products that overflow FP32, NaN scales, huge errors."""
    fq = require_cuda()
    rng = np.random.default_rng(26 + direction)
    rows, cols = 96, 128
    x = (rng.standard_normal((rows, cols)) * 2.0 ** rng.integers(-100, 100, size=(rows, cols))).astype(np.float32)
    x[rng.random(x.shape) < 0.01] = np.inf
    x[rng.random(x.shape) < 0.01] = np.nan
    qshape = (rows, cols) if direction == 1 else (cols, rows)
    sshape = (rows, cols // 32) if direction == 1 else (cols, (rows + 31) // 32)
    q = rng.integers(0, 256, size=qshape, dtype=np.uint64).astype(np.uint8)
    s = rng.integers(0, 256, size=sshape, dtype=np.uint64).astype(np.uint8)
    s.reshape(-1)[:3] = [0, 254, 255]
    want = oracle.qstats_mx(x, q, s, fmt, direction)
    got = _gpu(fq, fq.mxfp8_qstats(dev(x), dev(q), dev(s), fmt, direction))
    assert got["n_nonfinite"] > 0 and got["n_zero"] > 0
    _same(got, want)


def test_per_tensor_special_scales():
    """scale_inv of 0, Inf and NaN per group, and codes of every value."""
    fq = require_cuda()
    rng = np.random.default_rng(28)
    x = rng.standard_normal((64, 256)).astype(np.float32)
    q = np.tile(np.arange(256, dtype=np.uint8), (64, 1))
    off = np.array([0, 16, 32, 48, 64], np.int64)
    si = np.array([0.0, np.inf, np.nan, 0.5], np.float32)
    want = oracle.qstats_per_tensor(x, q, 0, si, offsets=off)
    got = _gpu(fq, fq.fp8q_qstats_per_tensor(dev(x), dev(q), torch.from_numpy(si), 0, group_offsets=list(off)))
    _same(got, want)


def test_tiny_and_huge_tensors():
    """All magnitudes near 1e-30 (squares below FP32's range) and near 1e30
    (squares above it): both take the FP64 path and keep full accuracy."""
    fq = require_cuda()
    rng = np.random.default_rng(29)
    for mag in (1e-30, 1e30):
        x = (rng.standard_normal((64, 128)) * mag).astype(np.float32)
        _mx_case(fq, x, 0)
        _pt_case(fq, x, 0)


def test_empty_and_exact():
    """An empty tensor gives all zeros; powers of two quantize exactly."""
    fq = require_cuda()
    got = _gpu(fq, fq.mxfp8_qstats(torch.empty((0, 64), dtype=torch.bfloat16, device="cuda"),
                                   torch.empty(0, dtype=torch.uint8, device="cuda"),
                                   torch.empty((0, 2), dtype=torch.uint8, device="cuda"), 0, 1))
    assert (got["n"], got["signal"], got["noise"]) == (0, 0.0, 0.0)
    x = (2.0 ** np.random.default_rng(30).integers(-6, 8, size=(64, 64))).astype(np.float32)
    r = oracle.mx_quantize(x, 0, 1)
    got = _gpu(fq, fq.mxfp8_qstats(dev(x), dev(r["q_row"]), dev(r["s_row"]), 0, 1))
    assert got["noise"] == 0.0 and got["sqnr_db"] == float("inf") and got["n_flushed"] == 0


def test_repeatable():
    """Two calls on the same data give the same bits."""
    fq = require_cuda()
    x = synth.config2(1024, 1024, seed=31)
    r = oracle.mx_quantize(x, 0, 2)
    xd, qd, sd = dev(x), dev(r["q_col"]), dev(r["s_col"])
    a = fq.mxfp8_qstats(xd, qd, sd, 0, 2).clone()
    b = fq.mxfp8_qstats(xd, qd, sd, 0, 2)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int64), b.view(torch.int64))


def test_activation_8192_both_copies_and_per_tensor():
    """The 8192 x 8192 BF16 activation: the library's own MX and per-tensor
    copies, each measured on the GPU, against the oracle's copies measured
    by the oracle (the quantizers are bit-exact, so the statistics agree)."""
    fq = require_cuda()
    x = synth.config2(8192, 8192, seed=0)
    xd = dev(x)
    r = fq.mxfp8_quantize(xd, fq.E4M3, fq.BOTH)
    c = fq.fp8q_cast_per_tensor(xd, fq.E4M3)
    got = {1: _gpu(fq, fq.mxfp8_qstats(xd, r["q_row"], r["s_row"], 0, 1)),
           2: _gpu(fq, fq.mxfp8_qstats(xd, r["q_col"], r["s_col"], 0, 2)),
           0: _gpu(fq, fq.fp8q_qstats_per_tensor(xd, c["q"], c["scale_inv"], 0))}
    del r, c
    ro = oracle.mx_quantize(x, 0, 3)
    _same(got[1], oracle.qstats_mx(x, ro["q_row"], ro["s_row"], 0, 1))
    _same(got[2], oracle.qstats_mx(x, ro["q_col"], ro["s_col"], 0, 2))
    del ro
    co = oracle.current_scaling(x, 0)
    _same(got[0], oracle.qstats_per_tensor(x, co["q"].reshape(x.shape), 0, co["scale_inv"]))
