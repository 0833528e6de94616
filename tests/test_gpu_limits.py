"""Limits: the largest group count the library takes, and a tensor of more
than 2^32 elements (64-bit indexing), against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import dev, host, require_cuda

pytestmark = pytest.mark.gpu

G_MAX = 4096


def _offsets(rows, G, seed):
    counts = np.random.default_rng(seed).multinomial(rows, [1.0 / G] * G)
    return np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)


def test_mx_max_groups():
    fq = require_cuda()
    rows, cols = 20000, 256
    x = synth.student_t(rows, cols, 4.0, seed=7)
    offs = _offsets(rows, G_MAX, 1)
    T = oracle.mx_col_blocks(rows, offs)
    ld = (T + 15) // 16 * 16
    r = fq.mxfp8_quantize(dev(x), fq.E4M3, fq.BOTH, group_offsets=list(offs), s_col_ld=ld)
    ref = oracle.mx_quantize(x, oracle.E4M3, 3, offsets=offs, s_col_ld=ld)
    for k in ("q_row", "s_row", "q_col"):
        np.testing.assert_array_equal(host(r[k]), ref[k], err_msg=k)
    np.testing.assert_array_equal(host(r["s_col"])[:, :T], ref["s_col"][:, :T])


def test_current_scaling_max_groups():
    fq = require_cuda()
    rows, cols = 20000, 256
    x = synth.student_t(rows, cols, 4.0, seed=8)
    offs = _offsets(rows, G_MAX, 2)
    c = fq.fp8q_cast_per_tensor(dev(x), fq.E4M3, group_offsets=list(offs))
    ref = oracle.current_scaling(x, oracle.E4M3, offsets=offs)
    np.testing.assert_array_equal(host(c["q"]).reshape(-1), ref["q"])
    np.testing.assert_array_equal(host(c["amax"]).view(np.uint32), ref["amax"].view(np.uint32))
    np.testing.assert_array_equal(host(c["scale"]).view(np.uint32), ref["scale"].view(np.uint32))


def test_dequant_columnwise_max_groups():
    fq = require_cuda()
    rows, cols = 20000, 64
    offs = _offsets(rows, G_MAX, 3)
    T = oracle.mx_col_blocks(rows, offs)
    rng = np.random.default_rng(9)
    q = rng.integers(0, 256, size=(cols, rows), dtype=np.uint64).astype(np.uint8)
    s = rng.integers(100, 150, size=(cols, T), dtype=np.uint64).astype(np.uint8)
    y = fq.mxfp8_dequantize(dev(q), dev(s), rows, cols, fq.E4M3, fq.COL, group_offsets=list(offs))
    want = oracle.mx_dequantize(q, s, oracle.E4M3, 2, rows, cols, offsets=offs)
    np.testing.assert_array_equal(host(y.view(torch.int16)).view(np.uint16), want)


@pytest.mark.slow
def test_more_than_2_32_elements():
    """33024 x 131072 BF16 (4.33e9 elements): a tiled random block with the
    largest magnitude planted in the very last element, beyond element 2^32.
    amax and scale over the whole tensor; codes checked on the last rows and
    on the last columnwise block."""
    fq = require_cuda()
    rows, cols = 33024, 131072
    assert rows * cols > 2 ** 32
    block = synth.normal_outliers(64, cols, seed=10, std=1.0, p=0.001, factor=100.0)
    x = np.tile(block, (rows // 64, 1))
    big = synth.to_bf16_bits(np.array([-3.0e4], np.float32))[0]
    x[-1, -1] = big
    xd = dev(x)

    amax_bits = max(oracle.amax_bits(block), int(big & 0x7FFF) << 16)
    a = fq.fp8q_amax(xd)
    assert int(host(a).view(np.uint32)[0]) == amax_bits

    c = fq.fp8q_cast_per_tensor(xd, fq.E4M3)
    s, _ = oracle.per_tensor_scale(amax_bits, oracle.E4M3, 0)
    assert host(c["scale"]).view(np.uint32)[0] == np.float32(s).view(np.uint32)
    tail = np.ascontiguousarray(x[-2:])
    q_tail, _ = oracle.cast(tail, s, oracle.E4M3)
    np.testing.assert_array_equal(host(c["q"][-2:]).reshape(-1), q_tail)
    del c

    r = fq.mxfp8_quantize(xd, fq.E4M3, fq.BOTH)
    ref_rows = oracle.mx_quantize(tail, oracle.E4M3, 1)
    np.testing.assert_array_equal(host(r["q_row"][-2:]), ref_rows["q_row"])
    np.testing.assert_array_equal(host(r["s_row"][-2:]), ref_rows["s_row"])
    corner = np.ascontiguousarray(x[rows - 32:, cols - 64:])
    ref_cols = oracle.mx_quantize(corner, oracle.E4M3, 2)
    np.testing.assert_array_equal(host(r["q_col"][cols - 64:, rows - 32:]), ref_cols["q_col"])
    np.testing.assert_array_equal(host(r["s_col"][cols - 64:, -1:]), ref_cols["s_col"])
    fq.check_device()
