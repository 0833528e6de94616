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


# ---------------------------------------------------------------------------
# the MX quantizers writing their scales straight into the block layout
# ---------------------------------------------------------------------------
def _moe_offsets(rows, G, seed):
    counts = np.random.default_rng(seed).multinomial(rows, [1.0 / G] * G)
    return [0] + [int(v) for v in np.cumsum(counts)]


FUSED = [
    # name, make x, fmt, offsets, rule, count saturation
    ("256x512, no padding", lambda: synth.config2(256, 512, seed=93), 0, None, 0, False),
    ("300x320, padded rows and columns", lambda: synth.config2(300, 320, seed=94), 1, None, 0, False),
    ("fp32 200x256", lambda: synth.f32_tensor(200, 256, seed=95), 0, None, 0, False),
    ("grouped 1600x320, bands", lambda: synth.student_t(1600, 320, 4.0, seed=96), 0,
     [0, 0, 1, 32, 65, 65, 98, 131, 163, 200, 201, 511, 512, 513, 600, 1023, 1024, 1025, 1056, 1100, 1536, 1537,
      1599, 1600], 0, False),
    ("grouped 2048x512 on 128-row groups, no padding", lambda: synth.student_t(2048, 512, 4.0, seed=97), 0,
     [0, 128, 128, 640, 1024, 2048], 0, False),
    ("64 experts 8192x512", lambda: synth.student_t(8192, 512, 4.0, seed=98), 0, _moe_offsets(8192, 64, 98), 0,
     False),
    ("grouped OCP rule with counts", lambda: synth.config2(1024, 256, seed=99), 0, [0, 300, 301, 777, 1024], 1,
     True),
    ("grouped 300 rows (unit kernel)", lambda: synth.student_t(300, 256, 4.0, seed=100), 1, [0, 45, 46, 130, 300],
     0, False),
]


@pytest.mark.parametrize("case", FUSED, ids=[c[0] for c in FUSED])
def test_quantizer_writes_mma_layout(case):
    """mxfp8_quantize_ex in the 128 x 4 layout: codes as in the row-major call,
    scales equal to the oracle's layout of the oracle's own scales, every byte
    of the canary-filled buffers written (padding 0)."""
    fq = require_cuda()
    _, make, fmt, offsets, rule, count = case
    x = make()
    rows, cols = x.shape
    off_np = None if offsets is None else np.array(offsets)
    T = oracle.mx_col_blocks(rows, off_np)
    gs_row = Guarded((fq.mxfp8_mma_scale_bytes(rows, cols // 32),))
    gs_col = Guarded((fq.mxfp8_mma_scale_bytes(cols, T),))
    for g in (gs_row, gs_col):
        g.t.fill_(0xA5)
    r = fq.mxfp8_quantize(dev(x), fmt, fq.BOTH, group_offsets=offsets, s_col_ld=T, rule=rule,
                          count_saturation=count, scale_layout=fq.SCALES_MMA,
                          out={"s_row": gs_row.t, "s_col": gs_col.t})
    torch.cuda.synchronize()
    gs_row.check()
    gs_col.check()
    orc_rule = oracle.MX_RULE_OCP if rule == fq.RULE_OCP else oracle.MX_RULE_UP
    ref = oracle.mx_quantize_rule(x, fmt, 3, orc_rule, offsets=off_np) if count else \
        oracle.mx_quantize(x, fmt, 3, offsets=off_np)
    np.testing.assert_array_equal(host(r["q_row"]), ref["q_row"])
    np.testing.assert_array_equal(host(r["q_col"]), ref["q_col"])
    np.testing.assert_array_equal(host(gs_row.t), oracle.mma_scale_layout(ref["s_row"]))
    np.testing.assert_array_equal(host(gs_col.t), oracle.mma_scale_layout(ref["s_col"], T))
    if count:
        assert host(r["sat"]).tolist() == ref["sat"]


def test_mma_layout_refuses_padded_column_count():
    """Without groups the column-block count is known: another s_col_ld is refused."""
    fq = require_cuda()
    x = dev(synth.config2(64, 64, seed=101))
    with pytest.raises(fq.Fp8qError):
        fq.mxfp8_quantize(x, fq.E4M3, fq.BOTH, s_col_ld=3, scale_layout=fq.SCALES_MMA)
