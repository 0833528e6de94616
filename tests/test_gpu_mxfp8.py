"""GPU parity: MXFP8 rowwise / columnwise / grouped quantization against the
oracle, bit for bit (element codes and E8M0 scale bytes)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import Guarded, bf16_to_f32, dev, host, require_cuda

pytestmark = pytest.mark.gpu
FMTS = [oracle.E4M3, oracle.E5M2]


@pytest.fixture(scope="module")
def fq():
    return require_cuda()


def run_mx(fq, x, fmt, direction=3, offsets=None, s_col_ld=None):
    rows, cols = x.shape
    T = oracle.mx_col_blocks(rows, None if offsets is None else np.array(offsets))
    ld = T if s_col_ld is None else s_col_ld
    out = {}
    guards = []
    if direction & 1:
        g1, g2 = Guarded((rows, cols)), Guarded((rows, cols // 32))
        out["q_row"], out["s_row"] = g1.t, g2.t
        guards += [g1, g2]
    if direction & 2:
        g3, g4 = Guarded((cols, rows)), Guarded((cols, ld))
        out["q_col"], out["s_col"] = g3.t, g4.t
        guards += [g3, g4]
    off = None if offsets is None else torch.tensor(offsets, dtype=torch.int64, device="cuda")
    r = fq.mxfp8_quantize(dev(x), fmt, direction, group_offsets=off, s_col_ld=ld, out=out)
    torch.cuda.synchronize()
    for g in guards:
        g.check()
    res = {k: (host(v) if isinstance(v, torch.Tensor) else v) for k, v in r.items()}
    res["T"] = T
    return res


def check_mx(fq, x, fmt, direction=3, offsets=None, s_col_ld=None):
    got = run_mx(fq, x, fmt, direction, offsets, s_col_ld)
    ref = oracle.mx_quantize(x, fmt, direction, offsets=None if offsets is None else np.array(offsets),
                             s_col_ld=s_col_ld)
    if direction & 1:
        np.testing.assert_array_equal(got["s_row"], ref["s_row"])
        np.testing.assert_array_equal(got["q_row"], ref["q_row"])
    if direction & 2:
        T = got["T"]
        np.testing.assert_array_equal(got["s_col"][:, :T], ref["s_col"][:, :T])
        np.testing.assert_array_equal(got["q_col"], ref["q_col"])
        if s_col_ld is not None and s_col_ld > T:  # padding columns untouched
            assert (got["s_col"][:, T:] == 0xA5).all()
    return got


# ---------------------------------------------------------------------------
# exhaustive element path: every BF16 value under every reachable scale
# ---------------------------------------------------------------------------
def _all_values_under_every_scale(fmt):
    """Rows of 32: [destmax * 2^X, 31 BF16 values v with |v| <= destmax * 2^X].
    Over all reachable X every finite BF16 value appears under every scale
    that can apply to it."""
    destmax = oracle.fp8_max(fmt)
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = bf16_to_f32(bits)
    finite = np.isfinite(vals)
    bits, vals = bits[finite], vals[finite]
    rows = []
    for X in range(-127, 128):
        A = np.float32(destmax * 2.0 ** X)
        if not np.isfinite(A):
            break
        a_bits = synth.to_bf16_bits(np.array([A], np.float32))[0]
        assert bf16_to_f32(np.array([a_bits]))[0] == A
        sel = bits[np.abs(vals) <= A]
        pad = (-sel.size) % 31
        sel = np.concatenate([sel, np.zeros(pad, np.uint16)]).reshape(-1, 31)
        rows.append(np.concatenate([np.full((sel.shape[0], 1), a_bits, np.uint16), sel], axis=1))
    x = np.concatenate(rows)
    pad = (-x.shape[0]) % 32
    return np.concatenate([x, np.zeros((pad, 32), np.uint16)])


@pytest.mark.parametrize("fmt", FMTS)
def test_every_bf16_value_under_every_scale_rowwise(fq, fmt):
    x = _all_values_under_every_scale(fmt)
    got = check_mx(fq, x, fmt, direction=1)
    # every scale byte from -127 up to the largest finite block appears
    assert len(np.unique(got["s_row"])) > 230


@pytest.mark.parametrize("fmt", FMTS)
def test_every_bf16_value_under_every_scale_columnwise(fq, fmt):
    x = np.ascontiguousarray(_all_values_under_every_scale(fmt).T)  # 32 x R: blocks down the columns
    check_mx(fq, x, fmt, direction=2)


# ---------------------------------------------------------------------------
# random and structured tensors
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("direction", [1, 2, 3])
@pytest.mark.parametrize("shape", [(1, 32), (31, 64), (273, 512), (96, 288), (64, 800)])
def test_activation_like_bf16(fq, fmt, direction, shape):
    x = synth.config2(*shape, seed=5)
    check_mx(fq, x, fmt, direction)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("shape", [(33, 96), (200, 256), (64, 1056)])
def test_fp32_input(fq, fmt, shape):
    x = synth.f32_tensor(*shape, seed=9)
    x[0, :32] = 0.0
    x[1, 3] = np.float32(1e-42)
    check_mx(fq, x, fmt, 3)


def test_special_blocks(fq):
    x = synth.config2(64, 128, seed=11).copy()
    x[0, 0:32] = 0                      # zero block
    x[1, 0:32] = 0x8000                 # all negative zeros -> 0x00
    x[2, 5] = 0x7FC0                    # NaN block
    x[3, 40] = 0xFF80                   # -Inf block
    x[4, 0:32] = 0x0001                 # subnormal amax: X = -127
    x[5, 32:64] = 0x7F7F                # amax near the BF16 max
    x[6, 64:96] = 0xC3E0                # -448 exactly
    x[7, 96:128] = 0x43E8               # 464 > 448: X = 1
    x[32:64, 7] = 0x8000                # a column block of -0 only
    x[9, 100] = 0x7F81                  # signalling-NaN payload
    for fmt in FMTS:
        got = check_mx(fq, x, fmt, 3)
        assert got["s_row"][0, 0] == 0 and not got["q_row"][1, :32].any()
        assert got["s_row"][2, 0] == 0xFF and (got["q_row"][2, :32] == 0x7F).all()
    xf = synth.f32_tensor(64, 64, seed=12)
    xf[0, 0] = np.inf
    xf[1, 33] = np.nan
    xf[2, 0:32] = np.float32(3.4e38)
    xf[3, 0:32] = np.float32(1.4e-45)
    for fmt in FMTS:
        check_mx(fq, xf, fmt, 3)


# ---------------------------------------------------------------------------
# groups
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("fmt", FMTS)
def test_ragged_groups(fq, fmt):
    """Column blocks restart at each group; empty, 1-row, 31/33-row groups and
    offsets that leave the transposed stores unaligned."""
    rows, cols = 300, 320
    x = synth.student_t(rows, cols, 4.0, seed=13)
    offsets = [0, 0, 1, 32, 65, 65, 98, 131, 163, 200, 201, 300]
    check_mx(fq, x, fmt, 3, offsets=offsets)
    check_mx(fq, x, fmt, 2, offsets=offsets, s_col_ld=oracle.mx_col_blocks(rows, np.array(offsets)) + 5)


BAND_OFFSETS = [0, 0, 1, 32, 65, 65, 98, 131, 163, 200, 201, 511, 512, 513, 600, 1023, 1024, 1025, 1056, 1100,
                1536, 1537, 1599, 1600]


@pytest.mark.parametrize("fmt", FMTS)
def test_ragged_groups_aligned_rows(fq, fmt):
    """rows % 32 == 0 (the kernel that walks 512-row bands): empty, 1-row and
    31/33-row groups, groups that straddle a band edge and groups that end
    exactly on one, both directions and the columnwise copy alone with an
    odd scale stride."""
    rows, cols = 1600, 320
    x = synth.student_t(rows, cols, 4.0, seed=23)
    check_mx(fq, x, fmt, 3, offsets=BAND_OFFSETS)
    T = oracle.mx_col_blocks(rows, np.array(BAND_OFFSETS))
    check_mx(fq, x, fmt, 2, offsets=BAND_OFFSETS, s_col_ld=T + 5)


def test_grouped_rowwise_only_ignores_groups(fq):
    """The rowwise copy does not depend on the groups."""
    x = synth.config2(1600, 256, seed=24)
    got = check_mx(fq, x, oracle.E4M3, 1, offsets=BAND_OFFSETS)
    ref = oracle.mx_quantize(x, oracle.E4M3, 1)
    np.testing.assert_array_equal(got["q_row"], ref["q_row"])


def test_one_group_covering_all_rows(fq):
    """Explicit offsets [0, rows] give the ungrouped result."""
    x = synth.config2(2048, 512, seed=25)
    got = check_mx(fq, x, oracle.E5M2, 3, offsets=[0, 2048])
    ref = oracle.mx_quantize(x, oracle.E5M2, 3)
    np.testing.assert_array_equal(got["q_col"], ref["q_col"])


def test_grouped_special_blocks(fq):
    """Zero, -0, NaN, Inf and subnormal column blocks inside ragged groups,
    including blocks that straddle a band edge and a group's short last block."""
    rows, cols = 1056, 256
    x = synth.student_t(rows, cols, 4.0, seed=26).copy()
    offsets = [0, 500, 530, 1000, 1056]
    x[500:530, 0] = 0                    # a whole 30-row group, zero in column 0
    x[500:530, 1] = 0x8000               # ... and -0 in column 1
    x[510, 2] = 0x7FC0                   # NaN in a short group
    x[520, 3] = 0xFF80                   # -Inf
    x[0:32, 4] = 0x0001                  # subnormal amax
    x[490:522, 5] = 0                    # crosses a group boundary
    x[507:515, 6] = 0x7F81               # NaN rows straddling the 512 band edge
    x[1040, 7] = 0x7F80                  # +Inf in the last group's short block
    x[996:1000, 8] = 0x43E8              # 464 > 448 at a group's end
    for fmt in FMTS:
        check_mx(fq, x, fmt, 3, offsets=offsets)


def test_grouped_unaligned_transposed_output(fq):
    """A q_col that is 16 but not 32-byte aligned takes the unit kernel."""
    rows, cols = 1600, 256
    x = synth.student_t(rows, cols, 4.0, seed=27)
    T = oracle.mx_col_blocks(rows, np.array(BAND_OFFSETS))
    raw = torch.full((cols * rows + 64,), 0xA5, dtype=torch.uint8, device="cuda")
    base = (32 - raw.data_ptr() % 32) % 32 + 16
    q_col = raw[base:base + cols * rows].view(cols, rows)
    assert q_col.data_ptr() % 32 == 16
    out = {"q_col": q_col, "s_col": torch.empty((cols, T), dtype=torch.uint8, device="cuda")}
    off = torch.tensor(BAND_OFFSETS, dtype=torch.int64, device="cuda")
    r = fq.mxfp8_quantize(dev(x), oracle.E4M3, 2, group_offsets=off, s_col_ld=T, out=out)
    ref = oracle.mx_quantize(x, oracle.E4M3, 2, offsets=np.array(BAND_OFFSETS))
    np.testing.assert_array_equal(host(r["q_col"]), ref["q_col"])
    np.testing.assert_array_equal(host(r["s_col"]), ref["s_col"][:, :T])
    rawh = host(raw)
    assert (rawh[:base] == 0xA5).all() and (rawh[base + cols * rows:] == 0xA5).all()


def test_moe_groups_fp32(fq):
    x = synth.f32_tensor(517, 96, seed=17)
    check_mx(fq, x, oracle.E5M2, 3, offsets=[0, 17, 17, 300, 517])


def test_moe_routing_64_experts(fq):
    """64 experts, multinomial token counts (8192 tokens x 512 hidden)."""
    x = synth.student_t(8192, 512, 4.0, seed=19)
    offs = list(synth.moe_offsets(8192, 64, seed=19))
    check_mx(fq, x, oracle.E4M3, 3, offsets=offs)


# ---------------------------------------------------------------------------
# full-size workloads
# ---------------------------------------------------------------------------
def test_activation_4096x4096_full(fq):
    """The MXFP8 workload: 4096x4096 BF16 activation, both directions, E4M3."""
    check_mx(fq, synth.config2(), oracle.E4M3, 3)
