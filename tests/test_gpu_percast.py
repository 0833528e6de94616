"""GPU parity: per-tensor amax, current scaling and given-scale casts against
the CPU oracle, bit for bit (codes, amax bits, scales, saturation counts)."""
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


def f32bits(a):
    return np.asarray(a, dtype=np.float32).view(np.uint32)


def run_cast(fq, x_np, fmt, margin=0, scale=None, offsets=None, want_sat=True):
    rows, cols = x_np.shape
    G = 1 if offsets is None else len(offsets) - 1
    q = Guarded((rows, cols))
    outs = [Guarded((G,), torch.float32) for _ in range(3)]
    sat = Guarded((G,), torch.int64)
    x = dev(x_np)
    off = None if offsets is None else torch.tensor(offsets, dtype=torch.int64, device="cuda")
    scale_t = None if scale is None else torch.tensor(np.asarray(scale, np.float32).reshape(-1), device="cuda")
    ws = torch.zeros(fq.fp8q_cast_workspace_bytes(G), dtype=torch.uint8, device="cuda")
    st = fq.lib().fp8q_cast_per_tensor(
        x.data_ptr(), 0 if x_np.dtype == np.uint16 else 1, rows, cols,
        None if off is None else off.data_ptr(), G, fmt, margin,
        None if scale_t is None else scale_t.data_ptr(), q.t.data_ptr(), outs[0].t.data_ptr(),
        outs[1].t.data_ptr(), outs[2].t.data_ptr(), sat.t.data_ptr() if want_sat else None,
        ws.data_ptr(), ws.numel(), torch.cuda.current_stream().cuda_stream)
    assert st == 0, fq.lib().fp8q_last_error_string()
    torch.cuda.synchronize()
    for g in [q, sat] + outs:
        g.check()
    assert int(ws.count_nonzero()) == 0, "workspace not left zero-filled"
    return {"q": host(q.t).reshape(-1), "amax": host(outs[0].t), "scale": host(outs[1].t),
            "scale_inv": host(outs[2].t), "sat": host(sat.t)}


def check_current(fq, x, fmt, margin=0, offsets=None):
    got = run_cast(fq, x, fmt, margin=margin, offsets=offsets)
    ref = oracle.current_scaling(x, fmt, margin=margin, offsets=offsets)
    np.testing.assert_array_equal(got["q"], ref["q"])
    np.testing.assert_array_equal(f32bits(got["amax"]), f32bits(ref["amax"]))
    np.testing.assert_array_equal(f32bits(got["scale"]), f32bits(ref["scale"]))
    np.testing.assert_array_equal(f32bits(got["scale_inv"]), f32bits(ref["scale_inv"]))
    np.testing.assert_array_equal(got["sat"], ref["sat"])


# ---------------------------------------------------------------------------
# exhaustive codec sweeps
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("scale", [1.0, 22400.0, 0.0173, 3.0e30, 1.0e-30, 448.0 / 7.3])
def test_all_bf16_patterns(fq, fmt, scale):
    x = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16).reshape(2048, 32)
    got = run_cast(fq, x, fmt, scale=[scale])
    ref, sat = oracle.cast(x, np.float32(scale), fmt)
    np.testing.assert_array_equal(got["q"], ref)
    assert got["sat"][0] == sat
    assert f32bits(got["scale"])[0] == f32bits([scale])[0]


@pytest.mark.parametrize("fmt", FMTS)
def test_all_fp32_patterns(fq, fmt):
    """Every one of the 2^32 FP32 patterns through the device cast (scale 1)."""
    chunk = 1 << 26
    scale = torch.ones(1, dtype=torch.float32, device="cuda")
    ws = torch.zeros(fq.fp8q_cast_workspace_bytes(1), dtype=torch.uint8, device="cuda")
    q = torch.empty(chunk, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    for first in range(0, 1 << 32, chunk):
        bits = np.arange(first, first + chunk, dtype=np.uint64).astype(np.uint32)
        x = torch.from_numpy(bits.view(np.float32)).cuda()
        st = fq.lib().fp8q_cast_per_tensor(x.data_ptr(), 1, 1, chunk, None, 1, fmt, 0, scale.data_ptr(),
                                          q.data_ptr(), None, None, None, None, ws.data_ptr(), ws.numel(),
                                          stream)
        assert st == 0
        ref = oracle.encode_f32_range(fmt, first, chunk)
        got = q.cpu().numpy()
        if not np.array_equal(got, ref):
            bad = np.nonzero(got != ref)[0][:5]
            raise AssertionError(f"fmt {fmt}: patterns {[hex(first + int(i)) for i in bad]} "
                                 f"got {got[bad]} want {ref[bad]}")


# ---------------------------------------------------------------------------
# current scaling
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("fmt", FMTS)
def test_current_scaling_1024x1024(fq, fmt):
    """The per-tensor workload: 1024x1024 BF16, N(0,1) with 0.1% x100."""
    check_current(fq, synth.config1(), fmt)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("margin", [0, 3])
def test_current_scaling_fp32(fq, fmt, margin):
    check_current(fq, synth.f32_tensor(300, 777, seed=21), fmt, margin=margin)


@pytest.mark.parametrize("shape", [(1, 1), (1, 7), (3, 5), (1, 8193), (5, 8192 * 3 + 5), (129, 64)])
def test_current_scaling_ragged_sizes(fq, shape):
    x = synth.normal_outliers(shape[0], shape[1], seed=31)
    check_current(fq, x, oracle.E4M3)
    check_current(fq, synth.f32_tensor(shape[0], shape[1], seed=32), oracle.E5M2)


def test_current_scaling_one_cluster_boundary(fq):
    """Up to 2 MB, current scaling is one thread-block cluster of 16 CTAs
    (the tensor in their shared memory, the amax exchanged between them):
    the largest such tensors in both input types, one row more, a tensor
    smaller than one 16-byte vector per CTA, and a ragged tail."""
    for rows, seed in ((256, 101), (257, 102), (255, 103)):
        check_current(fq, synth.normal_outliers(rows, 4096, seed=seed), oracle.E4M3)
    for rows, seed in ((128, 104), (129, 105)):
        check_current(fq, synth.f32_tensor(rows, 4096, seed=seed), oracle.E5M2, margin=2)
    check_current(fq, synth.normal_outliers(1, 100, seed=106), oracle.E4M3)
    check_current(fq, synth.normal_outliers(3, 1000 * 16 + 5, seed=107), oracle.E5M2)


def test_current_scaling_single_launch_boundary(fq):
    """Ungrouped current scaling takes one launch while the 32 KB slices of x
    fit one per resident CTA (4 per SM here), then two slices per CTA (the
    second staged in shared memory), and two passes beyond: the largest
    tensors of each kind, one slice more, and ragged last slices in either
    position, in both input types."""
    cap = 4 * torch.cuda.get_device_properties(0).multi_processor_count
    bf16_rows = (cap * 4, cap * 4 + 4, cap * 4 - 1,     # one slice per CTA, then two
                 cap * 4 + 2,                            # a ragged slice held in registers
                 cap * 8, cap * 8 - 1, cap * 8 + 4)      # two per CTA (ragged second), then two passes
    for i, rows in enumerate(bf16_rows):
        check_current(fq, synth.normal_outliers(rows, 4096, seed=71 + i), oracle.E4M3)
    for i, rows in enumerate((cap * 2, cap * 2 + 1, cap * 4, cap * 4 + 1)):
        check_current(fq, synth.f32_tensor(rows, 4096, seed=81 + i), oracle.E5M2, margin=1)
    # one element short of the largest single-slice tensor: a ragged last slice
    check_current(fq, synth.normal_outliers(1, cap * 16384 - 1, seed=86), oracle.E4M3)


def test_current_scaling_single_launch_streamed(fq):
    """Past the on-chip slices the single launch also streams an equal range
    of the remaining chunks per CTA (reduced, then cast after the wait), up
    to 8 times the on-chip capacity; beyond it, two passes.  Ragged last
    chunks, both input types, a margin, and the saturation count."""
    cap = 4 * torch.cuda.get_device_properties(0).multi_processor_count  # CTAs; 2 slices each on chip
    for i, rows in enumerate((cap * 8 * 3 + 5, cap * 8 * 8, cap * 8 * 8 + 4)):
        check_current(fq, synth.normal_outliers(rows, 4096, seed=91 + i), oracle.E4M3, margin=i)
    check_current(fq, synth.f32_tensor(cap * 4 * 3 + 3, 4096, seed=95), oracle.E5M2)
    # an odd row count: the last chunk holds one row of four
    check_current(fq, synth.normal_outliers(cap * 8 * 2 + 1, 4096, seed=96), oracle.E5M2)


def test_current_scaling_single_launch_specials(fq):
    """Special values in each part of the single launch: a NaN or an Inf in
    a streamed chunk, in the shared-memory slice and in the register slice
    (each makes the scale 1 and the amax the largest magnitude bits), and an
    all-zero tensor (amax 0, scale 1) at each size."""
    cap = 4 * torch.cuda.get_device_properties(0).multi_processor_count
    rows = cap * 8 * 2  # on-chip slices plus a streamed range of the same size
    base = synth.normal_outliers(rows, 4096, seed=97)
    flat_of = lambda r, c: r * 4096 + c
    cases = [(rows - 3, 17, 0x7FC1),        # NaN with a payload, in a streamed chunk
             (1, 4000, 0xFF80),             # -Inf, in CTA 0's register slice (rows 0-3 are slice 0)
             (6, 9, 0x7F80)]                # +Inf, in CTA 0's shared-memory slice (rows 4-7)
    for r, c, bits in cases:
        x = base.copy()
        x.reshape(-1)[flat_of(r, c)] = bits
        check_current(fq, x, oracle.E4M3)
    for n_rows in (4, cap * 4 * 2, rows):
        check_current(fq, np.zeros((n_rows, 4096), np.uint16), oracle.E5M2)


@pytest.mark.parametrize("fmt", FMTS)
def test_current_scaling_grouped(fq, fmt):
    """Per-expert scaling on ragged groups (empty, 1-row, boundary-straddling chunks)."""
    rows, cols = 700, 72
    x = synth.student_t(rows, cols, 4.0, seed=41)
    x = x.copy()
    # give each expert a different magnitude
    xf = bf16_to_f32(x) * np.repeat(np.exp(np.linspace(-4, 4, 7)), 100)[:, None].astype(np.float32)
    x = synth.to_bf16_bits(xf)
    offsets = [0, 0, 1, 130, 131, 131, 500, 700]
    check_current(fq, x, fmt, offsets=offsets)
    check_current(fq, x, fmt, margin=2, offsets=offsets)


def test_current_scaling_grouped_moe_shape(fq):
    """MoE routing: 64 experts over 8192 tokens x 1024 hidden, multinomial counts."""
    x = synth.student_t(8192, 1024, 4.0, seed=43)
    offs = synth.moe_offsets(8192, 64, seed=43)
    check_current(fq, x, oracle.E4M3, offsets=list(offs))


def test_special_values(fq):
    vals = np.array([0.0, -0.0, np.inf, -np.inf, 1e-40, -1e-42, 3e38, -3e38, 1.0, -2.5, 448.0, 449.0,
                     57344.0, 61440.0, 1e-3, 7.0], dtype=np.float32)
    x32 = np.tile(vals, 4).reshape(4, 16)
    for fmt in FMTS:
        check_current(fq, x32, fmt)  # Inf in the tensor: scale 1, amax Inf
        for s in (1.0, 0.5, 1e30):
            got = run_cast(fq, x32, fmt, scale=[s])
            ref, sat = oracle.cast(x32, np.float32(s), fmt)
            np.testing.assert_array_equal(got["q"], ref)
            assert got["sat"][0] == sat
            np.testing.assert_array_equal(f32bits(got["amax"]), [oracle.amax_bits(x32)])
    xn = x32.copy()
    xn[1, 3] = np.nan
    xn[2, 5] = -np.float32(np.nan)
    for fmt in FMTS:
        check_current(fq, xn, fmt)  # NaN: amax NaN, scale 1, NaN codes 0x7F
    # BF16 subnormals, zeros of both signs, NaN payloads
    b = np.array([0x0001, 0x8001, 0x007F, 0x0000, 0x8000, 0x7FC1, 0xFF80, 0x3F80, 0x4F00, 0x0080],
                 dtype=np.uint16)
    xb = np.tile(b, 32).reshape(10, 32)
    for fmt in FMTS:
        check_current(fq, xb, fmt)
        got = run_cast(fq, xb, fmt, scale=[2.0 ** 100])
        np.testing.assert_array_equal(got["q"], oracle.cast(xb, np.float32(2.0 ** 100), fmt)[0])


def test_zero_tensor_and_empty(fq):
    z = np.zeros((64, 64), np.uint16)
    z[3, 3] = 0x8000
    check_current(fq, z, oracle.E4M3)  # amax 0 -> scale 1, -0 keeps its sign
    e = np.zeros((0, 64), np.uint16)
    got = run_cast(fq, e, oracle.E4M3)
    assert got["amax"][0] == 0 and got["scale"][0] == 1.0 and got["sat"][0] == 0
    got = run_cast(fq, np.zeros((0, 8), np.uint16), oracle.E5M2, offsets=[0, 0, 0])
    assert (got["scale"] == 1.0).all() and (got["amax"] == 0).all()


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_given_scale_with_fused_amax(fq, dtype):
    rows, cols = 333, 96
    x = synth.normal_outliers(rows, cols, seed=51) if dtype == "bf16" else synth.f32_tensor(rows, cols, seed=51)
    offsets = [0, 100, 100, 333]
    scales = np.array([3.5, 1e-3, 90.25], np.float32)
    got = run_cast(fq, x, oracle.E5M2, scale=scales, offsets=offsets)
    flat = x.reshape(-1)
    for g in range(3):
        a, b = offsets[g] * cols, offsets[g + 1] * cols
        ref, sat = oracle.cast(flat, scales[g], oracle.E5M2, a, b)
        np.testing.assert_array_equal(got["q"][a:b], ref[a:b])
        assert got["sat"][g] == sat
        assert f32bits(got["amax"])[g] == oracle.amax_bits(flat, a, b)
        assert got["scale"][g] == scales[g]
        assert f32bits(got["scale_inv"])[g] == f32bits(oracle.reciprocal(scales[g]))


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_amax_entry_point(fq, dtype):
    rows, cols = 1000, 257
    x = synth.normal_outliers(rows, cols, seed=61) if dtype == "bf16" else synth.f32_tensor(rows, cols, seed=61)
    offsets = [0, 3, 3, 400, 999, 1000]
    out = Guarded((5,), torch.float32)
    fq.fp8q_amax(dev(x), group_offsets=offsets, out=out.t)
    torch.cuda.synchronize()
    out.check()
    flat = x.reshape(-1)
    want = [oracle.amax_bits(flat, offsets[g] * cols, offsets[g + 1] * cols) for g in range(5)]
    np.testing.assert_array_equal(f32bits(host(out.t)), want)
    one = fq.fp8q_amax(dev(x))
    assert f32bits(host(one))[0] == oracle.amax_bits(flat)
