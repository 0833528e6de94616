"""Pins for the CPU oracle: page values, closed forms and library routines.

Nothing here touches a GPU or the product library.  Each check ties the
oracle to something other than itself: a value printed on a page
(tests/golden/page_values.json, delayed_traces.txt), a closed form, an
invariant, or torch's own float8 conversion, so that a plausible slip in
the oracle (a wrong bias, a tie rounded away from even, a dropped sign, a
floor where the rule says ceil, a transposed index) fails at least one.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from synth import to_bf16_bits

GOLD = os.path.join(os.path.dirname(__file__), "golden")
PAGES = json.load(open(os.path.join(GOLD, "page_values.json"), encoding="utf-8"))
FMT = {"e4m3": oracle.E4M3, "e5m2": oracle.E5M2}
TORCH_FP8 = {oracle.E4M3: torch.float8_e4m3fn, oracle.E5M2: torch.float8_e5m2}


def torch_encode(fmt, values):
    """Library routine: clamp to +-max, then torch's RNE float8 conversion."""
    m = oracle.fp8_max(fmt)
    t = torch.from_numpy(np.asarray(values, dtype=np.float64)).clamp(-m, m)
    return t.to(TORCH_FP8[fmt]).view(torch.uint8).numpy()


# ---------------------------------------------------------------------------
# Page values
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("case", PAGES["encode"], ids=lambda c: c["id"])
def test_page_encode_examples(case):
    fmt = FMT[case["fmt"]]
    x = np.array([case["input"]], dtype=np.float32)
    if case["input_dtype"] == "bf16":
        x = to_bf16_bits(x)
    if "amax" in case:
        a = oracle.amax_bits(np.array([case["amax"]], dtype=np.float32))
        s, nf = oracle.per_tensor_scale(a, fmt, 0)
        assert not nf
        assert float(s) == case["scale"]
    else:
        s = np.float32(case["scale"])
    q, _ = oracle.cast(x, s, fmt)
    assert q[0] == int(case["code"], 16)
    assert oracle.fp8_value(fmt, int(q[0])) == case["value"]


def test_page_bf16_example():
    case = PAGES["bf16"][0]
    b = to_bf16_bits(np.array([case["input"]], dtype=np.float32))
    assert float(np.array([int(b[0]) << 16], dtype=np.uint32).view(np.float32)[0]) == case["bf16_value"]


@pytest.mark.parametrize("case", PAGES["formats"], ids=lambda c: c["id"])
def test_page_format_facts(case):
    fmt = FMT[case["fmt"]]
    assert oracle.fp8_max(fmt) == case["max"]
    vals = [oracle.fp8_value(fmt, c) for c in range(256)]
    finite_pos = sorted({v for v in vals if math.isfinite(v) and v > 0})
    # smallest subnormal / normal
    assert finite_pos[0] == 2.0 ** case["min_subnormal_exp"]
    min_normal = min(v for c, v in enumerate(vals) if math.isfinite(v) and v > 0 and (c & 0x7F) >> (3 if fmt == oracle.E4M3 else 2))
    assert min_normal == 2.0 ** case["min_normal_exp"]
    # binades: log2(max / smallest subnormal)
    assert round(math.log2(case["max"] / finite_pos[0]), 1) == case["binades"]
    # values per binade [1, 2)
    assert sum(1 for v in finite_pos if 1.0 <= v < 2.0) == case["values_per_binade"]
    if fmt == oracle.E4M3:
        nan_codes = [c for c in range(256) if math.isnan(vals[c])]
        assert nan_codes == [int(c, 16) for c in case["nan_codes"]]
        assert not any(math.isinf(v) for v in vals)
        assert [v for v in finite_pos if v >= 256] == case["top_binade"]
    else:
        assert vals[0x7C] == math.inf and vals[0xFC] == -math.inf
        assert all(math.isnan(vals[c]) for c in (0x7D, 0x7E, 0x7F))


@pytest.mark.parametrize("fmt,count", [(oracle.E4M3, 7), (oracle.E5M2, 3)])
def test_page_interior_values_in_1_2(fmt, count):
    """"混合精度与 FP8 训练" 3: 10000 points in [1,2] land on 7 (E4M3) / 3 (E5M2) interior values."""
    pts = np.linspace(1.0, 2.0, 10000)
    q = oracle.encode_array(fmt, pts)
    vals = {oracle.fp8_value(fmt, int(c)) for c in np.unique(q)}
    interior = sorted(v for v in vals if 1.0 < v < 2.0)
    assert len(interior) == count
    if fmt == oracle.E4M3:
        assert interior == [1.125, 1.25, 1.375, 1.5, 1.625, 1.75, 1.875]


def test_page_delayed_saturation_T5():
    case = PAGES["delayed_saturation"]
    fmt = FMT[case["fmt"]]
    d = oracle.DelayedScaling(history_len=16, interval=1, margin=case["margin"], fmt=fmt)
    x0 = np.array([case["history_amax"], 1.0, -3.0], dtype=np.float32)
    r0 = d.step(x0)
    assert np.isclose(float(r0["scale"]), case["scale_before"], rtol=1e-6)
    x1 = np.array([case["spike"], 1.0], dtype=np.float32)
    r1 = d.step(x1)
    assert np.isclose(float(r1["scale"]), case["scale_before"], rtol=1e-6)
    assert np.isclose(case["spike"] * float(r1["scale"]), case["spike_scaled"], rtol=1e-6)
    assert oracle.fp8_value(fmt, int(r1["q"][0])) == case["spike_code_value"]
    assert np.isclose(case["spike_code_value"] / float(r1["scale"]), case["spike_dequant"], rtol=1e-6)
    assert r1["sat"] == 1
    r2 = d.step(np.array([1.0], dtype=np.float32))
    assert np.isclose(float(r2["scale"]), case["scale_after"], rtol=1e-6)


def _read_traces():
    traces, cur = {}, None
    for line in open(os.path.join(GOLD, "delayed_traces.txt"), encoding="utf-8"):
        line = line.strip()
        if line.startswith("# trace"):
            parts = line[2:].split()
            cur = {"name": parts[1]}
            for kv in parts[2:]:
                k, _, v = kv.partition("=")
                if k in ("H", "margin") and v.isdigit():
                    cur[k] = int(v)
            cur["rows"] = []
            traces[cur["name"]] = cur
        elif line and not line.startswith("#") and cur is not None:
            t, a, used, rec = line.split()
            cur["rows"].append((int(t), float(a), float(used), rec == "yes"))
    return traces


@pytest.mark.parametrize("name", ["interval1", "interval5", "fifo"])
def test_page_delayed_interval_traces(name):
    tr = _read_traces()[name]
    interval = 5 if name == "interval5" else 1
    d = oracle.DelayedScaling(history_len=tr["H"], interval=interval, margin=tr["margin"],
                              fmt=oracle.E4M3)
    for t, a, used, rec in tr["rows"]:
        r = d.step(np.array([a, -a / 2], dtype=np.float32))
        expect, _ = oracle.per_tensor_scale(oracle.f32_to_bits(np.float32(used)), oracle.E4M3, 0)
        assert float(r["scale"]) == float(expect), (name, t)
        assert float(r["scale"]) == float(np.float32(448.0 / used)) or used == 0
        assert r["recorded"] == rec, (name, t)
        if rec:
            assert float(r["amax"]) == a


def test_delayed_margin_and_reset():
    """Margin N divides the delayed scale by 2^N; the first step (and the first
    after a reset) uses current scaling with no margin."""
    d = oracle.DelayedScaling(history_len=4, interval=1, margin=3, fmt=oracle.E4M3)
    r0 = d.step(np.array([2.0], dtype=np.float32))
    assert float(r0["scale"]) == 224.0  # current scaling, margin not applied
    r1 = d.step(np.array([1.0], dtype=np.float32))
    assert float(r1["scale"]) == 28.0  # 448/2 / 2^3
    d.reset()
    r2 = d.step(np.array([0.5], dtype=np.float32))
    assert float(r2["scale"]) == 896.0  # history forgotten: current scaling on 0.5


@pytest.mark.parametrize("case", PAGES["mx"], ids=lambda c: c["id"])
def test_page_mx_examples(case):
    fmt = FMT[case["fmt"]]
    v = np.zeros(32, dtype=np.float32)
    v[5] = case["amax"]
    v[7] = -case["amax"] / 3
    byte, q = oracle.mx_block(v, fmt)
    if "X" in case:
        assert byte == case["scale_byte"] and byte - 127 == case["X"]
    if case.get("all_zero"):
        assert not q.any()
    if "scaled_max" in case:
        assert np.isclose(case["amax"] * 2.0 ** -case["X"], case["scaled_max"])
        assert case["scaled_max"] < oracle.fp8_max(fmt)
    if "X_ocp" in case:
        ocp = math.floor(math.log2(case["amax"])) - 8  # "混合精度与 FP8 训练" 13.1 rule
        assert ocp == case["X_ocp"]
        assert case["amax"] * 2.0 ** -ocp > oracle.fp8_max(fmt)  # would saturate
        assert byte - 127 == case["X_roundup"]
        assert case["amax"] * 2.0 ** -(byte - 127) <= oracle.fp8_max(fmt)


# ---------------------------------------------------------------------------
# Closed forms and library routines
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_every_code_round_trips(fmt):
    for c in range(256):
        v = oracle.fp8_value(fmt, c)
        if math.isnan(v):
            assert oracle.fp8_encode(fmt, v) == 0x7F
        elif math.isinf(v):
            assert oracle.fp8_encode(fmt, v) == (c & 0x80) | oracle.fp8_max_code(fmt)
        else:
            assert oracle.fp8_encode(fmt, v) == c


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_midpoints_go_to_even_code(fmt):
    maxc = oracle.fp8_max_code(fmt)
    for c in range(maxc):
        lo, hi = oracle.fp8_value(fmt, c), oracle.fp8_value(fmt, c + 1)
        mid = (lo + hi) / 2
        even = c if c % 2 == 0 else c + 1
        assert oracle.fp8_encode(fmt, mid) == even
        assert oracle.fp8_encode(fmt, -mid) == 0x80 | even
        # just off the midpoint goes to the nearer side
        assert oracle.fp8_encode(fmt, np.nextafter(mid, -np.inf)) == c
        assert oracle.fp8_encode(fmt, np.nextafter(mid, np.inf)) == c + 1


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_all_bf16_patterns_match_torch(fmt):
    """All 2^16 BF16 patterns at scale 1 against torch's RNE float8 conversion."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = (bits.astype(np.uint32) << 16).view(np.float32)
    q, _ = oracle.cast(bits, 1.0, fmt)
    finite = ~np.isnan(vals)
    np.testing.assert_array_equal(q[finite], torch_encode(fmt, vals[finite].astype(np.float64)))
    assert (q[~finite] == 0x7F).all()  # NaN convention


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_random_fp32_patterns_match_torch(fmt):
    rng = np.random.default_rng(11)
    bits = rng.integers(0, 1 << 32, size=1 << 20, dtype=np.uint64).astype(np.uint32)
    # concentrate half of them in the FP8 range so that rounding is exercised
    bits[::2] = (rng.integers(0x33000000, 0x47800000, size=bits[::2].size, dtype=np.uint64)
                 | (rng.integers(0, 2, size=bits[::2].size, dtype=np.uint64) << 31)).astype(np.uint32)
    vals = bits.view(np.float32)
    q, _ = oracle.cast(vals, 1.0, fmt)
    ok = ~np.isnan(vals)
    np.testing.assert_array_equal(q[ok], torch_encode(fmt, vals[ok].astype(np.float64)))
    assert (q[~ok] == 0x7F).all()


def test_scaled_cast_matches_torch():
    """q = RNE_sat(fl32(x*s)): fl32 product by torch float32 multiply, then torch cast."""
    rng = np.random.default_rng(5)
    x = (rng.standard_normal(1 << 16) * 3).astype(np.float32)
    for s in [np.float32(1.7), np.float32(22400.0), np.float32(3.0e-3), np.float32(448.0 / 7.3)]:
        prod = (torch.from_numpy(x) * torch.tensor(s, dtype=torch.float32)).numpy()
        for fmt in (oracle.E4M3, oracle.E5M2):
            q, sat = oracle.cast(x, s, fmt)
            np.testing.assert_array_equal(q, torch_encode(fmt, prod.astype(np.float64)))
            assert sat == int((np.abs(prod) > oracle.fp8_max(fmt)).sum())


def test_amax_matches_numpy():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(100001) * 7).astype(np.float32)
    assert oracle.amax(x) == np.max(np.abs(x))
    b = to_bf16_bits(x)
    bf = (b.astype(np.uint32) << 16).view(np.float32)
    assert oracle.amax(b) == np.max(np.abs(bf))
    assert oracle.amax(b, 10, 20) == np.max(np.abs(bf[10:20]))
    x[77] = -np.inf
    assert oracle.amax(x) == np.inf
    x[78] = np.nan
    assert np.isnan(oracle.amax(x))
    assert oracle.amax(np.zeros(5, np.float32)) == 0.0
    assert oracle.amax(np.zeros(0, np.float32)) == 0.0


def test_per_tensor_scale_definition():
    for a in [0.02, 1.0, 3.7, 1e-30, 6e4]:
        s, nf = oracle.per_tensor_scale(oracle.f32_to_bits(np.float32(a)), oracle.E4M3, 0)
        assert s == np.float32(448.0) / np.float32(a) and not nf
        s3, _ = oracle.per_tensor_scale(oracle.f32_to_bits(np.float32(a)), oracle.E4M3, 3)
        assert s3 == np.float32(s / np.float32(8.0))
        s5, _ = oracle.per_tensor_scale(oracle.f32_to_bits(np.float32(a)), oracle.E5M2, 0)
        assert s5 == np.float32(57344.0) / np.float32(a)
    # special cases (our readings)
    assert oracle.per_tensor_scale(0, oracle.E4M3, 0) == (1.0, False)
    assert oracle.per_tensor_scale(0x7F800000, oracle.E4M3, 0) == (1.0, True)
    assert oracle.per_tensor_scale(0x7FC00000, oracle.E4M3, 0) == (1.0, True)
    s, _ = oracle.per_tensor_scale(1, oracle.E4M3, 0)  # smallest subnormal: overflow
    assert s == np.finfo(np.float32).max
    assert oracle.reciprocal(np.float32(3.0)) == np.float32(1.0) / np.float32(3.0)


def _ceil_log2_fraction(r: Fraction) -> int:
    """ceil(log2 r) for a positive rational, by integer bit lengths."""
    p, q = r.numerator, r.denominator
    k = p.bit_length() - q.bit_length()  # floor(log2 r) is k or k-1
    if Fraction(2) ** k > r:
        k -= 1
    return k if Fraction(2) ** k == r else k + 1


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_mx_scale_is_exact_ceil_log2(fmt):
    """X = ceil(log2(amax/destmax)) over the whole BF16 range, by rational
    arithmetic, and the invariant destmax/2 < amax*2^-X <= destmax."""
    destmax = Fraction(oracle.fp8_max(fmt))
    bits = np.arange(1, 0x7F80, dtype=np.uint32).astype(np.uint16)  # all positive finite BF16
    vals = (bits.astype(np.uint32) << 16).view(np.float32)
    for v in vals[::7]:
        blk = np.zeros(32, np.float32)
        blk[3] = v
        blk[9] = -v / 4
        byte, _ = oracle.mx_block(blk, fmt)
        X = _ceil_log2_fraction(Fraction(float(v)) / destmax)
        Xc = max(-127, min(127, X))
        assert byte == Xc + 127
        if Xc == X:
            scaled = Fraction(float(v)) / Fraction(2) ** X
            assert destmax / 2 < scaled <= destmax


def test_mx_integer_exponent_rule():
    """The same X by the exponent/mantissa rule: e - e_max + [m > 1.75]."""
    for fmt, emax in ((oracle.E4M3, 8), (oracle.E5M2, 15)):
        rng = np.random.default_rng(1)
        bits = rng.integers(0x00800000, 0x7F800000, size=20000, dtype=np.uint64).astype(np.uint32)
        for b in bits:
            e = (int(b) >> 23) - 127
            man = int(b) & 0x7FFFFF
            X = max(-127, min(127, e - emax + (1 if man > 0x600000 else 0)))
            blk = np.zeros(32, np.float32)
            blk[0] = np.array([b], np.uint32).view(np.float32)[0]
            assert oracle.mx_block(blk, fmt)[0] == X + 127


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_mx_elements_all_bf16_times_all_X(fmt):
    """Every BF16 value scaled by every 2^-X, against torch (the MX element step)."""
    bits = np.arange(1 << 16, dtype=np.uint32)
    vals = (bits << 16).view(np.float32)
    vals = vals[np.isfinite(vals)].astype(np.float64)
    for X in range(-127, 128):
        a = np.ldexp(vals, -X)
        np.testing.assert_array_equal(oracle.encode_array(fmt, a), torch_encode(fmt, a))


def test_mx_block_special_blocks():
    z = np.zeros(32, np.float32)
    z[4] = -0.0
    byte, q = oracle.mx_block(z, oracle.E4M3)
    assert byte == 0 and not q.any()  # zero block: X = -127, all 0 (no -0)
    v = np.ones(32, np.float32)
    v[2] = np.inf
    assert oracle.mx_block(v, oracle.E4M3)[0] == 0xFF
    assert (oracle.mx_block(v, oracle.E4M3)[1] == 0x7F).all()
    v[2] = np.nan
    assert oracle.mx_block(v, oracle.E5M2)[0] == 0xFF
    # negative zero inside a non-zero block keeps its sign
    v = np.ones(32, np.float32)
    v[1] = -0.0
    assert oracle.mx_block(v, oracle.E4M3)[1][1] == 0x80
    # a short block (trailing rows of a group) uses only the rows present
    b3, q3 = oracle.mx_block(np.array([1.0, -2.0, 0.5], np.float32), oracle.E4M3)
    assert b3 == 127 - 7 and q3.size == 3  # 2/448 -> X = ceil(log2(2/448)) = -7


def _bf16_from_f32(a):
    return to_bf16_bits(np.asarray(a, np.float32))


def test_mx_rowwise_matches_blocks():
    rng = np.random.default_rng(2)
    x = _bf16_from_f32(rng.standard_normal((5, 96)) * np.exp(rng.standard_normal((5, 1)) * 3))
    r = oracle.mx_quantize(x, oracle.E4M3, 1)
    xf = (x.astype(np.uint32) << 16).view(np.float32)
    for i in range(5):
        for j in range(3):
            b, q = oracle.mx_block(xf[i, 32 * j:32 * j + 32], oracle.E4M3)
            assert r["s_row"][i, j] == b
            np.testing.assert_array_equal(r["q_row"][i, 32 * j:32 * j + 32], q)


def test_mx_columnwise_is_rowwise_of_transpose_T11():
    """Column copy = rowwise quantization of x^T, taken from the BF16 tensor,
    not from re-quantizing the rowwise FP8 copy ("混合精度与 FP8 训练" 13.1)."""
    rng = np.random.default_rng(4)
    x = _bf16_from_f32(rng.standard_normal((64, 64)) * np.exp(rng.standard_normal((64, 1)) * 2))
    both = oracle.mx_quantize(x, oracle.E4M3, 3)
    rt = oracle.mx_quantize(np.ascontiguousarray(x.T), oracle.E4M3, 1)
    np.testing.assert_array_equal(both["q_col"], rt["q_row"])
    np.testing.assert_array_equal(both["s_col"], rt["s_row"])
    # requantizing the dequantized rowwise copy along columns gives something else
    deq = np.empty((64, 64), np.float32)
    for i in range(64):
        for j in range(2):
            s = 2.0 ** (int(both["s_row"][i, j]) - 127)
            for k in range(32):
                deq[i, 32 * j + k] = oracle.fp8_value(oracle.E4M3, int(both["q_row"][i, 32 * j + k])) * s
    requant = oracle.mx_quantize(np.ascontiguousarray(deq.T), oracle.E4M3, 1)
    assert (requant["q_row"] != both["q_col"]).any()


def test_mx_grouped_columns_restart_at_group_offsets():
    rng = np.random.default_rng(6)
    rows, cols = 150, 64
    x = _bf16_from_f32(rng.standard_normal((rows, cols)))
    offs = np.array([0, 0, 33, 34, 100, 150], np.int64)  # empty, 33, 1, 66, 50 rows
    r = oracle.mx_quantize(x, oracle.E4M3, 3, offsets=offs)
    assert r["col_blocks"] == 0 + 2 + 1 + 3 + 2
    base = 0
    for g in range(len(offs) - 1):
        r0, r1 = int(offs[g]), int(offs[g + 1])
        if r1 == r0:
            continue
        part = oracle.mx_quantize(np.ascontiguousarray(x[r0:r1]), oracle.E4M3, 2)
        nb = part["col_blocks"]
        np.testing.assert_array_equal(r["q_col"][:, r0:r1], part["q_col"])
        np.testing.assert_array_equal(r["s_col"][:, base:base + nb], part["s_col"])
        base += nb
    # the rowwise copy ignores groups
    np.testing.assert_array_equal(r["q_row"], oracle.mx_quantize(x, oracle.E4M3, 1)["q_row"])


def test_current_scaling_grouped_equals_per_slice():
    rng = np.random.default_rng(8)
    x = _bf16_from_f32(rng.standard_normal((40, 16)) * np.arange(1, 41)[:, None])
    offs = np.array([0, 7, 7, 40], np.int64)
    r = oracle.current_scaling(x, oracle.E4M3, offsets=offs)
    assert r["amax"][1] == 0 and r["scale"][1] == 1.0  # empty group
    for g, (a, b) in enumerate([(0, 7), (7, 40)]):
        gi = 0 if g == 0 else 2
        part = oracle.current_scaling(np.ascontiguousarray(x[a:b]), oracle.E4M3)
        np.testing.assert_array_equal(r["q"].reshape(40, 16)[a:b], part["q"].reshape(b - a, 16))
        assert r["scale"][gi] == part["scale"][0]


def test_current_scaling_max_element_lands_at_top():
    """Scale = F8max/amax maps the largest element to (about) F8max."""
    rng = np.random.default_rng(9)
    x = (rng.standard_normal((32, 32)) * 5).astype(np.float32)
    r = oracle.current_scaling(x, oracle.E4M3)
    i = np.argmax(np.abs(x))
    assert oracle.fp8_value(oracle.E4M3, int(r["q"][i]) & 0x7F) == 448.0


def test_scaled_cast_overflow_matches_ieee_single():
    """Products beyond the float range follow IEEE single overflow (to +-Inf),
    then saturate; torch's float32 multiply is the reference."""
    x = np.array([3e38, -3e38, 1.0, 2e38, -np.inf, 7e37], dtype=np.float32)
    for s in (np.float32(448.0), np.float32(1.5), np.float32(4.0)):
        prod = (torch.from_numpy(x) * torch.tensor(s, dtype=torch.float32)).numpy()
        for fmt in (oracle.E4M3, oracle.E5M2):
            q, sat = oracle.cast(x, s, fmt)
            np.testing.assert_array_equal(q, torch_encode(fmt, prod.astype(np.float64)))
            assert sat == int((np.abs(prod) > oracle.fp8_max(fmt)).sum())
    assert oracle.reciprocal(np.float32(1e-45)) == np.inf


# --------------------------------------------------------------------------
# Dequantization ("HiFloat8：高性能训练之路" 1.1-1.2: de-scaling by
# scale_inv; "Blackwell GPU MXFP8 预训练最佳实践" 4.1, 4.3: value * 2^X)
# --------------------------------------------------------------------------
F8_TORCH = {oracle.E4M3: torch.float8_e4m3fn, oracle.E5M2: torch.float8_e5m2}


def _torch_bf16_bits(f32: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(f32, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_bf16_rounding_matches_torch():
    """The oracle's nearest-BF16 against torch's float32 -> bfloat16 (RNE)."""
    rng = np.random.default_rng(21)
    bits = rng.integers(0, 1 << 32, size=1 << 20, dtype=np.uint64).astype(np.uint32)
    # exact midpoints and their neighbours, the top binade, subnormals
    mids = (rng.integers(0, 1 << 16, size=4096, dtype=np.uint64).astype(np.uint32) << 16) | 0x8000
    edge = np.array([0x7F7F7FFF, 0x7F7F8000, 0x7F7F8001, 0x7F7FFFFF, 0xFF7F8000, 0x00008000,
                     0x00018000, 0x00000001, 0x80000001, 0x3DCCCCCD], np.uint32)
    bits = np.concatenate([bits, mids, mids + 1, mids - 1, edge])
    f = bits.view(np.float32)
    got = oracle.bf16_round(f)
    want = _torch_bf16_bits(f)
    ok = ~np.isnan(f)
    np.testing.assert_array_equal(got[ok], want[ok])
    assert (got[~ok] == 0x7FC0).all()


def test_bf16_rounding_page_example():
    """BF16(0.1) = 0.10009765625 ("混合精度与 FP8 训练" 2.2)."""
    b = int(oracle.bf16_round([np.float32(0.1)])[0])
    assert np.array([b << 16], np.uint32).view(np.float32)[0] == np.float32(0.10009765625)


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_dequant_decode_matches_torch(fmt):
    """All 256 codes at scale_inv 1 (FP32 out) against torch's float8 -> float32."""
    codes = np.arange(256, dtype=np.uint8).reshape(1, 256)
    y = oracle.dequant_per_tensor(codes, fmt, [1.0], out_dt=1).view(np.float32).reshape(-1)
    want = torch.from_numpy(codes.reshape(-1)).view(F8_TORCH[fmt]).to(torch.float32).numpy()
    nan = np.isnan(want)
    np.testing.assert_array_equal(y[~nan], want[~nan])
    assert np.isnan(y[nan]).all() and (y[nan].view(np.uint32) == 0x7FC00000).all()


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
@pytest.mark.parametrize("out_dt", [0, 1])
def test_dequant_per_tensor_matches_torch(fmt, out_dt):
    """y = round_out(fl32(value * scale_inv)) against torch float32 arithmetic."""
    rng = np.random.default_rng(22)
    q = rng.integers(0, 256, size=(64, 256), dtype=np.uint64).astype(np.uint8)
    offs = np.array([0, 5, 5, 40, 64], np.int64)
    si = np.array([1.0 / 448, 3.7e-3, 1.0, 2.0 ** 100], np.float32)
    y = oracle.dequant_per_tensor(q, fmt, si, out_dt=out_dt, offsets=offs)
    v = torch.from_numpy(q.reshape(-1)).view(F8_TORCH[fmt]).to(torch.float32).reshape(64, 256)
    srow = torch.from_numpy(np.repeat(si, np.diff(offs)).astype(np.float32)).reshape(64, 1)
    prod = (v * srow).numpy()
    want = _torch_bf16_bits(prod) if out_dt == 0 else prod.view(np.uint32)
    nan = np.isnan(prod)
    np.testing.assert_array_equal(y[~nan], want[~nan])
    assert (y[nan] == (0x7FC0 if out_dt == 0 else 0x7FC00000)).all()


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_mx_dequant_then_quantize_round_trips(fmt):
    """Every finite code under every scale byte: a block holding
    value(c) * 2^X next to the format's maximum times 2^X quantizes back to
    byte X + 127 and code c, so the dequantizer applies exactly the
    exponent the quantizer chose."""
    fin = [c for c in range(256) if np.isfinite(oracle.fp8_value(fmt, c))]
    maxc = oracle.fp8_max_code(fmt)
    for byte in range(0, 255, 1):
        X = byte - 127
        if X > 127 - 16:  # max * 2^X would overflow FP32
            continue
        q = np.zeros((len(fin), 32), np.uint8)
        q[:, 0] = fin
        q[:, 1] = maxc
        s = np.full((len(fin), 1), byte, np.uint8)
        y = oracle.mx_dequantize(q, s, fmt, 1, len(fin), 32, out_dt=1).view(np.float32)
        r = oracle.mx_quantize(y, fmt, 1)
        assert (r["s_row"][:, 0] == byte).all(), byte
        np.testing.assert_array_equal(r["q_row"][:, 0], np.array(fin, np.uint8))


def test_mx_dequant_special_bytes_and_codes():
    q = np.array([[0x00, 0x80, 0x7F, 0x01] * 8], np.uint8)
    y = oracle.mx_dequantize(q, np.array([[0xFF]], np.uint8), oracle.E4M3, 1, 1, 32, out_dt=1).view(np.uint32)
    assert (y == 0x7FC00000).all()  # scale byte 0xFF: every element NaN
    y = oracle.mx_dequantize(q, np.array([[0]], np.uint8), oracle.E4M3, 1, 1, 32, out_dt=1).view(np.float32)
    assert y[0, 0] == 0.0 and np.signbit(y[0, 1]) and np.isnan(y[0, 2])
    assert y[0, 3] == np.float32(2.0 ** -9 * 2.0 ** -127)  # smallest subnormal code at X = -127, exact
    big = oracle.mx_dequantize(np.array([[0x7E] * 32], np.uint8), np.array([[254]], np.uint8), oracle.E4M3, 1, 1,
                               32, out_dt=0)
    assert (big == 0x7F80).all()  # 448 * 2^127 overflows to +Inf


def test_mx_dequant_columnwise_is_rowwise_of_transpose():
    """The columnwise copy dequantizes in its own [cols][rows] layout exactly
    as the rowwise copy of x^T does; with groups, as each group's slice."""
    rng = np.random.default_rng(23)
    x = _bf16_from_f32(rng.standard_normal((96, 64)) * np.exp(rng.standard_normal((96, 1)) * 3))
    both = oracle.mx_quantize(x, oracle.E4M3, 3)
    yc = oracle.mx_dequantize(both["q_col"], both["s_col"], oracle.E4M3, 2, 96, 64)
    rt = oracle.mx_quantize(np.ascontiguousarray(x.T), oracle.E4M3, 1)
    yr = oracle.mx_dequantize(rt["q_row"], rt["s_row"], oracle.E4M3, 1, 64, 96)
    np.testing.assert_array_equal(yc, yr)
    offs = np.array([0, 7, 7, 45, 96], np.int64)
    g = oracle.mx_quantize(x, oracle.E5M2, 2, offsets=offs)
    yg = oracle.mx_dequantize(g["q_col"], g["s_col"], oracle.E5M2, 2, 96, 64, offsets=offs)
    for a, b in zip(offs[:-1], offs[1:]):
        if a == b:
            continue
        sl = oracle.mx_quantize(np.ascontiguousarray(x[a:b]), oracle.E5M2, 2)
        ys = oracle.mx_dequantize(sl["q_col"], sl["s_col"], oracle.E5M2, 2, b - a, 64)
        np.testing.assert_array_equal(yg[:, a:b], ys)


# --------------------------------------------------------------------------
# MX scale rules: round-up (built) and the OCP round-down rule
# ("混合精度与 FP8 训练" 13.1; "Blackwell GPU MXFP8 预训练最佳实践" 4.1)
# --------------------------------------------------------------------------
def _floor_log2_fraction(r: Fraction) -> int:
    """Exact floor(log2 r) of a positive rational."""
    e = r.numerator.bit_length() - r.denominator.bit_length()
    while Fraction(2) ** e > r:
        e -= 1
    while Fraction(2) ** (e + 1) <= r:
        e += 1
    return e


def test_page_mx_ocp_examples():
    """13.1's example: amax 5.3 in E4M3 -> shared exponent 2 - 8 = -6, the top
    element becomes about 339 and nothing saturates; and the T8 case: amax 480
    -> X_ocp = 0 saturates to 448 where the round-up rule's X = 1 does not."""
    v = np.zeros(32, np.float32)
    v[5], v[7] = 5.3, -5.3 / 3
    b, q, n = oracle.mx_block_rule(v, oracle.E4M3, oracle.MX_RULE_OCP)
    assert b - 127 == -6 and n == 0
    assert abs(oracle.fp8_value(oracle.E4M3, int(q[5])) - 5.3 * 64) < 16
    case = next(c for c in json.load(open(os.path.join(GOLD, "page_values.json")))["mx"] if c["id"] == "T8-ocp")
    v[5], v[7] = case["amax"], -case["amax"] / 3
    b, q, n = oracle.mx_block_rule(v, oracle.E4M3, oracle.MX_RULE_OCP)
    assert b - 127 == case["X_ocp"] and n == 1 and q[5] == oracle.fp8_max_code(oracle.E4M3)
    b, q, n = oracle.mx_block_rule(v, oracle.E4M3, oracle.MX_RULE_UP)
    assert b - 127 == case["X_roundup"] and n == 0


@pytest.mark.parametrize("fmt,emax", [(oracle.E4M3, 8), (oracle.E5M2, 15)])
def test_mx_ocp_exponent_is_exact_floor_log2(fmt, emax):
    """Over every positive finite BF16 value as the block amax, X equals
    floor(log2 amax) - e_max in exact rational arithmetic, clamped to the
    UE8M0 range."""
    for bits in range(1, 0x7F80, 7):
        a = float(np.array([bits << 16], np.uint32).view(np.float32)[0])
        v = np.zeros(32, np.float32)
        v[3] = a
        b, _, _ = oracle.mx_block_rule(v, fmt, oracle.MX_RULE_OCP)
        want = min(max(_floor_log2_fraction(Fraction(a)) - emax, -127), 127)
        assert b - 127 == want, (hex(bits), b)


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_mx_rules_relation_and_saturation(fmt):
    """On random blocks: the round-up exponent is the OCP one or one above
    it; the round-up rule never saturates; the OCP rule saturates exactly the
    elements the round-up rule keeps below the maximum only by choosing the
    larger exponent; equal exponents give equal codes."""
    rng = np.random.default_rng(31)
    for _ in range(3000):
        v = (rng.standard_normal(32) * np.exp(rng.standard_normal() * 8)).astype(np.float32)
        bu, qu, nu = oracle.mx_block_rule(v, fmt, oracle.MX_RULE_UP)
        bo, qo, no = oracle.mx_block_rule(v, fmt, oracle.MX_RULE_OCP)
        assert bu - bo in (0, 1) and nu == 0
        if bu == bo:
            np.testing.assert_array_equal(qu, qo)
            assert no == 0
        else:
            mx = oracle.fp8_max(fmt)
            assert no == int(np.sum(np.abs(v.astype(np.float64)) * 2.0 ** -(bo - 127) > mx))


def test_mx_quantize_rule_matches_blocks_and_transpose():
    rng = np.random.default_rng(32)
    x = _bf16_from_f32(rng.standard_normal((64, 96)) * np.exp(rng.standard_normal((64, 1)) * 3))
    up = oracle.mx_quantize_rule(x, oracle.E4M3, 3, oracle.MX_RULE_UP)
    base = oracle.mx_quantize(x, oracle.E4M3, 3)
    for k in ("q_row", "s_row", "q_col", "s_col"):
        np.testing.assert_array_equal(up[k], base[k])
    assert up["sat"] == [0, 0]
    ocp = oracle.mx_quantize_rule(x, oracle.E4M3, 3, oracle.MX_RULE_OCP)
    xf = (x.astype(np.uint32) << 16).view(np.float32)
    nrow = 0
    for i in range(64):
        for j in range(3):
            b, q, n = oracle.mx_block_rule(xf[i, 32 * j:32 * j + 32], oracle.E4M3, oracle.MX_RULE_OCP)
            assert ocp["s_row"][i, j] == b
            np.testing.assert_array_equal(ocp["q_row"][i, 32 * j:32 * j + 32], q)
            nrow += n
    assert ocp["sat"][0] == nrow
    rt = oracle.mx_quantize_rule(np.ascontiguousarray(x.T), oracle.E4M3, 1, oracle.MX_RULE_OCP)
    np.testing.assert_array_equal(ocp["q_col"], rt["q_row"])
    np.testing.assert_array_equal(ocp["s_col"], rt["s_row"])
    assert ocp["sat"][1] == rt["sat"][0]


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_mx_ocp_value_on_the_maximum_is_not_saturated(fmt):
    """An element that scales exactly onto the format's maximum is
    representable: it is not counted as saturated (|v * 2^-X| > max only)."""
    mx = oracle.fp8_max(fmt)
    for k in (-20, 0, 7):
        v = np.zeros(32, np.float32)
        v[0] = mx * 2.0 ** k
        v[1] = -mx * 2.0 ** k
        b, q, n = oracle.mx_block_rule(v, fmt, oracle.MX_RULE_OCP)
        assert n == 0 and q[0] == oracle.fp8_max_code(fmt)
        v[2] = np.float32(mx * 2.0 ** k * 1.0625)  # just above: saturates
        b, q, n = oracle.mx_block_rule(v, fmt, oracle.MX_RULE_OCP)
        assert n == 1


# --------------------------------------------------------------------------
# Blockwise FP8 ("混合精度与 FP8 训练" 10.2-10.5)
# --------------------------------------------------------------------------
def _act(rows, cols, seed):
    rng = np.random.default_rng(seed)
    return _bf16_from_f32(rng.standard_normal((rows, cols)) * np.exp(rng.standard_normal((rows, 1)) * 2))


@pytest.mark.parametrize("group", [(1, 128), (128, 128)])
def test_blockwise_groups_are_current_scaling_of_each_slice(group):
    """Each group is quantized exactly as current scaling of that slice alone
    (its amax, Scale = F8max / amax, the saturating cast)."""
    x = _act(200, 300, 41)
    q, si = oracle.blockwise(x, oracle.E4M3, group)
    gr, gc = group
    for br in range(si.shape[0]):
        for bc in range(si.shape[1]):
            sl = np.ascontiguousarray(x[br * gr:(br + 1) * gr, bc * gc:(bc + 1) * gc])
            ref = oracle.current_scaling(sl, oracle.E4M3)
            np.testing.assert_array_equal(q[br * gr:(br + 1) * gr, bc * gc:(bc + 1) * gc].reshape(-1), ref["q"])
            assert si[br, bc].view(np.uint32) == ref["scale_inv"][0].view(np.uint32)


def test_blockwise_128x1_is_1x128_of_the_transpose():
    """The transposed copy's 128x1 groups are the 1x128 groups of x^T (10.5:
    a 1x128 result cannot simply be transposed, so both come from x)."""
    x = _act(300, 160, 42)
    q, si = oracle.blockwise(x, oracle.E4M3, (128, 1))
    qt, sit = oracle.blockwise(np.ascontiguousarray(x.T), oracle.E4M3, (1, 128))
    np.testing.assert_array_equal(q.T, qt)
    np.testing.assert_array_equal(si.T, sit)


def test_pow2_floor_closed_form():
    rng = np.random.default_rng(43)
    for s in np.concatenate([rng.lognormal(0, 20, 2000), [1.0, 2.0, 0.5, 3.4e38, 1e-30]]).astype(np.float32):
        p = float(oracle.pow2_floor(s))
        assert math.frexp(p)[0] == 0.5 and p <= float(s) < 2 * p, s


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_blockwise_power_of_two_scales(fmt):
    """10.4's power-of-two scales: the largest power of two that keeps the
    group's amax at or below the format maximum; codes are the cast with it."""
    x = _act(64, 256, 44)
    q, si = oracle.blockwise(x, fmt, (1, 128), pow2=True)
    xf = (x.astype(np.uint32) << 16).view(np.float32)
    mx = oracle.fp8_max(fmt)
    for r in range(64):
        for b in range(2):
            s = 1.0 / float(si[r, b])
            assert math.frexp(s)[0] == 0.5
            amax = float(np.max(np.abs(xf[r, 128 * b:128 * b + 128])))
            assert amax * s <= mx < 2 * amax * s
            qc, _ = oracle.cast(np.ascontiguousarray(x[r, 128 * b:128 * b + 128]), np.float32(s), fmt)
            np.testing.assert_array_equal(q[r, 128 * b:128 * b + 128], qc)


def test_page_outlier_demo_only_touches_its_groups():
    """Section 9's demo: a 128x256 activation with two outlier channels in the
    first 128 columns.  Every 1x128 group that holds them gets a larger
    scale_inv; the right half is exactly what it is without the outliers."""
    rng = np.random.default_rng(45)
    base = rng.standard_normal((128, 256)).astype(np.float32)
    out = base.copy()
    out[:, 7] *= 1000.0
    out[:, 100] *= 300.0
    xb, xo = _bf16_from_f32(base), _bf16_from_f32(out)
    qb, sb = oracle.blockwise(xb, oracle.E4M3, (1, 128))
    qo, so = oracle.blockwise(xo, oracle.E4M3, (1, 128))
    assert (so[:, 0] > sb[:, 0]).all()
    np.testing.assert_array_equal(qo[:, 128:], qb[:, 128:])
    np.testing.assert_array_equal(so[:, 1], sb[:, 1])


# --------------------------------------------------------------------------
# NVFP4 ("混合精度与 FP8 训练" 13.2)
# --------------------------------------------------------------------------
def test_page_e2m1_values():
    """E2M1 represents 0, 0.5, 1, 1.5, 2, 3, 4, 6 and their negatives."""
    vals = [oracle.e2m1_value(c) for c in range(16)]
    assert vals[:8] == [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    assert vals[8:] == [-v for v in vals[:8]]


def test_page_nvfp4_example():
    """The amax-5.3 block: block scale 5.3/6 ~ 0.883 stored in E4M3 as
    0.875; 5.3/0.875 ~ 6.06 rounds to 6; dequantized 5.25, under 1% off."""
    v = np.zeros(16, np.float32)
    v[3] = 5.3
    code, q = oracle.nvfp4_block(v, 1.0)
    d = oracle.fp8_value(oracle.E4M3, code)
    assert d == 0.875 and abs(5.3 / 6 - 0.883) < 1e-3
    assert oracle.e2m1_value(int(q[3])) == 6.0
    assert oracle.e2m1_value(int(q[3])) * d == 5.25 and abs(5.25 - 5.3) / 5.3 < 0.01


def test_e2m1_encoding_brute_force():
    """Nearest E2M1 value with ties to the even code, saturating at 6, over a
    fine grid and every midpoint (the rounding of "混合精度与 FP8 训练" 4.1)."""
    mags = [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    grid = np.concatenate([np.linspace(-8, 8, 4097), [(a + b) / 2 for a, b in zip(mags, mags[1:])]])
    for a in grid:
        m = abs(a)
        best = min(range(8), key=lambda c: (abs(mags[c] - m), c & 1))
        if m >= 6:
            best = 7
        want = best | (8 if a < 0 or (a == 0 and math.copysign(1, a) < 0) else 0)
        assert oracle.e2m1_encode(a) == want, a


def test_nvfp4_tensor_scale_and_blocks():
    """S = 448 * 6 / amax puts the block holding the tensor's amax on the
    E4M3 maximum (no block scale overflows); every block is the block rule
    under S; codes pack two per byte, the even element low."""
    rng = np.random.default_rng(51)
    x = _bf16_from_f32(rng.standard_normal((8, 64)) * np.exp(rng.standard_normal((8, 1)) * 3))
    r = oracle.nvfp4(x)
    xf = (x.astype(np.uint32) << 16).view(np.float32)
    amax = float(np.max(np.abs(xf)))
    assert r["S"] == np.float32(448.0 * 6.0 / amax)
    assert max(oracle.fp8_value(oracle.E4M3, int(c)) for c in r["s"].reshape(-1)) == 448.0
    for i in range(8):
        for j in range(4):
            code, q = oracle.nvfp4_block(xf[i, 16 * j:16 * j + 16], r["S"])
            assert r["s"][i, j] == code
            packed = r["q"][i, 8 * j:8 * j + 8]
            np.testing.assert_array_equal(packed & 0xF, q[0::2])
            np.testing.assert_array_equal(packed >> 4, q[1::2])


def test_nvfp4_zero_block_and_dequant_error():
    """An all-zero block gets scale 0 and zero codes; on random blocks the
    dequantized values (code * scale / S) stay within half an E2M1 step of x
    except where the element saturates."""
    code, q = oracle.nvfp4_block(np.zeros(16, np.float32), 1.0)
    assert code == 0 and not q.any()
    rng = np.random.default_rng(52)
    for _ in range(500):
        v = (rng.standard_normal(16) * np.exp(rng.standard_normal() * 4)).astype(np.float32)
        S = np.float32(448 * 6 / np.max(np.abs(v)) * rng.uniform(0.5, 1.0))
        code, q = oracle.nvfp4_block(v, S)
        d = oracle.fp8_value(oracle.E4M3, code)
        for i in range(16):
            y = oracle.e2m1_value(int(q[i])) * d / float(S)
            scaled = abs(float(v[i])) * float(S) / d
            if scaled < 6:
                assert abs(y - float(v[i])) <= 1.0 * d / float(S) + 1e-12 * abs(float(v[i]))


# --------------------------------------------------------------------------
# Quantization-error statistics ("昇腾 Ascend 950 低精度格式", appendix 3.4:
# SQNR and zero-rate of quantized tensors)
# --------------------------------------------------------------------------
def _uniform_sqnr_db(man_bits):
    """x uniform on [1, 2) rounded to a grid of step h = 2^-m: the error is
    uniform on [-h/2, h/2], so E[e^2] = h^2 / 12 and E[x^2] = 7/3."""
    return 10.0 * math.log10(7.0 / 3.0 * 12.0 * 4.0 ** man_bits)


def test_qstats_exact_copy_closed_form():
    """Powers of two are exact in both formats: noise 0 and signal the
    geometric sum; zeros count as zero but not as flushed."""
    for fmt in (oracle.E4M3, oracle.E5M2):
        ks = np.arange(-6, 9)
        x = np.zeros((1, 64), np.float32)
        x[0, :ks.size] = 2.0 ** ks
        x[0, 32:32 + ks.size] = -(2.0 ** ks)
        want_signal = 2 * sum(Fraction(4) ** int(k) for k in ks)
        q, _ = oracle.cast(x, 1.0, fmt)
        st = oracle.qstats_per_tensor(x, q.reshape(1, 64), fmt, [1.0])
        assert st["noise"] == 0.0 and Fraction(st["signal"]) == want_signal
        assert (st["n"], st["n_zero"], st["n_flushed"], st["n_nonfinite"]) == (64, 64 - 2 * ks.size, 0, 0)
        r = oracle.mx_quantize(x, fmt, 3)
        for d, (qq, ss) in ((1, ("q_row", "s_row")), (2, ("q_col", "s_col"))):
            st = oracle.qstats_mx(x, r[qq], r[ss], fmt, d)
            assert st["noise"] == 0.0 and Fraction(st["signal"]) == want_signal


def test_qstats_worked_elements():
    """Hand-computed elements under E4M3 with scale 1: 1 + 2^-5 rounds to 1;
    2^-11 is below half the smallest subnormal 2^-9 and is flushed; 0 is
    zero but not flushed; 500 saturates to 448; +Inf (cast to 448) and NaN
    (code 0x7F) are non-finite and left out of both sums."""
    vals = [1 + 2 ** -5, 2 ** -11, 0.0, 500.0, np.inf, np.nan]
    x = np.array([vals], np.float32)
    q, _ = oracle.cast(x, 1.0, oracle.E4M3)
    st = oracle.qstats_per_tensor(x, q.reshape(x.shape), oracle.E4M3, [1.0])
    F = Fraction
    assert F(st["signal"]) == (1 + F(1, 32)) ** 2 + F(1, 2 ** 22) + 500 ** 2
    assert F(st["noise"]) == F(1, 2 ** 10) + F(1, 2 ** 22) + 52 ** 2
    assert (st["n"], st["n_zero"], st["n_flushed"], st["n_nonfinite"]) == (6, 2, 1, 2)
    # one flushed element (2^-11) of the six compared
    assert oracle.zero_rate(st) == 1 / 6
    assert oracle.zero_rate({"n": 0, "n_flushed": 0}) == 0.0


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_qstats_uniform_per_tensor_sqnr(fmt):
    """Per-tensor copy of x = 2^-5 * U[1, 2) under scale 2^5: the SQNR of
    uniform rounding error (3 mantissa bits: 32.53 dB, 2 bits: 26.51 dB)
    to within sampling noise."""
    rng = np.random.default_rng(61)
    x = ((1.0 + rng.random((512, 1024))) / 32.0).astype(np.float32)
    q, _ = oracle.cast(x, 32.0, fmt)
    st = oracle.qstats_per_tensor(x, q.reshape(x.shape), fmt, [1.0 / 32.0])
    assert abs(oracle.sqnr_db(st) - _uniform_sqnr_db(3 if fmt == oracle.E4M3 else 2)) < 0.03
    assert st["n_zero"] == 0


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_qstats_mx_uniform_rows_of_any_magnitude(fmt):
    """MX copies of U[1, 2) * 2^k, k constant along each block (per row for
    the rowwise copy, per column for the columnwise one): every block
    scales its binade onto the format's, so both copies (grouped
    columnwise too) keep the uniform-rounding SQNR and flush nothing; a
    scale paired with the wrong block would not."""
    rng = np.random.default_rng(62)
    rows, cols = 600, 512
    u = 1.0 + rng.random((rows, cols))
    want = _uniform_sqnr_db(3 if fmt == oracle.E4M3 else 2)
    for K, offs in ((-40, None), (0, np.array([0, 0, 45, 46, 130, 600])), (40, None)):
        x_by = {1: (u * 2.0 ** (K + rng.integers(-2, 3, size=(rows, 1)))).astype(np.float32),
                2: (u * 2.0 ** (K + rng.integers(-2, 3, size=(1, cols)))).astype(np.float32)}
        for d, (qq, ss) in ((1, ("q_row", "s_row")), (2, ("q_col", "s_col"))):
            r = oracle.mx_quantize(x_by[d], fmt, d, offsets=offs)
            st = oracle.qstats_mx(x_by[d], r[qq], r[ss], fmt, d, offsets=offs)
            assert abs(oracle.sqnr_db(st) - want) < 0.06, (d, K)
            assert st["n_flushed"] == 0 and st["n"] == rows * cols


def test_page_mxfp8_sqnr_band():
    """Gaussian weights under MXFP8 E4M3 land in the SQNR band the page
    measured for MXFP8 activations (30.5-33.5 dB), within 0.5 dB of the
    highest weight SQNR it reports (31.4 dB)."""
    act = next(c for c in PAGES["sqnr"] if c["id"] == "SQNR-act")
    wt = next(c for c in PAGES["sqnr"] if c["id"] == "SQNR-weight")
    x = np.random.default_rng(63).standard_normal((512, 1024)).astype(np.float32)
    r = oracle.mx_quantize(x, oracle.E4M3, 1)
    db = oracle.sqnr_db(oracle.qstats_mx(x, r["q_row"], r["s_row"], oracle.E4M3, 1))
    lo, hi = act["sqnr_db_band"]
    assert lo <= db <= hi and abs(db - wt["sqnr_db_max"]) < 0.5


def test_qstats_nonfinite_elements_leave_the_sums():
    """Inf and NaN inputs, and a block whose scale byte is 0xFF, change only
    n_nonfinite: the sums are those of the finite elements alone."""
    rng = np.random.default_rng(64)
    x = rng.standard_normal((4, 64)).astype(np.float32)
    r = oracle.mx_quantize(x, oracle.E4M3, 1)
    base = oracle.qstats_mx(x, r["q_row"], r["s_row"], oracle.E4M3, 1)
    s = r["s_row"].copy()
    s[2, 1] = 0xFF
    st = oracle.qstats_mx(x, r["q_row"], s, oracle.E4M3, 1)
    keep = np.ones_like(x, bool)
    keep[2, 32:] = False
    xs, qs = x[keep].reshape(-1, 32), r["q_row"][keep].reshape(-1, 32)
    part = oracle.qstats_mx(xs, qs, np.delete(r["s_row"].reshape(-1), 5).reshape(-1, 1), oracle.E4M3, 1)
    assert st["n_nonfinite"] == 32 and st["n"] == base["n"]
    assert st["signal"] == pytest.approx(part["signal"], rel=1e-15)
    assert st["noise"] == pytest.approx(part["noise"], rel=1e-15)


# --------------------------------------------------------------------------
# MXFP4 / MXFP6 ("混合精度与 FP8 训练" 13.1-13.2; E2M3 / E3M2 are the OCP
# reading of the MXFP6 that "Blackwell GPU MXFP8 预训练最佳实践" 3.2 names)
# --------------------------------------------------------------------------
LP = {"e2m1": oracle.E2M1, "e2m3": oracle.E2M3, "e3m2": oracle.E3M2}
LP_CODES = {oracle.E2M1: 8, oracle.E2M3: 32, oracle.E3M2: 32}


def _lp_magnitudes(fmt):
    """The non-negative values built binade by binade (a uniform grid of
    2^m steps per binade, the subnormal range continuing the first
    binade's step down to 0), not from the bit fields."""
    m, lo_exp, hi_exp = {oracle.E2M1: (1, 0, 2), oracle.E2M3: (3, 0, 2), oracle.E3M2: (2, -2, 4)}[fmt]
    step0 = Fraction(2) ** lo_exp / 2 ** m
    vals = [k * step0 for k in range(2 ** m)]                      # [0, 2^lo_exp)
    for e in range(lo_exp, hi_exp + 1):
        vals += [Fraction(2) ** e * (1 + Fraction(k, 2 ** m)) for k in range(2 ** m)]
    return vals


@pytest.mark.parametrize("name", ["e2m1", "e2m3", "e3m2"])
def test_lp_values_binade_construction(name):
    """Codes 0 .. top decode to the binade-by-binade value list in order;
    the sign bit negates; E2M1 is the page's list 0, 0.5, 1, 1.5, 2, 3, 4,
    6; the largest values are 6, 7.5 and 28."""
    fmt = LP[name]
    n = LP_CODES[fmt]
    want = _lp_magnitudes(fmt)
    assert len(want) == n
    got = [Fraction(oracle.lp_value(fmt, c)) for c in range(n)]
    assert got == want
    assert [oracle.lp_value(fmt, c + n) for c in range(n)] == [-float(v) for v in want]
    assert float(want[-1]) == {"e2m1": 6.0, "e2m3": 7.5, "e3m2": 28.0}[name]
    if name == "e2m1":
        assert [float(v) for v in want] == [0, 0.5, 1, 1.5, 2, 3, 4, 6]


@pytest.mark.parametrize("name", ["e2m1", "e2m3", "e3m2"])
def test_lp_encoding_brute_force(name):
    """Nearest value, ties to the even code, saturating at the largest
    magnitude, sign (of zero too) kept -- over a fine grid and every
    midpoint."""
    fmt = LP[name]
    n = LP_CODES[fmt]
    mags = [float(v) for v in _lp_magnitudes(fmt)]
    top = mags[-1]
    grid = np.concatenate([np.linspace(-1.2 * top, 1.2 * top, 6001), [(a + b) / 2 for a, b in zip(mags, mags[1:])],
                           [-(a + b) / 2 for a, b in zip(mags, mags[1:])], [0.0, -0.0]])
    for a in grid:
        m = abs(a)
        best = n - 1 if m >= top else min(range(n), key=lambda c: (abs(mags[c] - m), c & 1))
        want = best | (n if math.copysign(1.0, a) < 0 else 0)
        assert oracle.lp_encode(fmt, a) == want, (name, a)


def test_page_mxfp4_example():
    """The amax-5.3 block with E2M1 elements: e_max 2, shared exponent 0,
    scale 1; 5.3 rounds to 6, a 13% error (OCP rule; the round-up rule
    gives the same exponent since 5.3 <= 6)."""
    case = next(c for c in PAGES["mx_lowbit"] if c["id"] == "T6-e2m1")
    v = np.zeros(32, np.float32)
    v[5] = case["amax"]
    for rule in (1, 0):
        byte, q, sat = oracle.mxlp_block(v, oracle.E2M1, rule)
        assert byte == case["scale_byte"] and byte - 127 == case["X"] and sat == 0
        assert oracle.lp_value(oracle.E2M1, int(q[5])) == case["element_value"]
        assert round(100 * (case["element_value"] - case["amax"]) / case["amax"]) == case["rel_err_pct"]
        assert not np.delete(q, 5).any()


@pytest.mark.parametrize("name", ["e2m1", "e2m3", "e3m2"])
def test_mxlp_rules(name):
    """Round-up X is the smallest with amax <= destmax * 2^X (never
    saturates); OCP X = floor(log2 amax) - e_max, never above round-up X and
    at most one below, saturating exactly the elements above destmax."""
    fmt = LP[name]
    destmax = float(_lp_magnitudes(fmt)[-1])
    emax = math.floor(math.log2(destmax))
    rng = np.random.default_rng(71)
    for _ in range(300):
        v = (rng.standard_normal(32) * 2.0 ** rng.integers(-30, 30)).astype(np.float32)
        amax = float(np.max(np.abs(v)))
        bu, qu, su = oracle.mxlp_block(v, fmt, 0)
        bo, qo, so = oracle.mxlp_block(v, fmt, 1)
        xu, xo = bu - 127, bo - 127
        assert amax <= destmax * 2.0 ** xu and not amax <= destmax * 2.0 ** (xu - 1)
        assert xo == math.floor(math.log2(amax)) - emax
        assert xu - xo in (0, 1) and su == 0
        assert so == int(np.sum(np.abs(v.astype(np.float64)) * 2.0 ** -xo > destmax))
        for c, q in ((xu, qu), (xo, qo)):
            for i in range(32):
                assert q[i] == oracle.lp_encode(fmt, math.ldexp(float(v[i]), -c))


@pytest.mark.parametrize("name", ["e2m1", "e2m3", "e3m2"])
def test_mxlp_exact_blocks_and_special_blocks(name):
    """A block of representable values times 2^X that holds the largest
    code quantizes back to its codes with scale byte X + 127; an all-zero
    block gets byte 0 and +0 codes; Inf or NaN gets 0xFF and +0 codes; a -0
    in a nonzero block keeps its sign."""
    fmt = LP[name]
    n = LP_CODES[fmt]
    rng = np.random.default_rng(72)
    for X in (-100, -3, 0, 5, 90):
        codes = rng.integers(0, 2 * n, size=32)
        codes[7] = n - 1
        v = np.array([oracle.lp_value(fmt, int(c)) * 2.0 ** X for c in codes], np.float32)
        byte, q, _ = oracle.mxlp_block(v, fmt, 0)
        assert byte == X + 127
        np.testing.assert_array_equal([oracle.lp_value(fmt, int(c)) for c in q],
                                      [oracle.lp_value(fmt, int(c)) for c in codes])
    zero = np.zeros(32, np.float32)
    zero[3] = -0.0
    assert oracle.mxlp_block(zero, fmt, 0)[0] == 0 and not oracle.mxlp_block(zero, fmt, 0)[1].any()
    for bad in (np.inf, np.nan):
        v = np.ones(32, np.float32)
        v[9] = bad
        byte, q, _ = oracle.mxlp_block(v, fmt, 1)
        assert byte == 0xFF and not q.any()
    v = np.ones(32, np.float32)
    v[2] = -0.0
    assert oracle.mxlp_block(v, fmt, 0)[1][2] == n


@pytest.mark.parametrize("name", ["e2m1", "e2m3", "e3m2"])
def test_mxlp_quantize_layout(name):
    """Rowwise copy = the blocks of each row (E2M1 two codes per byte, even
    element low); columnwise copy = the rowwise copy of the transpose,
    with a shorter last block when rows % 32 != 0."""
    fmt = LP[name]
    rng = np.random.default_rng(73)
    x = (rng.standard_normal((40, 64)) * np.exp(rng.standard_normal((40, 1)) * 3)).astype(np.float32)
    r = oracle.mxlp_quantize(x, fmt, 3, rule=1)
    for i in range(40):
        for j in range(2):
            byte, q, _ = oracle.mxlp_block(x[i, 32 * j:32 * j + 32], fmt, 1)
            assert r["s_row"][i, j] == byte
            row = r["q_row"][i]
            got = np.stack([row & 0xF, row >> 4], 1).reshape(-1) if fmt == oracle.E2M1 else row
            np.testing.assert_array_equal(got[32 * j:32 * j + 32], q)
    xt = np.ascontiguousarray(np.concatenate([x, np.zeros((24, 64), np.float32)]).T)  # 64 x 64
    rt = oracle.mxlp_quantize(xt, fmt, 1, rule=1)
    np.testing.assert_array_equal(r["s_col"][:, 0], rt["s_row"][:, 0])
    half = 16 if fmt == oracle.E2M1 else 32
    np.testing.assert_array_equal(r["q_col"][:, :half], rt["q_row"][:, :half])
    for c in range(64):  # the last block holds rows 32 .. 39 only
        byte, q, _ = oracle.mxlp_block(x[32:, c], fmt, 1)
        assert r["s_col"][c, 1] == byte


@pytest.mark.parametrize("name", ["e2m1", "e2m3", "e3m2"])
def test_mxlp_rule_boundaries(name):
    """Exact boundaries: an amax that is a power of two 2^k gets OCP X =
    k - e_max; an amax exactly on destmax * 2^X sits on the maximum code
    under both rules and is not counted as saturated."""
    fmt = LP[name]
    destmax = float(_lp_magnitudes(fmt)[-1])
    emax = math.floor(math.log2(destmax))
    for k in (-20, 0, 3, 17):
        v = np.full(32, 2.0 ** (k - 3), np.float32)
        v[11] = -(2.0 ** k)
        byte, q, sat = oracle.mxlp_block(v, fmt, 1)
        assert byte - 127 == k - emax and sat == 0
        assert oracle.lp_value(fmt, int(q[11])) == -(2.0 ** emax)
    for X in (-5, 0, 9):
        v = np.full(32, destmax * 2.0 ** (X - 2), np.float32)
        v[4] = destmax * 2.0 ** X
        for rule in (0, 1):
            byte, q, sat = oracle.mxlp_block(v, fmt, rule)
            assert byte - 127 == X and sat == 0
            assert oracle.lp_value(fmt, int(q[4])) == destmax


# --------------------------------------------------------------------------
# Block-scale layout for tensor-core MMA (not on the pages: NVIDIA's public
# 128 x 4 block layout; parity unpinned by the pages)
# --------------------------------------------------------------------------
def _mma_layout_by_reshape(s, scale_cols):
    """The same layout described another way: pad to 128 x 4 blocks; in a
    block, 16-byte row j holds the four scales of rows j, j + 32, j + 64,
    j + 96 in that order; blocks follow each other along a block row."""
    rows = s.shape[0]
    R, C = -(-rows // 128) * 128, -(-scale_cols // 4) * 4
    pad = np.zeros((R, C), np.uint8)
    pad[:rows, :scale_cols] = s[:, :scale_cols]
    blocks = pad.reshape(R // 128, 128, C // 4, 4).transpose(0, 2, 1, 3)     # [br][bc][128][4]
    inner = blocks.reshape(R // 128, C // 4, 4, 32, 4).transpose(0, 1, 3, 2, 4)  # [br][bc][j][r//32][c]
    return inner.reshape(-1)


@pytest.mark.parametrize("rows,scale_cols,s_ld", [(128, 4, 4), (300, 7, 7), (1, 1, 3), (257, 256, 260)])
def test_mma_scale_layout(rows, scale_cols, s_ld):
    rng = np.random.default_rng(81)
    s = rng.integers(1, 256, size=(rows, s_ld), dtype=np.uint64).astype(np.uint8)
    got = oracle.mma_scale_layout(s, scale_cols)
    np.testing.assert_array_equal(got, _mma_layout_by_reshape(s, scale_cols))
    # every real scale appears once, padding is zero
    assert np.count_nonzero(got) == rows * scale_cols
    assert sorted(got[got != 0].tolist()) == sorted(s[:, :scale_cols].reshape(-1).tolist())
