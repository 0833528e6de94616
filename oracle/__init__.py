"""CPU oracle for FP8 / MXFP8 quantization -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never does, and
this package never imports the product library: the two share no code.

The arithmetic lives in ``oracle.c`` (plain C, compiled here with gcc on
first use).  This module marshals numpy arrays into it and holds the one
piece of logic that is control flow rather than arithmetic: the
delayed-scaling state machine, written in the order the pages give it
("HiFloat8：高性能训练之路" 1.2 and 3; "混合精度与 FP8 训练" 8.2).

Inputs: BF16 tensors are numpy ``uint16`` arrays of raw BF16 bits, FP32
tensors are numpy ``float32`` arrays.  2-D tensors are row-major.

Parity unpinned by the pages (our own readings, pinned only by this
definition and the tests): the NaN output byte 0x7F, the MX non-finite
block (scale 0xFF, elements 0x7F), and the per-tensor special cases
(amax 0 -> scale 1; non-finite amax -> scale 1 plus a flag; an
overflowing quotient -> FLT_MAX).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

E4M3 = 0
E5M2 = 1
E2M1 = 2  # MXFP4 elements
E2M3 = 3  # MXFP6 elements (OCP reading)
E3M2 = 4  # MXFP6 elements (OCP reading)
BF16 = 0
FP32 = 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (plain gcc, no fast-math)."""
    with _lock:
        stale = (not os.path.exists(_LIB_PATH)) or (
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
        if force or stale:
            tmp = _LIB_PATH + f".tmp{os.getpid()}"
            cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
                   "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB_PATH)
    c = ctypes
    P = c.c_void_p
    sig = {
        "orc_fp8_value": (c.c_double, [c.c_int, c.c_uint]),
        "orc_fp8_max_code": (c.c_uint, [c.c_int]),
        "orc_fp8_max": (c.c_double, [c.c_int]),
        "orc_fp8_encode": (c.c_uint, [c.c_int, c.c_double]),
        "orc_amax_bits": (c.c_uint32, [P, c.c_int, c.c_int64, c.c_int64]),
        "orc_per_tensor_scale": (c.c_float, [c.c_uint32, c.c_int, c.c_int, c.POINTER(c.c_int)]),
        "orc_reciprocal": (c.c_float, [c.c_float]),
        "orc_cast": (None, [P, c.c_int, c.c_int64, c.c_int64, c.c_float, c.c_int, P,
                            c.POINTER(c.c_uint64), c.c_int]),
        "orc_mx_block": (c.c_uint8, [P, c.c_int, c.c_int, P]),
        "orc_mx_col_blocks": (c.c_int64, [P, c.c_int, c.c_int64]),
        "orc_mx_quantize": (None, [P, c.c_int, c.c_int64, c.c_int64, P, c.c_int, c.c_int,
                                   c.c_int, P, P, P, P, c.c_int64, c.c_int]),
        "orc_encode_array": (None, [c.c_int, P, c.c_int64, P, c.c_int]),
        "orc_encode_f32_range": (None, [c.c_int, c.c_uint64, c.c_int64, P, c.c_int]),
        "orc_max_threads": (c.c_int, []),
        "orc_bf16_round": (c.c_uint16, [c.c_float]),
        "orc_pow2_floor": (c.c_float, [c.c_float]),
        "orc_e2m1_value": (c.c_double, [c.c_uint]),
        "orc_e2m1_encode": (c.c_uint, [c.c_double]),
        "orc_nvfp4_tensor_scale": (c.c_float, [c.c_uint32]),
        "orc_nvfp4_block": (c.c_uint8, [P, c.c_int, c.c_float, P]),
        "orc_nvfp4": (None, [P, c.c_int, c.c_int64, c.c_int64, P, P, P, c.c_int]),
        "orc_blockwise": (None, [P, c.c_int, c.c_int64, c.c_int64, c.c_int, c.c_int, c.c_int, c.c_int, P, P,
                                 c.c_int]),
        "orc_mx_block_rule": (c.c_uint8, [P, c.c_int, c.c_int, c.c_int, P, c.POINTER(c.c_int64)]),
        "orc_mx_quantize_rule": (None, [P, c.c_int, c.c_int64, c.c_int64, P, c.c_int, c.c_int, c.c_int, c.c_int,
                                        P, P, P, P, c.c_int64, P, c.c_int]),
        "orc_bf16_round_array": (None, [P, c.c_int64, P, c.c_int]),
        "orc_dequant_per_tensor": (None, [P, c.c_int64, c.c_int64, P, c.c_int, c.c_int, P, c.c_int, P,
                                          c.c_int]),
        "orc_mx_dequantize": (None, [P, P, c.c_int64, c.c_int64, P, c.c_int, c.c_int, c.c_int, c.c_int64,
                                     c.c_int, P, c.c_int]),
        "orc_lp_value": (c.c_double, [c.c_int, c.c_uint]),
        "orc_lp_encode": (c.c_uint, [c.c_int, c.c_double]),
        "orc_mxlp_block": (c.c_uint8, [P, c.c_int, c.c_int, c.c_int, P, c.POINTER(c.c_int64)]),
        "orc_mxlp_quantize": (None, [P, c.c_int, c.c_int64, c.c_int64, c.c_int, c.c_int, c.c_int, P, P, P, P, P]),
        "orc_mma_scale_layout": (None, [P, c.c_int64, c.c_int64, c.c_int64, P]),
        "orc_qstats_per_tensor": (None, [P, c.c_int, c.c_int64, c.c_int64, P, c.c_int, c.c_int, P, P, P, P]),
        "orc_qstats_mx": (None, [P, c.c_int, c.c_int64, c.c_int64, P, c.c_int, c.c_int, c.c_int, P, P,
                                 c.c_int64, P, P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def max_threads() -> int:
    return int(_load().orc_max_threads())


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data) if a is not None else None


def _dtype_code(x: np.ndarray) -> int:
    if x.dtype == np.uint16:
        return BF16
    if x.dtype == np.float32:
        return FP32
    raise TypeError("oracle inputs are uint16 (BF16 bits) or float32")


# --------------------------------------------------------------------------
# Scalars
# --------------------------------------------------------------------------
def fp8_value(fmt: int, code: int) -> float:
    """Value of an E4M3/E5M2 code ("混合精度与 FP8 训练" 2.1-2.2)."""
    return float(_load().orc_fp8_value(fmt, code))


def fp8_max(fmt: int) -> float:
    return float(_load().orc_fp8_max(fmt))


def fp8_max_code(fmt: int) -> int:
    return int(_load().orc_fp8_max_code(fmt))


def fp8_encode(fmt: int, a: float) -> int:
    """Saturating RNE of the exact value ``a`` ("混合精度与 FP8 训练" 4.1, 8.1)."""
    return int(_load().orc_fp8_encode(fmt, float(a)))


def encode_array(fmt: int, a: np.ndarray, nthreads: int = 0) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.float64)
    q = np.empty(a.shape, dtype=np.uint8)
    _load().orc_encode_array(fmt, _ptr(a), a.size, _ptr(q), nthreads or max_threads())
    return q


def encode_f32_range(fmt: int, first: int, n: int, nthreads: int = 0) -> np.ndarray:
    """Codes of the FP32 bit patterns first .. first+n-1 (scale 1)."""
    q = np.empty(n, dtype=np.uint8)
    _load().orc_encode_f32_range(fmt, first, n, _ptr(q), nthreads or max_threads())
    return q


def bits_to_f32(bits: int) -> np.float32:
    return np.array([bits], dtype=np.uint32).view(np.float32)[0]


def f32_to_bits(f) -> int:
    return int(np.array([f], dtype=np.float32).view(np.uint32)[0])


# --------------------------------------------------------------------------
# Per-tensor scaling
# --------------------------------------------------------------------------
def amax_bits(x: np.ndarray, begin: int = 0, end: int | None = None) -> int:
    """FP32 bits of max |x| over the flat range [begin, end)."""
    x = np.ascontiguousarray(x)
    end = x.size if end is None else end
    return int(_load().orc_amax_bits(_ptr(x), _dtype_code(x), begin, end))


def amax(x: np.ndarray, begin: int = 0, end: int | None = None) -> np.float32:
    return bits_to_f32(amax_bits(x, begin, end))


def per_tensor_scale(amax_value_bits: int, fmt: int, margin: int) -> tuple[np.float32, bool]:
    """Scale = fl32(fl32(F8max/amax) * 2^-margin) with the special cases."""
    nf = ctypes.c_int(0)
    s = _load().orc_per_tensor_scale(amax_value_bits, fmt, margin, ctypes.byref(nf))
    return np.float32(s), bool(nf.value)


def reciprocal(s) -> np.float32:
    return np.float32(_load().orc_reciprocal(float(s)))


def cast(x: np.ndarray, scale, fmt: int, begin: int = 0, end: int | None = None,
         out: np.ndarray | None = None, nthreads: int = 0) -> tuple[np.ndarray, int]:
    """q = RNE_sat(fl32(x * scale)) over the flat range; returns (q, sat_count)."""
    x = np.ascontiguousarray(x)
    end = x.size if end is None else end
    q = np.zeros(x.size, dtype=np.uint8) if out is None else out
    sat = ctypes.c_uint64(0)
    _load().orc_cast(_ptr(x), _dtype_code(x), begin, end, float(np.float32(scale)), fmt,
                     _ptr(q), ctypes.byref(sat), nthreads or max_threads())
    return q, int(sat.value)


def _group_bounds(rows: int, offsets) -> list[tuple[int, int]]:
    if offsets is None:
        return [(0, rows)]
    o = [int(v) for v in offsets]
    return [(o[g], o[g + 1]) for g in range(len(o) - 1)]


def current_scaling(x: np.ndarray, fmt: int, margin: int = 0, offsets=None,
                    nthreads: int = 0) -> dict:
    """Per-tensor (or per-group) current scaling of a 2-D tensor.

    For each group of rows: amax, scale (eq. 1 of "HiFloat8：高性能训练之路"
    1.2, times 2^-margin), cast (eq. 2).  Returns q (flat), and per group
    amax / scale / scale_inv (float32), sat (int) and the non-finite flag.
    """
    rows, cols = x.shape
    flat = np.ascontiguousarray(x).reshape(-1)
    q = np.zeros(flat.size, dtype=np.uint8)
    res = {"q": q, "amax": [], "scale": [], "scale_inv": [], "sat": [], "nonfinite": []}
    for r0, r1 in _group_bounds(rows, offsets):
        a = amax_bits(flat, r0 * cols, r1 * cols)
        s, nf = per_tensor_scale(a, fmt, margin)
        _, sat = cast(flat, s, fmt, r0 * cols, r1 * cols, out=q, nthreads=nthreads)
        res["amax"].append(bits_to_f32(a))
        res["scale"].append(s)
        res["scale_inv"].append(reciprocal(s))
        res["sat"].append(sat)
        res["nonfinite"].append(nf)
    for k in ("amax", "scale", "scale_inv"):
        res[k] = np.array(res[k], dtype=np.float32)
    res["sat"] = np.array(res["sat"], dtype=np.uint64)
    return res


class DelayedScaling:
    """Delayed per-tensor scaling, the state machine of the pages.

    "HiFloat8：高性能训练之路" 1.2: an amax history buffer of fixed length;
    the scale uses the max over the history (eqs. 3-4, with 2^-N); every
    Interval steps the true amax of the current tensor is computed and
    appended, dropping the oldest entry once the buffer is full.  Section 3
    of the same page fixes the timing for Interval = 1: step 0 computes the
    amax, step 1 scales with it and then records its own, and so on.
    Section 5.2 (and "昇腾 950" 3.2): the first step after a (re)start has
    no history, so it uses current scaling.

    Readings where the pages are silent: a step records iff step % interval == 0,
    counting from creation or reset; the first step uses margin 0; the max
    runs over the filled entries only.
    """

    def __init__(self, history_len: int, interval: int, margin: int, fmt: int):
        self.H, self.interval, self.margin, self.fmt = history_len, interval, margin, fmt
        self.reset()

    def reset(self):
        self.hist = [np.float32(0.0)] * self.H
        self.head = 0
        self.count = 0
        self.step_no = 0
        self.nonfinite = False

    def _history_max_bits(self) -> int:
        return max(f32_to_bits(v) & 0x7FFFFFFF for v in self.hist[: self.count])

    def step(self, x: np.ndarray, nthreads: int = 0) -> dict:
        flat = np.ascontiguousarray(x).reshape(-1)
        recorded_amax = None
        if self.count == 0:
            a = amax_bits(flat)  # current scaling on the first step
            scale, nf = per_tensor_scale(a, self.fmt, 0)
            recorded_amax = a
        else:
            scale, nf = per_tensor_scale(self._history_max_bits(), self.fmt, self.margin)
        if nf:
            self.nonfinite = True
        q, sat = cast(flat, scale, self.fmt, nthreads=nthreads)
        recording = (self.step_no % self.interval) == 0
        if recording:
            if recorded_amax is None:
                recorded_amax = amax_bits(flat)
            if (recorded_amax & 0x7FFFFFFF) >= 0x7F800000:
                self.nonfinite = True
            self.hist[self.head] = bits_to_f32(recorded_amax)
            self.head = (self.head + 1) % self.H
            self.count = min(self.count + 1, self.H)
        self.step_no += 1
        return {"q": q, "scale": scale, "scale_inv": reciprocal(scale), "sat": sat,
                "amax": bits_to_f32(recorded_amax) if recording else None,
                "recorded": recording}


# --------------------------------------------------------------------------
# MXFP8
# --------------------------------------------------------------------------
def mx_block(values: np.ndarray, fmt: int) -> tuple[int, np.ndarray]:
    """One MX block of k <= 32 float32 values -> (scale byte, codes)."""
    v = np.ascontiguousarray(values, dtype=np.float32)
    q = np.zeros(v.size, dtype=np.uint8)
    b = _load().orc_mx_block(_ptr(v), v.size, fmt, _ptr(q))
    return int(b), q


MX_RULE_UP, MX_RULE_OCP = 0, 1


def mx_block_rule(values: np.ndarray, fmt: int, rule: int) -> tuple[int, np.ndarray, int]:
    """One MX block under a scale rule -> (scale byte, codes, saturated count)."""
    v = np.ascontiguousarray(values, dtype=np.float32)
    q = np.zeros(v.size, dtype=np.uint8)
    n = ctypes.c_int64(0)
    b = _load().orc_mx_block_rule(_ptr(v), v.size, fmt, rule, _ptr(q), ctypes.byref(n))
    return int(b), q, int(n.value)


def mx_col_blocks(rows: int, offsets=None) -> int:
    """sum over groups of ceil(n_g / 32) (one group when offsets is None)."""
    if offsets is None:
        return (rows + 31) // 32
    o = np.ascontiguousarray(offsets, dtype=np.int64)
    return int(_load().orc_mx_col_blocks(_ptr(o), o.size - 1, rows))


def mx_quantize(x: np.ndarray, fmt: int, direction: int = 3, offsets=None,
                s_col_ld: int | None = None, nthreads: int = 0) -> dict:
    """MX quantization of a 2-D tensor (rows x cols, cols % 32 == 0).

    direction: 1 rowwise, 2 columnwise, 3 both.  Returns q_row [rows, cols],
    s_row [rows, cols/32], q_col [cols, rows] (the transpose), s_col
    [cols, s_col_ld] with the first mx_col_blocks() entries of each row used.
    """
    x = np.ascontiguousarray(x)
    rows, cols = x.shape
    assert cols % 32 == 0
    G = 1 if offsets is None else len(offsets) - 1
    o = None if offsets is None else np.ascontiguousarray(offsets, dtype=np.int64)
    T = mx_col_blocks(rows, o)
    ld = T if s_col_ld is None else s_col_ld
    q_row = np.zeros((rows, cols), np.uint8) if direction & 1 else None
    s_row = np.zeros((rows, cols // 32), np.uint8) if direction & 1 else None
    q_col = np.zeros((cols, rows), np.uint8) if direction & 2 else None
    s_col = np.zeros((cols, max(ld, 1)), np.uint8) if direction & 2 else None
    dummy = np.zeros(1, np.uint8)
    _load().orc_mx_quantize(
        _ptr(x), _dtype_code(x), rows, cols, _ptr(o) if o is not None else None, G, fmt,
        direction,
        _ptr(q_row if q_row is not None else dummy), _ptr(s_row if s_row is not None else dummy),
        _ptr(q_col if q_col is not None else dummy), _ptr(s_col if s_col is not None else dummy),
        ld, nthreads or max_threads())
    return {"q_row": q_row, "s_row": s_row, "q_col": q_col, "s_col": s_col, "col_blocks": T}


def mx_quantize_rule(x: np.ndarray, fmt: int, direction: int, rule: int, offsets=None,
                     s_col_ld: int | None = None, nthreads: int = 0) -> dict:
    """mx_quantize under a scale rule (MX_RULE_UP or MX_RULE_OCP), plus
    'sat': the saturated-element counts [rowwise, columnwise]."""
    x = np.ascontiguousarray(x)
    rows, cols = x.shape
    assert cols % 32 == 0
    G = 1 if offsets is None else len(offsets) - 1
    o = None if offsets is None else np.ascontiguousarray(offsets, dtype=np.int64)
    T = mx_col_blocks(rows, o)
    ld = T if s_col_ld is None else s_col_ld
    q_row = np.zeros((rows, cols), np.uint8) if direction & 1 else None
    s_row = np.zeros((rows, cols // 32), np.uint8) if direction & 1 else None
    q_col = np.zeros((cols, rows), np.uint8) if direction & 2 else None
    s_col = np.zeros((cols, max(ld, 1)), np.uint8) if direction & 2 else None
    sat = np.zeros(2, np.int64)
    dummy = np.zeros(1, np.uint8)
    _load().orc_mx_quantize_rule(
        _ptr(x), _dtype_code(x), rows, cols, _ptr(o) if o is not None else None, G, fmt, direction, rule,
        _ptr(q_row if q_row is not None else dummy), _ptr(s_row if s_row is not None else dummy),
        _ptr(q_col if q_col is not None else dummy), _ptr(s_col if s_col is not None else dummy),
        ld, _ptr(sat), nthreads or max_threads())
    return {"q_row": q_row, "s_row": s_row, "q_col": q_col, "s_col": s_col, "col_blocks": T,
            "sat": [int(sat[0]), int(sat[1])]}


# --------------------------------------------------------------------------
# Dequantization
# --------------------------------------------------------------------------
def bf16_round(f) -> np.ndarray:
    """Nearest BF16 bit patterns (ties to even, NaN -> 0x7FC0) of float32 values."""
    f = np.ascontiguousarray(np.asarray(f, dtype=np.float32).reshape(-1))
    out = np.zeros(f.size, dtype=np.uint16)
    _load().orc_bf16_round_array(_ptr(f), f.size, _ptr(out), max_threads())
    return out


def _out_array(n: int, out_dt: int) -> np.ndarray:
    return np.zeros(n, dtype=np.uint16 if out_dt == 0 else np.uint32)


def dequant_per_tensor(q: np.ndarray, fmt: int, scale_inv, out_dt: int = 0, offsets=None,
                       nthreads: int = 0) -> np.ndarray:
    """y = round_out(fl32(value(q) * scale_inv[g])) over a 2-D code array.

    out_dt 0: BF16 bit patterns (uint16), 1: FP32 bit patterns (uint32);
    the result has q's shape.
    """
    q = np.ascontiguousarray(q, dtype=np.uint8)
    rows, cols = q.shape
    o = None if offsets is None else np.ascontiguousarray(offsets, dtype=np.int64)
    G = 1 if o is None else o.size - 1
    si = np.ascontiguousarray(np.asarray(scale_inv, dtype=np.float32).reshape(-1))
    assert si.size == G
    y = _out_array(q.size, out_dt)
    _load().orc_dequant_per_tensor(_ptr(q), rows, cols, _ptr(o) if o is not None else None, G, fmt, _ptr(si),
                                   out_dt, _ptr(y), nthreads or max_threads())
    return y.reshape(rows, cols)


def mx_dequantize(q: np.ndarray, s: np.ndarray, fmt: int, direction: int, rows: int, cols: int,
                  out_dt: int = 0, offsets=None, nthreads: int = 0) -> np.ndarray:
    """MX dequantization of one copy: value(q) * 2^(s - 127), byte 0xFF -> NaN.

    direction 1: q [rows, cols], s [rows, cols/32] -> y [rows, cols].
    direction 2: q [cols, rows], s [cols, s_ld] -> y [cols, rows].
    """
    q = np.ascontiguousarray(q, dtype=np.uint8)
    s = np.ascontiguousarray(s, dtype=np.uint8)
    o = None if offsets is None else np.ascontiguousarray(offsets, dtype=np.int64)
    G = 1 if o is None else o.size - 1
    s_ld = s.shape[1]
    y = _out_array(q.size, out_dt)
    _load().orc_mx_dequantize(_ptr(q), _ptr(s), rows, cols, _ptr(o) if o is not None else None, G, fmt,
                              direction, s_ld, out_dt, _ptr(y), nthreads or max_threads())
    return y.reshape(q.shape)


# --------------------------------------------------------------------------
# MXFP4 / MXFP6 (E2M1, E2M3, E3M2 elements with E8M0 block scales)
# --------------------------------------------------------------------------
def lp_value(fmt: int, code: int) -> float:
    """Value of an E2M1 / E2M3 / E3M2 code from its fields."""
    return float(_load().orc_lp_value(fmt, code))


def lp_encode(fmt: int, a: float) -> int:
    """Nearest E2M1 / E2M3 / E3M2 code (ties to even), saturating."""
    return int(_load().orc_lp_encode(fmt, float(a)))


def mxlp_block(values: np.ndarray, fmt: int, rule: int) -> tuple[int, np.ndarray, int]:
    """(scale byte, codes, saturated count) of one MX block of <= 32 values."""
    v = np.ascontiguousarray(values, dtype=np.float32).reshape(-1)
    q = np.zeros(v.size, dtype=np.uint8)
    sat = ctypes.c_int64(0)
    b = _load().orc_mxlp_block(_ptr(v), v.size, fmt, rule, _ptr(q), ctypes.byref(sat))
    return int(b), q, int(sat.value)


def mxlp_quantize(x: np.ndarray, fmt: int, direction: int = 3, rule: int = 0) -> dict:
    """MXFP4 (E2M1, two codes per byte, even element low) or MXFP6 (E2M3 /
    E3M2, one code per byte) of a 2-D tensor, rowwise and/or columnwise."""
    x = np.ascontiguousarray(x)
    rows, cols = x.shape
    fp4 = fmt == E2M1
    nb = (rows + 31) // 32
    out = {"q_row": np.zeros((rows, cols // 2 if fp4 else cols), np.uint8),
           "s_row": np.zeros((rows, cols // 32), np.uint8),
           "q_col": np.zeros((cols, rows // 2 if fp4 else rows), np.uint8),
           "s_col": np.zeros((cols, nb), np.uint8)}
    sat = np.zeros(2, dtype=np.int64)
    _load().orc_mxlp_quantize(_ptr(x), _dtype_code(x), rows, cols, fmt, direction, rule, _ptr(out["q_row"]),
                              _ptr(out["s_row"]), _ptr(out["q_col"]), _ptr(out["s_col"]), _ptr(sat))
    out["sat"] = sat.tolist()
    return out


# --------------------------------------------------------------------------
# Block-scale layout for block-scaled tensor-core MMA
# --------------------------------------------------------------------------
def mma_scale_layout(s: np.ndarray, scale_cols: int | None = None) -> np.ndarray:
    """A [rows, s_ld] scale array (the first scale_cols columns used) in
    the 128 x 4 block layout: a flat uint8 array of ceil(rows/128)*128 *
    ceil(scale_cols/4)*4 bytes."""
    s = np.ascontiguousarray(s, dtype=np.uint8)
    rows, s_ld = s.shape
    sc = s_ld if scale_cols is None else scale_cols
    out = np.zeros(((rows + 127) // 128 * 128) * ((sc + 3) // 4 * 4), dtype=np.uint8)
    _load().orc_mma_scale_layout(_ptr(s), rows, sc, s_ld, _ptr(out))
    return out


# --------------------------------------------------------------------------
# Quantization-error statistics (SQNR, zero-rate)
# --------------------------------------------------------------------------
def _stats_dict(sums: np.ndarray, counts: np.ndarray) -> dict:
    return {"signal": float(sums[0]), "noise": float(sums[1]), "n": int(counts[0]), "n_zero": int(counts[1]),
            "n_flushed": int(counts[2]), "n_nonfinite": int(counts[3])}


def qstats_per_tensor(x: np.ndarray, q: np.ndarray, fmt: int, scale_inv, offsets=None) -> dict:
    """Statistics of a per-tensor (per-group) copy q of x against x, with
    xh = fl32(value(q) * scale_inv[g]): signal = sum x^2 and noise =
    sum (x - xh)^2 over the elements where both are finite (double sums),
    n, n_zero (xh == 0), n_flushed (xh == 0, x != 0), n_nonfinite."""
    x = np.ascontiguousarray(x)
    rows, cols = x.shape
    q = np.ascontiguousarray(q, dtype=np.uint8).reshape(-1)
    assert q.size == x.size
    o = None if offsets is None else np.ascontiguousarray(offsets, dtype=np.int64)
    G = 1 if o is None else o.size - 1
    si = np.ascontiguousarray(np.asarray(scale_inv, dtype=np.float32).reshape(-1))
    assert si.size == G
    sums = np.zeros(2, dtype=np.float64)
    counts = np.zeros(4, dtype=np.int64)
    _load().orc_qstats_per_tensor(_ptr(x), _dtype_code(x), rows, cols, _ptr(o) if o is not None else None, G, fmt,
                                  _ptr(q), _ptr(si), _ptr(sums), _ptr(counts))
    return _stats_dict(sums, counts)


def qstats_mx(x: np.ndarray, q: np.ndarray, s: np.ndarray, fmt: int, direction: int, offsets=None) -> dict:
    """The statistics of qstats_per_tensor for one MX copy of x, xh =
    value(q) * 2^(s - 127) rounded to FP32 (byte 0xFF: NaN).  direction 1:
    q [rows, cols], s [rows, cols/32]; direction 2: q [cols, rows], s
    [cols, s_ld] with the column blocks of all groups in order."""
    x = np.ascontiguousarray(x)
    rows, cols = x.shape
    q = np.ascontiguousarray(q, dtype=np.uint8)
    s = np.ascontiguousarray(s, dtype=np.uint8)
    o = None if offsets is None else np.ascontiguousarray(offsets, dtype=np.int64)
    G = 1 if o is None else o.size - 1
    sums = np.zeros(2, dtype=np.float64)
    counts = np.zeros(4, dtype=np.int64)
    _load().orc_qstats_mx(_ptr(x), _dtype_code(x), rows, cols, _ptr(o) if o is not None else None, G, fmt,
                          direction, _ptr(q), _ptr(s), s.shape[1] if s.ndim == 2 else 0, _ptr(sums), _ptr(counts))
    return _stats_dict(sums, counts)


def sqnr_db(stats: dict) -> float:
    """10 log10(signal / noise); +inf for an exact copy of a nonzero signal."""
    if stats["noise"] == 0.0:
        return float("inf") if stats["signal"] > 0 else float("nan")
    return 10.0 * np.log10(stats["signal"] / stats["noise"])


def zero_rate(stats: dict) -> float:
    """The share of the compared elements whose quantized value is 0 while
    the input is not ("昇腾 Ascend 950 低精度格式", appendix 3.4, compares
    formats by it without defining it): n_flushed / n, 0 for an empty
    tensor."""
    return stats["n_flushed"] / stats["n"] if stats["n"] else 0.0


# --------------------------------------------------------------------------
# Blockwise FP8 (1x128, 128x1, 128x128 groups with FP32 scales)
# --------------------------------------------------------------------------
def pow2_floor(s: float) -> np.float32:
    """The largest power of two not above a positive float."""
    return np.float32(_load().orc_pow2_floor(float(s)))


def blockwise(x: np.ndarray, fmt: int, group: tuple[int, int], pow2: bool = False,
              nthreads: int = 0) -> tuple[np.ndarray, np.ndarray]:
    """Blockwise quantization of a 2-D tensor with (gr, gc) groups.

    Returns (q [rows, cols] uint8 in x's layout, scale_inv float32
    [ceil(rows/gr), ceil(cols/gc)]).
    """
    x = np.ascontiguousarray(x)
    rows, cols = x.shape
    gr, gc = group
    q = np.zeros((rows, cols), np.uint8)
    si = np.zeros(((rows + gr - 1) // gr, (cols + gc - 1) // gc), np.float32)
    _load().orc_blockwise(_ptr(x), _dtype_code(x), rows, cols, fmt, gr, gc, int(pow2), _ptr(q), _ptr(si),
                          nthreads or max_threads())
    return q, si


# --------------------------------------------------------------------------
# NVFP4 (E2M1 elements, E4M3 scale per 16, FP32 tensor scale)
# --------------------------------------------------------------------------
def e2m1_value(code: int) -> float:
    return float(_load().orc_e2m1_value(code))


def e2m1_encode(a: float) -> int:
    return int(_load().orc_e2m1_encode(float(a)))


def nvfp4_tensor_scale(amax_value_bits: int) -> np.float32:
    return np.float32(_load().orc_nvfp4_tensor_scale(amax_value_bits))


def nvfp4_block(values: np.ndarray, S: float) -> tuple[int, np.ndarray]:
    """One block (k <= 16 float32 values) under tensor scale S -> (E4M3 scale code, E2M1 codes)."""
    v = np.ascontiguousarray(values, dtype=np.float32)
    q = np.zeros(v.size, dtype=np.uint8)
    c = _load().orc_nvfp4_block(_ptr(v), v.size, float(np.float32(S)), _ptr(q))
    return int(c), q


def nvfp4(x: np.ndarray, nthreads: int = 0) -> dict:
    """NVFP4 of a 2-D tensor (cols % 16 == 0): q [rows, cols/2] (packed, even
    element in the low nibble), s [rows, cols/16] E4M3 codes, S the tensor scale."""
    x = np.ascontiguousarray(x)
    rows, cols = x.shape
    assert cols % 16 == 0
    q = np.zeros((rows, cols // 2), np.uint8)
    s = np.zeros((rows, cols // 16), np.uint8)
    S = ctypes.c_float(0)
    _load().orc_nvfp4(_ptr(x), _dtype_code(x), rows, cols, _ptr(q), _ptr(s), ctypes.byref(S), nthreads or max_threads())
    return {"q": q, "s": s, "S": np.float32(S.value)}
