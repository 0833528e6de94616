"""Python binding of libfp8q: FP8 / MXFP8 quantization kernels for GB300.

Thin ctypes marshalling over the C ABI declared in include/fp8q.h: every
function takes torch CUDA tensors, checks shapes and dtypes, allocates the
outputs with torch and calls the entry point of the same name on the
current CUDA stream.  All arithmetic runs in the library's kernels; there is
no fallback.  If libfp8q.so is missing, importing this package still works
but every call raises until ``build()`` has been run.

Formats: ``E4M3`` (max 448) and ``E5M2`` (max 57344).  Outputs are uint8
tensors of raw codes; ``view(torch.float8_e4m3fn)`` / ``float8_e5m2``
reinterprets them for torch.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

from ._build import LIB_PATH, build as _build_lib, is_stale

__all__ = [
    "E4M3", "E5M2", "ROW", "COL", "BOTH", "build", "library_path", "lib",
    "fp8q_amax", "fp8q_cast_per_tensor", "fp8q_cast_workspace_bytes", "DelayedScaling",
    "mxfp8_quantize", "mxfp8_col_blocks", "Fp8qError", "check_device", "set_wait_budget_ns",
    "fp8q_scale_from_amax", "debug_stall_mx_producer", "debug_stall_scale_publish", "fp8q_dequantize_per_tensor", "mxfp8_dequantize",
    "RULE_UP", "RULE_OCP", "BLOCK_1X128", "BLOCK_128X128", "fp8q_quantize_blockwise", "fp8q_quantize_nvfp4",
    "fp8q_qstats_workspace_bytes", "fp8q_qstats_per_tensor", "mxfp8_qstats", "qstats_dict",
    "E2M1", "E2M3", "E3M2", "mx_quantize_fp4_fp6", "mx_scales_to_mma_layout",
    "SCALES_ROW_MAJOR", "SCALES_MMA", "mxfp8_mma_scale_bytes",
]

E4M3 = 0
E5M2 = 1
E2M1 = 2  # MXFP4 elements
E2M3 = 3  # MXFP6 elements
E3M2 = 4  # MXFP6 elements
ROW = 1
COL = 2
BOTH = 3
MAX_GROUPS = 4096
SCALES_ROW_MAJOR = 0  # MX scale layouts (mxfp8_quantize scale_layout)
SCALES_MMA = 1        # the 128 x 4 blocks of block-scaled tensor-core MMA
RULE_UP = 0   # MX scale rule: X = ceil(log2(amax / destmax))
RULE_OCP = 1  # MX scale rule: X = floor(log2(amax)) - e_max (can saturate)
BLOCK_1X128 = 1      # blockwise groups: 1x128 (rowwise copy) / 128x1 (transposed copy)
BLOCK_128X128 = 128  # blockwise groups: 128x128 blocks

_c = ctypes
_P = _c.c_void_p
_SIGS = {
    "fp8q_version": (_c.c_int32, []),
    "fp8q_last_error_string": (_c.c_char_p, []),
    "fp8q_check_device": (_c.c_int, [_P]),
    "fp8q_debug_stall_mx_producer": (_c.c_int, [_c.c_int32]),
    "fp8q_debug_stall_scale_publish": (_c.c_int, [_c.c_int32]),
    "fp8q_scale_from_amax": (_c.c_int, [_P, _c.c_int32, _c.c_int32, _c.c_int32, _P, _P, _P]),
    "mxfp8_quantize_rule": (_c.c_int, [_P, _c.c_int32, _c.c_int64, _c.c_int64, _P, _c.c_int32, _c.c_int32,
                                       _c.c_int32, _c.c_int32, _P, _P, _P, _P, _c.c_int64, _P, _P]),
    "mxfp8_quantize_ex": (_c.c_int, [_P, _c.c_int32, _c.c_int64, _c.c_int64, _P, _c.c_int32, _c.c_int32,
                                     _c.c_int32, _c.c_int32, _c.c_int32, _P, _P, _P, _P, _c.c_int64, _P, _P]),
    "mxfp8_mma_scale_bytes": (_c.c_int64, [_c.c_int64, _c.c_int64]),
    "fp8q_quantize_blockwise": (_c.c_int, [_P, _c.c_int32, _c.c_int64, _c.c_int64, _c.c_int32, _c.c_int32,
                                           _c.c_int32, _c.c_int32, _P, _P, _P, _P, _P]),
    "fp8q_quantize_nvfp4": (_c.c_int, [_P, _c.c_int32, _c.c_int64, _c.c_int64, _P, _P, _P, _P, _P]),
    "fp8q_dequantize_per_tensor": (_c.c_int, [_P, _c.c_int64, _c.c_int64, _P, _c.c_int32, _c.c_int32, _P,
                                              _c.c_int32, _P, _P]),
    "mxfp8_dequantize": (_c.c_int, [_P, _P, _c.c_int64, _c.c_int64, _P, _c.c_int32, _c.c_int32, _c.c_int32,
                                    _c.c_int64, _c.c_int32, _P, _P]),
    "mx_quantize_fp4_fp6": (_c.c_int, [_P, _c.c_int32, _c.c_int64, _c.c_int64, _c.c_int32, _c.c_int32, _c.c_int32,
                                       _P, _P, _P, _P, _P, _P]),
    "mx_scales_to_mma_layout": (_c.c_int, [_P, _c.c_int64, _c.c_int64, _c.c_int64, _P, _P]),
    "fp8q_qstats_workspace_bytes": (_c.c_size_t, []),
    "fp8q_qstats_per_tensor": (_c.c_int, [_P, _c.c_int32, _c.c_int64, _c.c_int64, _P, _c.c_int32, _c.c_int32,
                                          _P, _P, _P, _P, _c.c_size_t, _P]),
    "mxfp8_qstats": (_c.c_int, [_P, _c.c_int32, _c.c_int64, _c.c_int64, _P, _c.c_int32, _c.c_int32, _c.c_int32,
                                _P, _P, _c.c_int64, _P, _P, _c.c_size_t, _P]),
    "fp8q_set_wait_budget_ns": (_c.c_int, [_c.c_uint64]),
    "fp8q_amax": (_c.c_int, [_P, _c.c_int32, _c.c_int64, _c.c_int64, _P, _c.c_int32, _P, _P]),
    "fp8q_cast_workspace_bytes": (_c.c_size_t, [_c.c_int32]),
    "fp8q_cast_per_tensor": (_c.c_int, [_P, _c.c_int32, _c.c_int64, _c.c_int64, _P, _c.c_int32,
                                        _c.c_int32, _c.c_int32, _P, _P, _P, _P, _P, _P, _P,
                                        _c.c_size_t, _P]),
    "fp8q_cast_per_tensor_static_ws": (_c.c_int, [_P, _c.c_int32, _c.c_int64, _c.c_int64, _P, _c.c_int32,
                                                  _c.c_int32, _c.c_int32, _P, _P, _P, _P, _P, _P, _P]),
    "fp8q_delayed_create": (_c.c_int, [_c.c_int32, _c.c_int32, _c.c_int32, _c.c_int32,
                                       _c.POINTER(_P)]),
    "fp8q_delayed_destroy": (_c.c_int, [_P]),
    "fp8q_delayed_reset": (_c.c_int, [_P, _P]),
    "fp8q_delayed_step": (_c.c_int, [_P, _P, _c.c_int32, _c.c_int64, _P, _P, _P, _P, _P, _P]),
    "fp8q_delayed_get": (_c.c_int, [_P, _P, _P, _P, _P, _P]),
    "fp8q_delayed_set": (_c.c_int, [_P, _P, _c.c_int32, _c.c_int32, _c.c_int64]),
    "mxfp8_col_blocks": (_c.c_int64, [_P, _c.c_int32, _c.c_int64]),
    "mxfp8_quantize": (_c.c_int, [_P, _c.c_int32, _c.c_int64, _c.c_int64, _P, _c.c_int32,
                                  _c.c_int32, _c.c_int32, _P, _P, _P, _P, _c.c_int64, _P]),
}

_lib = None
_lock = threading.Lock()


class Fp8qError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile libfp8q.so for sm_103a (in-tree) and load it."""
    global _lib
    path = _build_lib(force=force)
    with _lock:
        _lib = None
    lib()
    return path


def library_path() -> str:
    return LIB_PATH


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise Fp8qError(f"{LIB_PATH} is missing: run mxfp8_quantization_amax_gb300.build()")
            h = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in _SIGS.items():
                f = getattr(h, name)
                f.restype = res
                f.argtypes = args
            _lib = h
    return _lib


def _check(status: int, what: str):
    if status != 0:
        msg = lib().fp8q_last_error_string().decode(errors="replace")
        raise Fp8qError(f"{what} failed with status {status}: {msg}")


def _ptr(t):
    return None if t is None else _P(t.data_ptr())


def _stream():
    return _P(torch.cuda.current_stream().cuda_stream)


def _dt(x: torch.Tensor) -> int:
    if x.dtype == torch.bfloat16:
        return 0
    if x.dtype == torch.float32:
        return 1
    raise TypeError("x must be bfloat16 or float32")


def _check_input(x: torch.Tensor):
    if not x.is_cuda:
        raise ValueError("x must be a CUDA tensor")
    if not x.is_contiguous():
        raise ValueError("x must be contiguous")


def _as_2d(x: torch.Tensor):
    if x.dim() == 2:
        return x.shape[0], x.shape[1]
    if x.dim() == 1:
        return 1, x.shape[0]
    return x.numel() // x.shape[-1], x.shape[-1]


def _offsets(group_offsets, device):
    if group_offsets is None:
        return None, 1
    o = group_offsets
    if not isinstance(o, torch.Tensor):
        o = torch.tensor(list(o), dtype=torch.int64)
    o = o.to(device=device, dtype=torch.int64).contiguous()
    return o, o.numel() - 1


def check_device():
    """Synchronize the current stream and raise if a device-side wait gave up."""
    _check(lib().fp8q_check_device(_stream()), "fp8q_check_device")


def set_wait_budget_ns(ns: int):
    _check(lib().fp8q_set_wait_budget_ns(int(ns)), "fp8q_set_wait_budget_ns")


def debug_stall_mx_producer(on: bool):
    """Test hook: the BF16 MXFP8 kernel's producer issues no loads while on,
    so its consumers' bounded waits expire (reported by check_device)."""
    _check(lib().fp8q_debug_stall_mx_producer(1 if on else 0), "fp8q_debug_stall_mx_producer")


def debug_stall_scale_publish(on: bool):
    """Test hook: while on, the single-launch current scaling never publishes
    its scale, so the waits for it expire (reported by check_device)."""
    _check(lib().fp8q_debug_stall_scale_publish(1 if on else 0), "fp8q_debug_stall_scale_publish")


# ---------------------------------------------------------------------------
# amax
# ---------------------------------------------------------------------------
def fp8q_amax(x: torch.Tensor, group_offsets=None, out: torch.Tensor | None = None) -> torch.Tensor:
    """Per-tensor (or per-group) max |x|, bit-exact, as float32 [G]."""
    _check_input(x)
    rows, cols = _as_2d(x)
    off, G = _offsets(group_offsets, x.device)
    if out is None:
        out = torch.empty(G, dtype=torch.float32, device=x.device)
    _check(lib().fp8q_amax(_ptr(x), _dt(x), rows, cols, _ptr(off), G, _ptr(out), _stream()), "fp8q_amax")
    return out


def fp8q_scale_from_amax(amax: torch.Tensor, fmt: int = E4M3, margin: int = 0, out: dict | None = None) -> dict:
    """Per-group scale and its reciprocal from given amaxes (device float32 [G])."""
    if not amax.is_cuda or amax.dtype != torch.float32 or not amax.is_contiguous():
        raise ValueError("amax must be a contiguous float32 CUDA tensor")
    G = amax.numel()
    o = out or {}
    scale = o.get("scale")
    scale = torch.empty(G, dtype=torch.float32, device=amax.device) if scale is None else scale
    scale_inv = o.get("scale_inv")
    scale_inv = torch.empty(G, dtype=torch.float32, device=amax.device) if scale_inv is None else scale_inv
    _check(lib().fp8q_scale_from_amax(_ptr(amax), G, fmt, margin, _ptr(scale), _ptr(scale_inv), _stream()),
           "fp8q_scale_from_amax")
    return {"scale": scale, "scale_inv": scale_inv}


# ---------------------------------------------------------------------------
# per-tensor cast
# ---------------------------------------------------------------------------
def fp8q_cast_workspace_bytes(num_groups: int = 1) -> int:
    return int(lib().fp8q_cast_workspace_bytes(num_groups))


_ws_cache: dict = {}


def _workspace(device, G: int, stream_id: int) -> torch.Tensor:
    """Zero-filled workspace per (device, stream), grown as needed."""
    need = fp8q_cast_workspace_bytes(G)
    key = (device.index, stream_id)
    ws = _ws_cache.get(key)
    if ws is None or ws.numel() < need:
        ws = torch.zeros(max(need, 4096), dtype=torch.uint8, device=device)
        _ws_cache[key] = ws
    return ws


def fp8q_cast_per_tensor(x: torch.Tensor, fmt: int = E4M3, margin: int = 0, scale_in=None,
                         group_offsets=None, want_amax: bool = True, want_sat: bool = False,
                         q: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                         out: dict | None = None) -> dict:
    """q = RNE_sat(fl32(x * scale)).  scale_in None: current scaling.

    Returns dict(q uint8 like x, amax, scale, scale_inv float32 [G], sat uint64 [G] or None).
    `out` may hold preallocated "amax", "scale", "scale_inv", "sat" tensors.
    """
    _check_input(x)
    rows, cols = _as_2d(x)
    off, G = _offsets(group_offsets, x.device)
    dev = x.device
    o = out or {}

    def buf(name, dtype, wanted=True):
        if not wanted:
            return None
        t = o.get(name)
        return t if t is not None else torch.empty(G, dtype=dtype, device=dev)

    q = torch.empty(x.shape, dtype=torch.uint8, device=dev) if q is None else q
    amax = buf("amax", torch.float32, want_amax)
    scale = buf("scale", torch.float32)
    scale_inv = buf("scale_inv", torch.float32)
    sat = buf("sat", torch.int64, want_sat)
    if scale_in is not None:
        if not isinstance(scale_in, torch.Tensor):
            scale_in = torch.tensor(scale_in, dtype=torch.float32)
        scale_in = scale_in.to(device=dev, dtype=torch.float32).reshape(-1).contiguous()
        if scale_in.numel() != G:
            raise ValueError("scale_in must hold one scale per group")
    stream = torch.cuda.current_stream()
    ws = workspace if workspace is not None else _workspace(dev, G, stream.cuda_stream)
    _check(lib().fp8q_cast_per_tensor(
        _ptr(x), _dt(x), rows, cols, _ptr(off), G, fmt, margin, _ptr(scale_in), _ptr(q), _ptr(amax),
        _ptr(scale), _ptr(scale_inv), _ptr(sat), _ptr(ws), ws.numel(), _P(stream.cuda_stream)),
        "fp8q_cast_per_tensor")
    return {"q": q, "amax": amax, "scale": scale, "scale_inv": scale_inv, "sat": sat}


# ---------------------------------------------------------------------------
# delayed scaling
# ---------------------------------------------------------------------------
class DelayedScaling:
    """Library-owned delayed-scaling state (history ring on the device)."""

    def __init__(self, history_len: int = 16, interval: int = 1, margin: int = 0, fmt: int = E4M3):
        self.history_len, self.interval, self.margin, self.fmt = history_len, interval, margin, fmt
        h = _P()
        _check(lib().fp8q_delayed_create(history_len, interval, margin, fmt, ctypes.byref(h)),
               "fp8q_delayed_create")
        self._h = h

    def close(self):
        if getattr(self, "_h", None):
            lib().fp8q_delayed_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def reset(self):
        _check(lib().fp8q_delayed_reset(self._h, _stream()), "fp8q_delayed_reset")

    def step(self, x: torch.Tensor, q: torch.Tensor | None = None, want_sat: bool = False,
             outs: dict | None = None) -> dict:
        """Cast x with the predicted scale; records amax on recording steps.

        Returns dict(q, scale [1], scale_inv [1], amax [1] (valid only on
        recording steps), sat [1] or None).
        """
        _check_input(x)
        dev = x.device
        o = outs or {}

        def buf(name, dtype):
            t = o.get(name)
            return t if t is not None else torch.empty(1, dtype=dtype, device=dev)

        q = q if q is not None else torch.empty(x.shape, dtype=torch.uint8, device=dev)
        scale = buf("scale", torch.float32)
        scale_inv = buf("scale_inv", torch.float32)
        amax = buf("amax", torch.float32)
        sat = buf("sat", torch.int64) if want_sat else None
        _check(lib().fp8q_delayed_step(self._h, _ptr(x), _dt(x), x.numel(), _ptr(q), _ptr(scale),
                                       _ptr(scale_inv), _ptr(amax), _ptr(sat), _stream()),
               "fp8q_delayed_step")
        return {"q": q, "scale": scale, "scale_inv": scale_inv, "amax": amax, "sat": sat}

    def get(self) -> dict:
        hist = (ctypes.c_float * self.history_len)()
        head, count, nonfinite = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
        step = ctypes.c_int64()
        _check(lib().fp8q_delayed_get(self._h, ctypes.cast(hist, _P), ctypes.byref(head),
                                      ctypes.byref(count), ctypes.byref(step), ctypes.byref(nonfinite)),
               "fp8q_delayed_get")
        return {"history": list(hist), "head": head.value, "count": count.value, "step": step.value,
                "nonfinite": bool(nonfinite.value)}

    def set(self, history, head: int, count: int, step: int):
        arr = (ctypes.c_float * self.history_len)(*[float(v) for v in history])
        _check(lib().fp8q_delayed_set(self._h, ctypes.cast(arr, _P), head, count, step), "fp8q_delayed_set")


# ---------------------------------------------------------------------------
# MXFP8
# ---------------------------------------------------------------------------
def mxfp8_col_blocks(rows: int, group_offsets=None) -> int:
    """sum_g ceil(n_g / 32) from host offsets (None: ceil(rows / 32))."""
    if group_offsets is None:
        return int(lib().mxfp8_col_blocks(None, 1, rows))
    o = torch.as_tensor(list(group_offsets) if not isinstance(group_offsets, torch.Tensor) else group_offsets,
                        dtype=torch.int64).cpu().contiguous()
    n = int(lib().mxfp8_col_blocks(_P(o.data_ptr()), o.numel() - 1, rows))
    if n < 0:
        raise ValueError("invalid group offsets")
    return n


def mxfp8_mma_scale_bytes(rows: int, scale_cols: int) -> int:
    """Bytes of a rows x scale_cols scale matrix in the 128 x 4 block layout."""
    return int(lib().mxfp8_mma_scale_bytes(rows, scale_cols))


def mxfp8_quantize(x: torch.Tensor, fmt: int = E4M3, direction: int = BOTH, group_offsets=None,
                   s_col_ld: int | None = None, out: dict | None = None, rule: int = RULE_UP,
                   count_saturation: bool = False, scale_layout: int = SCALES_ROW_MAJOR) -> dict:
    """MXFP8 rowwise and/or columnwise quantization of a 2-D tensor.

    Returns dict(q_row [rows, cols], s_row [rows, cols/32], q_col [cols, rows],
    s_col [cols, s_col_ld]) (uint8; unused direction -> None).  The default
    s_col_ld is ceil(rows / 32) without groups, and the column-block count
    rounded up to a multiple of 16 with groups (the padding is not written).
    scale_layout SCALES_MMA writes both scale arrays in the 128 x 4 block
    layout of block-scaled MMA instead (flat uint8 tensors of
    mxfp8_mma_scale_bytes bytes; s_col_ld is then the column-block count).
    """
    _check_input(x)
    rows, cols = _as_2d(x)
    off, G = _offsets(group_offsets, x.device)
    dev = x.device
    mma = scale_layout == SCALES_MMA
    if s_col_ld is None:
        if group_offsets is None:
            s_col_ld = (rows + 31) // 32
        else:
            host = group_offsets.cpu() if isinstance(group_offsets, torch.Tensor) else group_offsets
            s_col_ld = mxfp8_col_blocks(rows, host)
            if not mma:
                # padded to 16 bytes: scale rows then start aligned, which
                # lets the kernel store a column's scales in whole 8-byte words
                s_col_ld = (s_col_ld + 15) // 16 * 16
    o = out or {}

    def buf(name, shape):
        t = o.get(name)
        return t if t is not None else torch.empty(shape, dtype=torch.uint8, device=dev)

    q_row = s_row = q_col = s_col = None
    if direction & ROW:
        q_row = buf("q_row", (rows, cols))
        nsc = cols // 32 if cols % 32 == 0 else 0
        s_row = buf("s_row", (mxfp8_mma_scale_bytes(rows, nsc),) if mma else (rows, nsc))
    if direction & COL:
        q_col = buf("q_col", (cols, rows))
        s_col = buf("s_col", (mxfp8_mma_scale_bytes(cols, s_col_ld),) if mma else (cols, max(s_col_ld, 1)))
    sat = o.get("sat")
    if count_saturation and sat is None:
        sat = torch.empty(2, dtype=torch.int64, device=dev)
    if rule == RULE_UP and not count_saturation and not mma:
        _check(lib().mxfp8_quantize(_ptr(x), _dt(x), rows, cols, _ptr(off), G, fmt, direction,
                                    _ptr(q_row), _ptr(s_row), _ptr(q_col), _ptr(s_col), s_col_ld, _stream()),
               "mxfp8_quantize")
    else:
        _check(lib().mxfp8_quantize_ex(_ptr(x), _dt(x), rows, cols, _ptr(off), G, fmt, direction, rule, scale_layout,
                                       _ptr(q_row), _ptr(s_row), _ptr(q_col), _ptr(s_col), s_col_ld,
                                       _ptr(sat) if count_saturation else None, _stream()),
               "mxfp8_quantize_ex")
    return {"q_row": q_row, "s_row": s_row, "q_col": q_col, "s_col": s_col, "s_col_ld": s_col_ld,
            "sat": sat if count_saturation else None}


def _out_dtype(out_dtype) -> int:
    if out_dtype == torch.bfloat16:
        return 0
    if out_dtype == torch.float32:
        return 1
    raise TypeError("out_dtype must be torch.bfloat16 or torch.float32")


def fp8q_dequantize_per_tensor(q: torch.Tensor, scale_inv: torch.Tensor, fmt: int = E4M3, group_offsets=None,
                               out_dtype=torch.bfloat16, out: torch.Tensor | None = None) -> torch.Tensor:
    """y = round_out(fl32(value(q) * scale_inv[g])), shaped like q (uint8 codes)."""
    if not q.is_cuda or q.dtype != torch.uint8 or not q.is_contiguous():
        raise ValueError("q must be a contiguous uint8 CUDA tensor")
    rows, cols = _as_2d(q)
    off, G = _offsets(group_offsets, q.device)
    si = scale_inv.to(device=q.device, dtype=torch.float32).reshape(-1).contiguous()
    if si.numel() != G:
        raise ValueError("scale_inv must hold one value per group")
    y = torch.empty(q.shape, dtype=out_dtype, device=q.device) if out is None else out
    _check(lib().fp8q_dequantize_per_tensor(_ptr(q), rows, cols, _ptr(off), G, fmt, _ptr(si),
                                            _out_dtype(out_dtype), _ptr(y), _stream()),
           "fp8q_dequantize_per_tensor")
    return y


def mxfp8_dequantize(q: torch.Tensor, s: torch.Tensor, rows: int, cols: int, fmt: int = E4M3,
                     direction: int = ROW, group_offsets=None, out_dtype=torch.bfloat16,
                     out: torch.Tensor | None = None) -> torch.Tensor:
    """One MX copy back to high precision, in the copy's own layout.

    direction ROW: q [rows, cols], s [rows, cols/32] -> y [rows, cols].
    direction COL: q [cols, rows], s [cols, s_ld] -> y [cols, rows].
    """
    if not q.is_cuda or q.dtype != torch.uint8 or not q.is_contiguous() or not s.is_contiguous():
        raise ValueError("q and s must be contiguous uint8 CUDA tensors")
    off, G = _offsets(group_offsets, q.device)
    s_ld = s.shape[-1] if s.dim() == 2 else 0
    y = torch.empty(q.shape, dtype=out_dtype, device=q.device) if out is None else out
    _check(lib().mxfp8_dequantize(_ptr(q), _ptr(s), rows, cols, _ptr(off), G, fmt, direction, s_ld,
                                  _out_dtype(out_dtype), _ptr(y), _stream()), "mxfp8_dequantize")
    return y


# ---------------------------------------------------------------------------
# MXFP4 / MXFP6
# ---------------------------------------------------------------------------
def mx_quantize_fp4_fp6(x: torch.Tensor, elem: int = E2M1, direction: int = BOTH, rule: int = RULE_UP,
                        count_saturation: bool = False, out: dict | None = None) -> dict:
    """MXFP4 (elem E2M1: two codes per byte, even element low) or MXFP6
    (E2M3 / E3M2: one code per byte) with E8M0 scales per 32 elements.

    Returns q_row [rows, cols/2 or cols], s_row [rows, cols/32], q_col
    [cols, rows/2 or rows], s_col [cols, ceil(rows/32)] for the requested
    directions, and sat (uint64[2] saturated counts) when counted."""
    _check_input(x)
    rows, cols = _as_2d(x)
    out = {} if out is None else out
    fp4 = elem == E2M1
    shapes = {"q_row": (rows, cols // 2 if fp4 else cols), "s_row": (rows, cols // 32),
              "q_col": (cols, rows // 2 if fp4 else rows), "s_col": (cols, (rows + 31) // 32)}

    def buf(name, wanted):
        if not wanted:
            return None
        if name not in out:
            out[name] = torch.empty(shapes[name], dtype=torch.uint8, device=x.device)
        return out[name]

    q_row, s_row = buf("q_row", direction & ROW), buf("s_row", direction & ROW)
    q_col, s_col = buf("q_col", direction & COL), buf("s_col", direction & COL)
    sat = None
    if count_saturation:
        sat = out.setdefault("sat", torch.zeros(2, dtype=torch.int64, device=x.device))
    _check(lib().mx_quantize_fp4_fp6(_ptr(x), _dt(x), rows, cols, elem, direction, rule, _ptr(q_row), _ptr(s_row),
                                     _ptr(q_col), _ptr(s_col), _ptr(sat), _stream()), "mx_quantize_fp4_fp6")
    return out


# ---------------------------------------------------------------------------
# block scales for tensor-core MMA
# ---------------------------------------------------------------------------
def mx_scales_to_mma_layout(s: torch.Tensor, scale_cols: int | None = None,
                            out: torch.Tensor | None = None) -> torch.Tensor:
    """A [rows, s_ld] uint8 scale array (first scale_cols columns) in the
    128 x 4 block layout of block-scaled MMA: a flat uint8 tensor of
    ceil(rows/128)*128 * ceil(scale_cols/4)*4 bytes, padding 0."""
    if not s.is_cuda or s.dtype != torch.uint8 or s.dim() != 2 or not s.is_contiguous():
        raise ValueError("s must be a contiguous 2-D uint8 CUDA tensor")
    rows, s_ld = s.shape
    sc = s_ld if scale_cols is None else scale_cols
    n = ((rows + 127) // 128 * 128) * ((sc + 3) // 4 * 4)
    y = torch.empty(n, dtype=torch.uint8, device=s.device) if out is None else out
    _check(lib().mx_scales_to_mma_layout(_ptr(s), rows, sc, s_ld, _ptr(y), _stream()), "mx_scales_to_mma_layout")
    return y


# ---------------------------------------------------------------------------
# quantization-error statistics (SQNR, zero-rate)
# ---------------------------------------------------------------------------
QSTATS_BYTES = 64  # fp8q_qstats: 2 doubles, 4 uint64, 2 doubles


def fp8q_qstats_workspace_bytes() -> int:
    return int(lib().fp8q_qstats_workspace_bytes())


_qs_ws_cache: dict = {}


def _qstats_workspace(device, stream_id: int) -> torch.Tensor:
    key = (device.index, stream_id)
    ws = _qs_ws_cache.get(key)
    if ws is None:
        ws = torch.zeros(fp8q_qstats_workspace_bytes(), dtype=torch.uint8, device=device)
        _qs_ws_cache[key] = ws
    return ws


def _qstats_out(x: torch.Tensor, out):
    if out is None:
        return torch.empty(QSTATS_BYTES // 8, dtype=torch.float64, device=x.device)
    if not out.is_cuda or out.numel() * out.element_size() < QSTATS_BYTES or out.data_ptr() % 8:
        raise ValueError(f"out must be an 8-byte aligned CUDA tensor of at least {QSTATS_BYTES} bytes")
    return out


def fp8q_qstats_per_tensor(x: torch.Tensor, q: torch.Tensor, scale_inv: torch.Tensor, fmt: int = E4M3,
                           group_offsets=None, out: torch.Tensor | None = None) -> torch.Tensor:
    """Statistics of a per-tensor (per-group) copy q of x, as a device
    tensor holding an fp8q_qstats (read it with qstats_dict)."""
    _check_input(x)
    rows, cols = _as_2d(x)
    if not q.is_cuda or q.dtype != torch.uint8 or not q.is_contiguous() or q.numel() != x.numel():
        raise ValueError("q must be a contiguous uint8 CUDA tensor with x's element count")
    off, G = _offsets(group_offsets, x.device)
    si = scale_inv.to(device=x.device, dtype=torch.float32).reshape(-1).contiguous()
    if si.numel() != G:
        raise ValueError("scale_inv must hold one value per group")
    o = _qstats_out(x, out)
    stream = torch.cuda.current_stream(x.device)
    ws = _qstats_workspace(x.device, stream.cuda_stream)
    _check(lib().fp8q_qstats_per_tensor(_ptr(x), _dt(x), rows, cols, _ptr(off), G, fmt, _ptr(q), _ptr(si), _ptr(o),
                                        _ptr(ws), ws.numel(), _stream()), "fp8q_qstats_per_tensor")
    return o


def mxfp8_qstats(x: torch.Tensor, q: torch.Tensor, s: torch.Tensor, fmt: int = E4M3, direction: int = ROW,
                 group_offsets=None, out: torch.Tensor | None = None) -> torch.Tensor:
    """Statistics of one MX copy of x (direction ROW: q_row/s_row; COL:
    q_col/s_col), as a device tensor holding an fp8q_qstats."""
    _check_input(x)
    rows, cols = _as_2d(x)
    if not q.is_cuda or q.dtype != torch.uint8 or not q.is_contiguous() or not s.is_contiguous():
        raise ValueError("q and s must be contiguous uint8 CUDA tensors")
    off, G = _offsets(group_offsets, x.device)
    s_ld = s.shape[-1] if s.dim() == 2 else 0
    o = _qstats_out(x, out)
    stream = torch.cuda.current_stream(x.device)
    ws = _qstats_workspace(x.device, stream.cuda_stream)
    _check(lib().mxfp8_qstats(_ptr(x), _dt(x), rows, cols, _ptr(off), G, fmt, direction, _ptr(q), _ptr(s), s_ld,
                              _ptr(o), _ptr(ws), ws.numel(), _stream()), "mxfp8_qstats")
    return o


def qstats_dict(t: torch.Tensor) -> dict:
    """The fp8q_qstats in a device tensor as a dict (the library computes
    the SQNR in dB and the zero-rate on the device)."""
    raw = t.reshape(-1).view(torch.uint8)[:QSTATS_BYTES].cpu()
    f = raw[:16].view(torch.float64).tolist()
    c = raw[16:48].view(torch.int64).tolist()
    g = raw[48:64].view(torch.float64).tolist()
    return {"signal": f[0], "noise": f[1], "n": c[0], "n_zero": c[1], "n_flushed": c[2], "n_nonfinite": c[3],
            "sqnr_db": g[0], "zero_rate": g[1]}


# ---------------------------------------------------------------------------
# blockwise FP8
# ---------------------------------------------------------------------------
def fp8q_quantize_blockwise(x: torch.Tensor, fmt: int = E4M3, block: int = BLOCK_1X128, pow2_scales: bool = False,
                            direction: int = ROW, out: dict | None = None) -> dict:
    """Blockwise FP8 of a 2-D BF16 tensor with FP32 scales (see the C header).

    Returns dict(q [rows, cols], scale_inv, q_t [cols, rows], scale_inv_t);
    the unused copy is None.
    """
    _check_input(x)
    rows, cols = _as_2d(x)
    tr, tc = (rows + 127) // 128, (cols + 127) // 128
    o = out or {}

    def buf(name, shape, dtype):
        t = o.get(name)
        return t if t is not None else torch.empty(shape, dtype=dtype, device=x.device)

    q = si = q_t = si_t = None
    if direction & ROW:
        q = buf("q", (rows, cols), torch.uint8)
        si = buf("scale_inv", (rows, tc) if block == BLOCK_1X128 else (tr, tc), torch.float32)
    if direction & COL:
        q_t = buf("q_t", (cols, rows), torch.uint8)
        si_t = buf("scale_inv_t", (cols, tr) if block == BLOCK_1X128 else (tc, tr), torch.float32)
    _check(lib().fp8q_quantize_blockwise(_ptr(x), _dt(x), rows, cols, fmt, block, 1 if pow2_scales else 0,
                                         direction, _ptr(q), _ptr(si), _ptr(q_t), _ptr(si_t), _stream()),
           "fp8q_quantize_blockwise")
    return {"q": q, "scale_inv": si, "q_t": q_t, "scale_inv_t": si_t}


# ---------------------------------------------------------------------------
# NVFP4
# ---------------------------------------------------------------------------
def fp8q_quantize_nvfp4(x: torch.Tensor, out: dict | None = None) -> dict:
    """NVFP4 of a 2-D tensor: dict(q [rows, cols/2] packed E2M1, s [rows, cols/16]
    E4M3 codes, amax [1], scale [1] = the tensor scale S)."""
    _check_input(x)
    rows, cols = _as_2d(x)
    o = out or {}

    def buf(name, shape, dtype):
        t = o.get(name)
        return t if t is not None else torch.empty(shape, dtype=dtype, device=x.device)

    q = buf("q", (rows, cols // 2), torch.uint8)
    s = buf("s", (rows, cols // 16), torch.uint8)
    amax = buf("amax", (1,), torch.float32)
    scale = buf("scale", (1,), torch.float32)
    _check(lib().fp8q_quantize_nvfp4(_ptr(x), _dt(x), rows, cols, _ptr(q), _ptr(s), _ptr(amax), _ptr(scale),
                                     _stream()), "fp8q_quantize_nvfp4")
    return {"q": q, "s": s, "amax": amax, "scale": scale}
