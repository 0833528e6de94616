"""The C ABI without a GPU: the library builds for sm_103a, loads, exports
every entry point include/fp8q.h declares, and rejects bad arguments on the
host before any CUDA call."""
import ctypes
import os
import re

import pytest

import mxfp8_quantization_amax_gb300 as fq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8q.h")


@pytest.fixture(scope="module")
def lib():
    fq.build()
    return fq.lib()


def declared_symbols():
    text = open(HEADER).read()
    return re.findall(r"FP8Q_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)


def test_header_declares_the_entry_points():
    names = set(declared_symbols())
    for n in ("fp8q_amax", "fp8q_cast_per_tensor", "fp8q_delayed_step", "mxfp8_quantize",
              "fp8q_delayed_create", "fp8q_delayed_get", "fp8q_delayed_set", "fp8q_delayed_reset",
              "fp8q_delayed_destroy", "mxfp8_col_blocks", "fp8q_last_error_string",
              "fp8q_cast_workspace_bytes", "fp8q_version"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_only_declared_symbols_are_exported(lib):
    """Internal helpers stay hidden (the build uses -fvisibility=hidden)."""
    out = os.popen(f"nm -D --defined-only {fq.library_path()}").read()
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    ours = {s for s in exported if s.startswith(("fp8q", "mxfp8", "mx_"))}
    assert ours == set(declared_symbols())


def test_binding_exposes_the_same_names():
    for n in ("fp8q_amax", "fp8q_cast_per_tensor", "mxfp8_quantize", "mxfp8_col_blocks",
              "fp8q_cast_workspace_bytes", "DelayedScaling"):
        assert hasattr(fq, n)


def test_version_and_workspace_size(lib):
    assert lib.fp8q_version() == 10000
    assert lib.fp8q_cast_workspace_bytes(1) >= 64 + 16
    assert lib.fp8q_cast_workspace_bytes(64) >= 64 + 16 * 64


def test_col_blocks_host(lib):
    assert fq.mxfp8_col_blocks(100) == 4
    assert fq.mxfp8_col_blocks(150, [0, 0, 33, 34, 100, 150]) == 8
    with pytest.raises(ValueError):
        fq.mxfp8_col_blocks(150, [0, 40, 30, 150])
    with pytest.raises(ValueError):
        fq.mxfp8_col_blocks(150, [0, 40, 149])


def _status(fn, *args):
    return fn(*args)


def test_invalid_arguments_rejected_on_host(lib):
    P = ctypes.c_void_p
    buf = ctypes.create_string_buffer(256)
    aligned = P((ctypes.addressof(buf) + 15) & ~15)
    mis = P(aligned.value + 2)
    # bad dtype
    assert lib.fp8q_amax(aligned, 7, 4, 4, None, 1, aligned, None) == 1
    # misaligned x
    assert lib.fp8q_amax(mis, 0, 4, 4, None, 1, aligned, None) == 1
    assert b"aligned" in lib.fp8q_last_error_string()
    # groups without offsets
    assert lib.fp8q_amax(aligned, 0, 4, 4, None, 3, aligned, None) == 1
    # too many groups
    assert lib.fp8q_amax(aligned, 0, 4, 4, aligned, 5000, aligned, None) == 1
    # MX: cols % 32 != 0 is unsupported
    assert lib.mxfp8_quantize(aligned, 0, 4, 48, None, 1, 0, 3, aligned, aligned, aligned, aligned, 1,
                              None) == 2
    # MX: bad dir / fmt
    assert lib.mxfp8_quantize(aligned, 0, 4, 64, None, 1, 0, 0, aligned, aligned, aligned, aligned, 1,
                              None) == 1
    assert lib.mxfp8_quantize(aligned, 0, 4, 64, None, 1, 2, 3, aligned, aligned, aligned, aligned, 1,
                              None) == 1
    # MX: s_col_ld too small for the rows
    assert lib.mxfp8_quantize(aligned, 0, 100, 64, None, 1, 0, 2, None, None, aligned, aligned, 3,
                              None) == 1
    # cast: margin out of range, missing workspace, small workspace
    assert lib.fp8q_cast_per_tensor(aligned, 0, 4, 4, None, 1, 0, 99, None, aligned, None, None, None,
                                    None, aligned, 4096, None) == 1
    assert lib.fp8q_cast_per_tensor(aligned, 0, 4, 4, None, 1, 0, 0, None, aligned, None, None, None,
                                    None, None, 0, None) == 1
    assert lib.fp8q_cast_per_tensor(aligned, 0, 4, 4, None, 1, 0, 0, None, aligned, None, None, None,
                                    None, aligned, 8, None) == 1
    # delayed: bad history length / interval
    h = P()
    assert lib.fp8q_delayed_create(0, 1, 0, 0, ctypes.byref(h)) == 1
    assert lib.fp8q_delayed_create(16, 0, 0, 0, ctypes.byref(h)) == 1
    assert lib.fp8q_delayed_create(16, 1, 0, 5, ctypes.byref(h)) == 1
    assert lib.fp8q_delayed_step(None, aligned, 0, 4, aligned, None, None, None, None, None) == 1


def test_dequantize_arguments_rejected_on_host(lib):
    buf = ctypes.create_string_buffer(256)
    aligned = (ctypes.addressof(buf) + 15) // 16 * 16
    mis = aligned + 1
    # per-tensor: bad out_dt, bad fmt, missing scale_inv, misaligned y
    assert lib.fp8q_dequantize_per_tensor(aligned, 4, 4, None, 1, 0, aligned, 2, aligned, None) == 1
    assert lib.fp8q_dequantize_per_tensor(aligned, 4, 4, None, 1, 7, aligned, 0, aligned, None) == 1
    assert lib.fp8q_dequantize_per_tensor(aligned, 4, 4, None, 1, 0, None, 0, aligned, None) == 1
    assert lib.fp8q_dequantize_per_tensor(aligned, 4, 4, None, 1, 0, aligned, 0, mis, None) == 1
    # MX: both directions at once, cols % 32, s_ld too small, missing scales
    assert lib.mxfp8_dequantize(aligned, aligned, 4, 64, None, 1, 0, 3, 1, 0, aligned, None) == 1
    assert lib.mxfp8_dequantize(aligned, aligned, 4, 48, None, 1, 0, 1, 0, 0, aligned, None) == 2
    assert lib.mxfp8_dequantize(aligned, aligned, 100, 64, None, 1, 0, 2, 3, 0, aligned, None) == 1
    assert lib.mxfp8_dequantize(aligned, None, 4, 64, None, 1, 0, 1, 0, 0, aligned, None) == 1
    # empty tensors return before any launch
    assert lib.mxfp8_dequantize(None, None, 0, 64, None, 1, 0, 1, 0, 0, None, None) == 0
    assert lib.fp8q_dequantize_per_tensor(None, 0, 4, None, 1, 0, aligned, 0, None, None) == 0


def test_mx_rule_arguments_rejected_on_host(lib):
    buf = ctypes.create_string_buffer(256)
    aligned = (ctypes.addressof(buf) + 15) // 16 * 16
    # unknown rule, misaligned saturation counter
    assert lib.mxfp8_quantize_rule(aligned, 0, 4, 64, None, 1, 0, 3, 2, aligned, aligned, aligned, aligned, 1,
                                   None, None) == 1
    assert lib.mxfp8_quantize_rule(aligned, 0, 4, 64, None, 1, 0, 3, 1, aligned, aligned, aligned, aligned, 1,
                                   aligned + 4, None) == 1


def test_blockwise_arguments_rejected_on_host(lib):
    buf = ctypes.create_string_buffer(256)
    a = (ctypes.addressof(buf) + 15) // 16 * 16
    # FP32 input and shapes off the 16 grid are unsupported; bad block / dir
    assert lib.fp8q_quantize_blockwise(a, 1, 128, 128, 0, 1, 0, 3, a, a, a, a, None) == 2
    assert lib.fp8q_quantize_blockwise(a, 0, 130, 128, 0, 1, 0, 3, a, a, a, a, None) == 2
    assert lib.fp8q_quantize_blockwise(a, 0, 128, 128, 0, 64, 0, 3, a, a, a, a, None) == 1
    assert lib.fp8q_quantize_blockwise(a, 0, 128, 128, 0, 1, 0, 0, a, a, a, a, None) == 1
    # missing outputs of a requested copy, misaligned input
    assert lib.fp8q_quantize_blockwise(a, 0, 128, 128, 0, 1, 0, 2, a, a, None, a, None) == 1
    assert lib.fp8q_quantize_blockwise(a + 2, 0, 128, 128, 0, 1, 0, 1, a, a, None, None, None) == 1
    assert lib.fp8q_quantize_blockwise(None, 0, 0, 128, 0, 1, 0, 3, None, None, None, None, None) == 0


def test_nvfp4_arguments_rejected_on_host(lib):
    buf = ctypes.create_string_buffer(256)
    a = (ctypes.addressof(buf) + 15) // 16 * 16
    assert lib.fp8q_quantize_nvfp4(a, 0, 4, 24, a, a, a, None, None) == 2   # cols % 16
    assert lib.fp8q_quantize_nvfp4(a, 0, 4, 32, a, a, None, None, None) == 1  # amax_out required
    assert lib.fp8q_quantize_nvfp4(a, 0, 4, 32, a + 4, a, a, None, None) == 1  # q alignment


def test_mx_q_row_alignment_checked_before_any_write(lib):
    """A q_row that is 16- but not 32-byte aligned is refused (its codes leave
    in 32-byte stores) before any CUDA call: the call needs no GPU."""
    buf = ctypes.create_string_buffer(512)
    a = (ctypes.addressof(buf) + 63) // 64 * 64
    assert lib.mxfp8_quantize(a, 0, 32, 64, None, 1, 0, 1, a + 16, a, None, None, 0, None) == 1
    assert b"32-byte" in lib.fp8q_last_error_string()
    assert lib.mxfp8_quantize_rule(a, 0, 32, 64, None, 1, 0, 3, 0, a + 16, a, a, a, 2, a, None) == 1


def test_empty_mx_is_a_no_op(lib):
    # rows * cols == 0 returns before any launch
    assert lib.mxfp8_quantize(None, 0, 0, 64, None, 1, 0, 3, None, None, None, None, 0, None) == 0


def test_qstats_arguments_rejected_on_host(lib):
    buf = ctypes.create_string_buffer(256)
    a = (ctypes.addressof(buf) + 15) // 16 * 16
    wsb = lib.fp8q_qstats_workspace_bytes()
    assert 16 + 48 <= wsb < 100 * 1024
    # per-tensor: bad fmt, missing scale_inv, misaligned out, small workspace, misaligned q
    assert lib.fp8q_qstats_per_tensor(a, 0, 4, 4, None, 1, 9, a, a, a, a, wsb, None) == 1
    assert lib.fp8q_qstats_per_tensor(a, 0, 4, 4, None, 1, 0, a, None, a, a, wsb, None) == 1
    assert lib.fp8q_qstats_per_tensor(a, 0, 4, 4, None, 1, 0, a, a, a + 4, a, wsb, None) == 1
    assert lib.fp8q_qstats_per_tensor(a, 0, 4, 4, None, 1, 0, a, a, a, a, wsb - 1, None) == 1
    assert lib.fp8q_qstats_per_tensor(a, 0, 4, 4, None, 1, 0, a + 1, a, a, a, wsb, None) == 1
    # MX: both directions at once, cols % 32, s_ld too small, missing scales, no workspace
    assert lib.mxfp8_qstats(a, 0, 4, 64, None, 1, 0, 3, a, a, 1, a, a, wsb, None) == 1
    assert lib.mxfp8_qstats(a, 0, 4, 48, None, 1, 0, 1, a, a, 0, a, a, wsb, None) == 2
    assert lib.mxfp8_qstats(a, 0, 100, 64, None, 1, 0, 2, a, a, 3, a, a, wsb, None) == 1
    assert lib.mxfp8_qstats(a, 0, 4, 64, None, 1, 0, 1, a, None, 0, a, a, wsb, None) == 1
    assert lib.mxfp8_qstats(a, 0, 4, 64, None, 1, 0, 1, a, a, 0, a, None, wsb, None) == 1
    # a grouped call needs num_groups + 1 offsets; NULL offsets mean one group
    assert lib.mxfp8_qstats(a, 0, 4, 64, None, 2, 0, 2, a, a, 1, a, a, wsb, None) == 1


def test_fp4_fp6_arguments_rejected_on_host(lib):
    buf = ctypes.create_string_buffer(256)
    a = (ctypes.addressof(buf) + 15) // 16 * 16
    # an FP8 format, an unknown rule, cols % 32, odd rows for the packed E2M1 columnwise copy
    assert lib.mx_quantize_fp4_fp6(a, 0, 4, 64, 0, 3, 0, a, a, a, a, None, None) == 1
    assert lib.mx_quantize_fp4_fp6(a, 0, 4, 64, 2, 3, 2, a, a, a, a, None, None) == 1
    assert lib.mx_quantize_fp4_fp6(a, 0, 4, 48, 3, 1, 0, a, a, None, None, None, None) == 2
    assert lib.mx_quantize_fp4_fp6(a, 0, 5, 64, 2, 2, 0, None, None, a, a, None, None) == 2
    # missing outputs of a requested copy, misaligned codes or counter
    assert lib.mx_quantize_fp4_fp6(a, 0, 4, 64, 4, 2, 0, a, a, None, a, None, None) == 1
    assert lib.mx_quantize_fp4_fp6(a, 0, 4, 64, 4, 1, 0, a + 2, a, None, None, None, None) == 1
    assert lib.mx_quantize_fp4_fp6(a, 0, 4, 64, 4, 1, 0, a, a, None, None, a + 4, None) == 1


def test_mma_scale_layout_arguments_rejected_on_host(lib):
    buf = ctypes.create_string_buffer(64)
    a = (ctypes.addressof(buf) + 15) // 16 * 16
    assert lib.mx_scales_to_mma_layout(a, 4, 8, 4, a, None) == 1       # s_ld < scale_cols
    assert lib.mx_scales_to_mma_layout(None, 4, 8, 8, a, None) == 1    # no input
    assert lib.mx_scales_to_mma_layout(a, 4, 8, 8, a + 1, None) == 1   # misaligned output
    assert lib.mx_scales_to_mma_layout(None, 0, 8, 8, None, None) == 0  # empty: nothing to do
