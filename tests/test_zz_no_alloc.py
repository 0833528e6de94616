"""The allocation-free per-tensor cast (fp8q_cast_per_tensor_static_ws).

Callers that cannot allocate device memory where they quantize use this
entry point; its workspace is a fixed array inside the library.  Its
results must equal those of fp8q_cast_per_tensor with a caller workspace,
bit for bit, call after call (the shared array keeps the previous call's
contents, so the second call checks that nothing leaks between calls).
This file is collected last so that a failure here stops a run only after
every other test has run.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
from gpu_util import Guarded, dev, host, require_cuda

pytestmark = pytest.mark.gpu


def _call(fq, fn_name, x_np, fmt, margin, offsets, scale_in=None):
    rows, cols = x_np.shape
    G = 1 if offsets is None else len(offsets) - 1
    x = dev(x_np)
    off = None if offsets is None else torch.tensor(offsets, dtype=torch.int64, device="cuda")
    q = Guarded((rows, cols))
    outs = [Guarded((G,), torch.float32) for _ in range(3)]
    sat = Guarded((G,), torch.int64)
    sc = None if scale_in is None else torch.tensor(scale_in, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    args = [x.data_ptr(), 0 if x_np.dtype == np.uint16 else 1, rows, cols,
            None if off is None else off.data_ptr(), G, fmt, margin,
            None if sc is None else sc.data_ptr(), q.t.data_ptr(), outs[0].t.data_ptr(),
            outs[1].t.data_ptr(), outs[2].t.data_ptr(), sat.t.data_ptr()]
    lib = fq.lib()
    if fn_name == "workspace":
        ws = torch.zeros(fq.fp8q_cast_workspace_bytes(G), dtype=torch.uint8, device="cuda")
        st = lib.fp8q_cast_per_tensor(*args, ws.data_ptr(), ws.numel(), stream)
    else:
        st = lib.fp8q_cast_per_tensor_static_ws(*args, stream)
    assert st == 0, lib.fp8q_last_error_string()
    torch.cuda.synchronize()
    for g in [q, sat] + outs:
        g.check()
    return [host(q.t), host(outs[0].t).view(np.uint32), host(outs[1].t).view(np.uint32),
            host(outs[2].t).view(np.uint32), host(sat.t)]


def _offsets_256():
    """256 groups over 4096 rows: multinomial counts with every eighth group
    emptied into its neighbour, so empty, tiny and large groups all occur."""
    counts = np.random.default_rng(79).multinomial(4096, [1.0 / 256] * 256)
    for g in range(0, 256, 8):
        counts[g + 1] += counts[g]
        counts[g] = 0
    assert (counts == 0).sum() >= 32 and counts.sum() == 4096
    return [0] + [int(v) for v in np.cumsum(counts)]


CASES = [
    ("1024x1024 current scaling", lambda: synth.config1(), 0, 0, None, None),
    ("MoE groups, E5M2, margin 2", lambda: synth.student_t(1000, 96, 4.0, seed=77), 1, 2,
     [0, 13, 13, 500, 640, 1000], None),
    ("given scales, fused amax", lambda: synth.normal_outliers(300, 64, seed=78), 0, 0, [0, 100, 300],
     [2.5, 0.125]),
    # the documented maximum: 256 groups (4160 of the array's 8192 bytes)
    ("256 ragged groups with empty ones", lambda: synth.student_t(4096, 64, 4.0, seed=80), 0, 0,
     _offsets_256(), None),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_static_workspace_matches_caller_workspace_twice(case):
    fq = require_cuda()
    _, make, fmt, margin, offsets, scale_in = case
    x = make()
    want = _call(fq, "workspace", x, fmt, margin, offsets, scale_in)
    for _ in range(2):  # the second call sees whatever the first left in the shared array
        got = _call(fq, "static", x, fmt, margin, offsets, scale_in)
        for a, b in zip(got, want):
            np.testing.assert_array_equal(a, b)


def test_static_workspace_rejects_too_many_groups():
    """257 groups, one past the limit, is refused before anything runs."""
    fq = require_cuda()
    x = torch.zeros((257, 32), dtype=torch.bfloat16, device="cuda")
    off = torch.arange(0, 258, dtype=torch.int64, device="cuda")
    q = torch.full((257, 32), 0xA5, dtype=torch.uint8, device="cuda")
    st = fq.lib().fp8q_cast_per_tensor_static_ws(x.data_ptr(), 0, 257, 32, off.data_ptr(), 257, 0, 0, None,
                                                 q.data_ptr(), None, None, None, None,
                                                 torch.cuda.current_stream().cuda_stream)
    assert st == 1
    assert b"at most 256 groups" in fq.lib().fp8q_last_error_string()
    torch.cuda.synchronize()
    assert bool((q == 0xA5).all())


def test_static_workspace_rejected_call_then_valid_call():
    """A call refused for its arguments (a bad format) returns
    FP8Q_ERR_INVALID_ARG; the next valid call still matches the caller
    workspace path."""
    fq = require_cuda()
    x_np = synth.student_t(256, 64, 4.0, seed=81)
    x = dev(x_np)
    q = torch.empty((256, 64), dtype=torch.uint8, device="cuda")
    st = fq.lib().fp8q_cast_per_tensor_static_ws(x.data_ptr(), 0, 256, 64, None, 1, 7, 0, None, q.data_ptr(),
                                                 None, None, None, None, torch.cuda.current_stream().cuda_stream)
    assert st == 1 and b"fmt" in fq.lib().fp8q_last_error_string()
    want = _call(fq, "workspace", x_np, 0, 0, [0, 100, 256])
    got = _call(fq, "static", x_np, 0, 0, [0, 100, 256])
    for a, b in zip(got, want):
        np.testing.assert_array_equal(a, b)
