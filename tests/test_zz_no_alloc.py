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


CASES = [
    ("1024x1024 current scaling", lambda: synth.config1(), 0, 0, None, None),
    ("MoE groups, E5M2, margin 2", lambda: synth.student_t(1000, 96, 4.0, seed=77), 1, 2,
     [0, 13, 13, 500, 640, 1000], None),
    ("given scales, fused amax", lambda: synth.normal_outliers(300, 64, seed=78), 0, 0, [0, 100, 300],
     [2.5, 0.125]),
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
    fq = require_cuda()
    x = torch.zeros((300, 32), dtype=torch.bfloat16, device="cuda")
    off = torch.arange(0, 301, dtype=torch.int64, device="cuda")
    q = torch.empty((300, 32), dtype=torch.uint8, device="cuda")
    st = fq.lib().fp8q_cast_per_tensor_static_ws(x.data_ptr(), 0, 300, 32, off.data_ptr(), 300, 0, 0, None,
                                                 q.data_ptr(), None, None, None, None,
                                                 torch.cuda.current_stream().cuda_stream)
    assert st == 1
    assert b"at most 256 groups" in fq.lib().fp8q_last_error_string()
