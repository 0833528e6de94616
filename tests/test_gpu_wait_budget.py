"""Bounded device-side waits: an expired wait is reported, and the context
stays usable.

The MXFP8 kernel's producer and consumer warps meet on shared-memory
mbarriers.  Every wait on them gives up after a time budget
(fp8q_set_wait_budget_ns), sets the library's device error word and ends the
kernel; fp8q_check_device turns the word into FP8Q_ERR_TIMEOUT.  The test
hook fp8q_debug_stall_mx_producer makes the producer issue no loads, so the
consumers wait for data that never comes: a flag nothing sets.  No copy is
in flight, nothing faults, and the kernel ends once the budget (1 ms here)
runs out.
"""
import numpy as np
import pytest
import torch

from gpu_util import require_cuda

pytestmark = pytest.mark.gpu

FP8Q_ERR_TIMEOUT = 4


def test_expired_wait_is_reported_and_context_survives():
    fq = require_cuda()
    g = torch.Generator().manual_seed(7)
    x = torch.randn(2048, 4096, generator=g).to(torch.bfloat16).cuda()
    ref = fq.mxfp8_quantize(x, fq.E4M3, fq.BOTH)
    fq.check_device()
    ref = {k: v.cpu() for k, v in ref.items() if isinstance(v, torch.Tensor)}

    try:
        fq.set_wait_budget_ns(10 ** 6)
        fq.debug_stall_mx_producer(True)
        fq.mxfp8_quantize(x, fq.E4M3, fq.BOTH)
        status = fq.lib().fp8q_check_device(fq._stream())
        msg = fq.lib().fp8q_last_error_string()
    finally:
        fq.debug_stall_mx_producer(False)
        fq.set_wait_budget_ns(10 ** 9)
    assert status == FP8Q_ERR_TIMEOUT
    assert b"gave up" in msg

    # the error word was cleared by the check, and the next call is whole
    fq.check_device()
    again = fq.mxfp8_quantize(x, fq.E4M3, fq.BOTH)
    fq.check_device()
    for k, v in ref.items():
        assert np.array_equal(again[k].cpu().numpy(), v.numpy()), k


def test_expired_scale_wait_is_reported_and_workspace_cleared():
    """Single-launch current scaling: the CTA that should publish the scale
    holds it back (test hook), so every other CTA's wait for it expires.  No
    code is written, the call is reported, the workspace is zero again, and
    the next call is whole."""
    fq = require_cuda()
    g = torch.Generator().manual_seed(9)
    # 8 MB: above the one-cluster kernel's 2 MB, so the grid-wide ticket runs
    x = (torch.randn(2048, 2048, generator=g) * 3).to(torch.bfloat16).cuda()
    ws = torch.zeros(fq.fp8q_cast_workspace_bytes(1), dtype=torch.uint8, device="cuda")
    ref = fq.fp8q_cast_per_tensor(x, fq.E4M3, want_sat=True, workspace=ws)
    fq.check_device()
    ref = {k: v.cpu() for k, v in ref.items() if isinstance(v, torch.Tensor)}

    q = torch.full((2048, 2048), 0x5A, dtype=torch.uint8, device="cuda")
    try:
        fq.set_wait_budget_ns(10 ** 6)
        fq.debug_stall_scale_publish(True)
        fq.fp8q_cast_per_tensor(x, fq.E4M3, want_sat=True, q=q, workspace=ws)
        status = fq.lib().fp8q_check_device(fq._stream())
        msg = fq.lib().fp8q_last_error_string()
    finally:
        fq.debug_stall_scale_publish(False)
        fq.set_wait_budget_ns(10 ** 9)
    assert status == FP8Q_ERR_TIMEOUT
    assert b"gave up" in msg
    assert bool((q == 0x5A).all()), "codes written without a published scale"
    assert int(ws.count_nonzero()) == 0, "workspace not left zero-filled"

    fq.check_device()
    again = fq.fp8q_cast_per_tensor(x, fq.E4M3, want_sat=True, workspace=ws)
    fq.check_device()
    for k, v in ref.items():
        assert torch.equal(again[k].cpu(), v), k
    assert int(ws.count_nonzero()) == 0
