"""GPU parity at the workloads' full sizes, element by element against the
oracle: every code byte, every scale byte and every amax / scale bit.

  * delayed scaling: 32 drifting steps of one 8192 x 8192 BF16 tensor
    (sigma_{t+1} = sigma_t * U(0.8, 1.25)), history 16, margin 3, Interval 1
    and 5, E4M3 and E5M2, and current scaling of the same tensors
    ("HiFloat8：高性能训练之路" 1.2 and 3; "混合精度与 FP8 训练" 8.2);
  * one 8B-class linear layer's A 16384x4096, W 14336x4096 (E4M3) and
    E 16384x14336 (E5M2), MXFP8 in both directions;
  * MoE expert activations, 65536 x 7168 over 64 experts with multinomial
    token counts: grouped MXFP8 in both directions and grouped current
    scaling ("昇腾 Ascend 950" 1 and 2.2).

The oracle runs on all host cores; each test takes seconds to a couple of
minutes.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import dev, host, require_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fq():
    return require_cuda()


def f32bits(a):
    return np.asarray(a, dtype=np.float32).view(np.uint32)


def test_delayed_drift_8192_all_32_steps(fq):
    """Four delayed-scaling sequences (E4M3 / E5M2 x Interval 1 / 5) and
    current scaling in both formats, on the same 32 tensors, bit for bit
    at every step: codes, scale, scale_inv, recorded amax, saturation count,
    and the history ring at the end."""
    keys = [(fmt, iv) for fmt in (oracle.E4M3, oracle.E5M2) for iv in (1, 5)]
    gpu = {k: fq.DelayedScaling(history_len=16, interval=k[1], margin=3, fmt=k[0]) for k in keys}
    ref = {k: oracle.DelayedScaling(16, k[1], 3, k[0]) for k in keys}
    for t in range(32):
        x = synth.config3_step(t)
        xd = dev(x)
        for k in keys:
            got = gpu[k].step(xd, want_sat=True)
            want = ref[k].step(x)
            np.testing.assert_array_equal(host(got["q"]).reshape(-1), want["q"], err_msg=f"{k} step {t}")
            assert f32bits(host(got["scale"]))[0] == f32bits(want["scale"]), (k, t)
            assert f32bits(host(got["scale_inv"]))[0] == f32bits(want["scale_inv"]), (k, t)
            assert int(host(got["sat"])[0]) == int(want["sat"]), (k, t)
            if want["recorded"]:
                assert f32bits(host(got["amax"]))[0] == f32bits(want["amax"]), (k, t)
        for fmt in (oracle.E4M3, oracle.E5M2):
            got = fq.fp8q_cast_per_tensor(xd, fmt, want_sat=True)
            want = oracle.current_scaling(x, fmt)
            np.testing.assert_array_equal(host(got["q"]).reshape(-1), want["q"], err_msg=f"current {fmt} {t}")
            for name in ("amax", "scale", "scale_inv"):
                np.testing.assert_array_equal(f32bits(host(got[name])), f32bits(want[name]), err_msg=name)
            assert host(got["sat"]).tolist() == want["sat"].tolist()
        del xd
    for k in keys:
        s = gpu[k].get()
        r = ref[k]
        assert (s["head"], s["count"], s["step"]) == (r.head, r.count, r.step_no), k
        np.testing.assert_array_equal(f32bits(s["history"]), f32bits(r.hist))
        assert s["nonfinite"] == r.nonfinite
        gpu[k].close()


def _mx_full(fq, x, fmt, offsets=None):
    rows, cols = x.shape
    T = oracle.mx_col_blocks(rows, None if offsets is None else np.array(offsets))
    ld = (T + 15) // 16 * 16 if offsets is not None else T
    off = None if offsets is None else torch.tensor(offsets, dtype=torch.int64, device="cuda")
    r = fq.mxfp8_quantize(dev(x), fmt, fq.BOTH, group_offsets=off, s_col_ld=ld)
    got = {k: host(r[k]) for k in ("q_row", "s_row", "q_col", "s_col")}
    del r
    torch.cuda.empty_cache()
    want = oracle.mx_quantize(x, fmt, 3, offsets=None if offsets is None else np.array(offsets), s_col_ld=ld)
    for k in ("s_row", "q_row", "q_col"):
        np.testing.assert_array_equal(got[k], want[k], err_msg=k)
    np.testing.assert_array_equal(got["s_col"][:, :T], want["s_col"][:, :T], err_msg="s_col")


@pytest.mark.parametrize("name", ["A", "W", "E"])
def test_linear_layer_full(fq, name):
    """A and W in E4M3, E in E5M2: every element of both copies."""
    t = synth.config4()
    _mx_full(fq, t[name], oracle.E5M2 if name == "E" else oracle.E4M3)


def test_moe_mx_full(fq):
    """Grouped MXFP8, 64 experts: every element of both copies."""
    x, offs = synth.config5()
    _mx_full(fq, x, oracle.E4M3, offsets=[int(v) for v in offs])


def test_moe_current_scaling_full(fq):
    """Grouped current scaling, 64 experts: every code, and each expert's
    amax, scale and scale_inv bits."""
    x, offs = synth.config5()
    off = [int(v) for v in offs]
    got = fq.fp8q_cast_per_tensor(dev(x), fq.E4M3, group_offsets=off, want_sat=True)
    want = oracle.current_scaling(x, oracle.E4M3, offsets=np.array(off))
    np.testing.assert_array_equal(host(got["q"]).reshape(-1), want["q"])
    for name in ("amax", "scale", "scale_inv"):
        np.testing.assert_array_equal(f32bits(host(got[name])), f32bits(want[name]), err_msg=name)
    assert host(got["sat"]).tolist() == want["sat"].tolist()
