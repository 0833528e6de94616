"""GPU parity: delayed scaling (history ring, Interval, margin, first step
with current scaling, non-finite flag, checkpoint get/set) step by step
against the oracle's state machine."""
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


def compare_step(got, ref, t):
    np.testing.assert_array_equal(host(got["q"]).reshape(-1), ref["q"], err_msg=f"step {t}")
    assert f32bits(host(got["scale"]))[0] == f32bits(ref["scale"]), t
    assert f32bits(host(got["scale_inv"]))[0] == f32bits(ref["scale_inv"]), t
    if got["sat"] is not None:
        assert host(got["sat"])[0] == ref["sat"], t
    if ref["recorded"]:
        assert f32bits(host(got["amax"]))[0] == f32bits(ref["amax"]), t


def compare_state(st, ref):
    s = st.get()
    assert s["head"] == ref.head and s["count"] == ref.count and s["step"] == ref.step_no
    np.testing.assert_array_equal(f32bits(s["history"]), f32bits(ref.hist))
    assert s["nonfinite"] == ref.nonfinite


@pytest.mark.parametrize("interval", [1, 5])
@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_drifting_tensor_32_steps(fq, interval, fmt):
    """32 steps of x_t = sigma_t z_t, sigma drifting by U(0.8, 1.25) per step,
    history 16, margin 3 (1024x1024 here; the 8192x8192 sequence is in test_gpu_full_size.py)."""
    st = fq.DelayedScaling(history_len=16, interval=interval, margin=3, fmt=fmt)
    ref = oracle.DelayedScaling(16, interval, 3, fmt)
    for t in range(32):
        x = synth.config3_step(t, rows=1024, cols=1024)
        got = st.step(dev(x), want_sat=True)
        compare_step(got, ref.step(x), t)
    compare_state(st, ref)
    st.close()


def test_history_wraps_and_fifo(fq):
    """History length 3, amax falling then rising: the oldest entry drops out."""
    st = fq.DelayedScaling(history_len=3, interval=1, margin=0, fmt=oracle.E4M3)
    ref = oracle.DelayedScaling(3, 1, 0, oracle.E4M3)
    for t, a in enumerate([64.0, 8.0, 4.0, 2.0, 1.0, 0.5, 100.0, 3.0]):
        x = synth.to_bf16_bits((np.linspace(-1, 1, 4096) * a).astype(np.float32)).reshape(64, 64)
        compare_step(st.step(dev(x), want_sat=True), ref.step(x), t)
        compare_state(st, ref)


def test_interval_3_history_1_fp32(fq):
    st = fq.DelayedScaling(history_len=1, interval=3, margin=1, fmt=oracle.E5M2)
    ref = oracle.DelayedScaling(1, 3, 1, oracle.E5M2)
    for t in range(10):
        x = synth.f32_tensor(37, 129, seed=100 + t, std=float(2.0 ** (t - 5)))
        compare_step(st.step(dev(x), want_sat=True), ref.step(x), t)
    compare_state(st, ref)


def test_nonfinite_flag_and_reset(fq):
    st = fq.DelayedScaling(history_len=4, interval=1, margin=0, fmt=oracle.E4M3)
    ref = oracle.DelayedScaling(4, 1, 0, oracle.E4M3)
    x = synth.normal_outliers(32, 64, seed=7)
    compare_step(st.step(dev(x)), ref.step(x), 0)
    xn = x.copy()
    xn[5, 9] = 0x7FC0  # NaN
    compare_step(st.step(dev(xn)), ref.step(xn), 1)  # scaled with the old history, records NaN
    compare_state(st, ref)
    assert st.get()["nonfinite"]
    compare_step(st.step(dev(x)), ref.step(x), 2)  # history max is NaN: scale 1
    st.reset()
    ref.reset()
    compare_step(st.step(dev(x)), ref.step(x), 0)  # current scaling again
    compare_state(st, ref)
    assert not st.get()["nonfinite"]


def test_checkpoint_get_set(fq):
    """A state restored from get() continues exactly like the original."""
    a = fq.DelayedScaling(history_len=5, interval=2, margin=2, fmt=oracle.E4M3)
    ref = oracle.DelayedScaling(5, 2, 2, oracle.E4M3)
    xs = [synth.config3_step(t, rows=64, cols=256) for t in range(12)]
    for t in range(7):
        compare_step(a.step(dev(xs[t])), ref.step(xs[t]), t)
    s = a.get()
    b = fq.DelayedScaling(history_len=5, interval=2, margin=2, fmt=oracle.E4M3)
    b.set(s["history"], s["head"], s["count"], s["step"])
    for t in range(7, 12):
        r = ref.step(xs[t])
        compare_step(a.step(dev(xs[t])), r, t)
        compare_step(b.step(dev(xs[t])), r, t)
    compare_state(b, ref)
