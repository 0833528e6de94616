"""fp8q_scale_from_amax and the sharded current-scaling path on one GPU.

* The scale kernel against the oracle's scale rule, on special amaxes.
* Two row shards of one tensor, quantized through the exchange path
  (amax per shard, bitwise MAX of the amaxes, scale, cast per shard), equal
  the whole tensor's current scaling from fp8q_cast_per_tensor, bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import dev, host, require_cuda

pytestmark = pytest.mark.gpu

SPECIAL = [0.0, 1.4e-45, 1e-30, 5.877e-39, 1.0, 0.02, 448.0, 57344.0, 1e30, 3.4028235e38,
           float("inf"), float("nan"), -3.0, 2.5e-3]


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("margin", [0, 3, 63])
def test_scale_from_amax_matches_oracle(fmt, margin):
    fq = require_cuda()
    rng = np.random.default_rng(5)
    a = np.concatenate([np.array(SPECIAL, dtype=np.float32),
                        (rng.lognormal(0, 20, 300) * rng.choice([1, -1], 300)).astype(np.float32)])
    r = fq.fp8q_scale_from_amax(dev(a), fmt, margin)
    got_s, got_i = host(r["scale"]), host(r["scale_inv"])
    for k, v in enumerate(a):
        bits = int(np.array([abs(v)], dtype=np.float32).view(np.uint32)[0]) if not np.isnan(v) else 0x7FC00000
        s, _ = oracle.per_tensor_scale(bits, fmt, margin)
        assert got_s[k].view(np.uint32) == np.float32(s).view(np.uint32), (v, got_s[k], s)
        assert got_i[k].view(np.uint32) == oracle.reciprocal(s).view(np.uint32), (v, got_i[k])


def test_two_shards_equal_whole_tensor():
    fq = require_cuda()
    from mxfp8_quantization_amax_gb300 import sharded
    rows, cols, split = 3000, 1024, 1700
    x = synth.normal_outliers(rows, cols, seed=21, std=1.0, p=0.001, factor=300.0, tensor=0)
    off = [0, 500, 1600, 1600, 2900, 3000]
    xd = dev(x)
    whole = fq.fp8q_cast_per_tensor(xd, 0, 2, group_offsets=off)

    def local(r0, r1):
        return [min(max(o, r0), r1) - r0 for o in off]

    parts = [(0, split), (split, rows)]
    amaxes = [fq.fp8q_amax(xd[r0:r1].contiguous(), local(r0, r1)) for r0, r1 in parts]
    # the combine step of sharded.allreduce_amax_: MAX on the FP32 bit patterns
    comb = torch.maximum(amaxes[0].view(torch.int32), amaxes[1].view(torch.int32)).view(torch.float32)
    sc = fq.fp8q_scale_from_amax(comb, 0, 2)
    for r0, r1 in parts:
        q = fq.fp8q_cast_per_tensor(xd[r0:r1].contiguous(), 0, 0, scale_in=sc["scale"],
                                    group_offsets=local(r0, r1), want_amax=False)["q"]
        assert np.array_equal(host(q), host(whole["q"])[r0:r1])
    assert np.array_equal(host(comb).view(np.uint32), host(whole["amax"]).view(np.uint32))
    assert np.array_equal(host(sc["scale"]).view(np.uint32), host(whole["scale"]).view(np.uint32))
    assert np.array_equal(host(sc["scale_inv"]).view(np.uint32), host(whole["scale_inv"]).view(np.uint32))

    # one rank (no process group): the module's path is current scaling of the whole tensor
    one = sharded.current_scaling(xd, 0, 2, group_offsets=off)
    assert np.array_equal(host(one["q"]), host(whole["q"]))
    fq.check_device()
