"""Per-tensor current scaling of a tensor whose rows are split across ranks.

The scale of current scaling needs the amax of the whole tensor ("HiFloat8：
高性能训练之路" 1.2, eq. 1), so a tensor sharded by rows across devices has one
exchange step: each rank reduces its own part (fp8q_amax), the per-group
amaxes are combined with a MAX all-reduce, and each rank computes the scale
(fp8q_scale_from_amax) and casts its part with it (fp8q_cast_per_tensor).
The result is bit-identical to current scaling of the whole tensor on one
device.  MXFP8 needs no exchange: its blocks are independent, so a row split
at multiples of 32 (and at group boundaries) quantizes each part alone.

The all-reduce runs on the amaxes' FP32 bit patterns viewed as int32.  An
amax is non-negative, so its bits order like its values; a NaN amax (bits
above +Inf's) wins the max, which keeps the NaN a single device would have
produced.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from . import E4M3, fp8q_amax, fp8q_cast_per_tensor, fp8q_scale_from_amax


def allreduce_amax_(amax: torch.Tensor, group=None) -> torch.Tensor:
    """In place: amax[g] = max over ranks of amax[g] (float32, by bit pattern)."""
    if amax.dtype != torch.float32:
        raise TypeError("amax must be float32")
    if dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1:
        dist.all_reduce(amax.view(torch.int32), op=dist.ReduceOp.MAX, group=group)
    return amax


def current_scaling(x_local: torch.Tensor, fmt: int = E4M3, margin: int = 0, group_offsets=None,
                    group=None, q: torch.Tensor | None = None) -> dict:
    """Current scaling of this rank's rows of a row-sharded tensor.

    group_offsets are the row offsets of the groups within this rank's part
    (the same number of groups on every rank; empty groups allowed).
    Returns dict(q, amax, scale, scale_inv); amax and the scales are the
    whole tensor's, identical on every rank.
    """
    amax = fp8q_amax(x_local, group_offsets)
    allreduce_amax_(amax, group)
    sc = fp8q_scale_from_amax(amax, fmt, margin)
    r = fp8q_cast_per_tensor(x_local, fmt, 0, scale_in=sc["scale"], group_offsets=group_offsets,
                             want_amax=False, q=q)
    return {"q": r["q"], "amax": amax, "scale": sc["scale"], "scale_inv": sc["scale_inv"]}
