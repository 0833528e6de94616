"""The exchange step of current scaling for a row-sharded tensor, on CPU.

Two gloo ranks each hold half the rows of a grouped tensor.  Each computes
its part's per-group amax with the oracle, the ranks combine them with
sharded.allreduce_amax_ (the library's MAX all-reduce on FP32 bit
patterns), and each casts its part with the oracle using the combined
amax.  The result must equal the oracle's current scaling of the whole
tensor, bit for bit, including a group whose amax is NaN and one that is
empty on one rank.
"""
import os
import socket
import sys

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

ROWS, COLS = 64, 256
GLOBAL_OFF = [0, 10, 40, 64, 64]   # 4 groups, the last one empty
SPLIT = 32                          # rank 0: rows [0, 32), rank 1: [32, 64)
FMT, MARGIN = 0, 2


def _input():
    import synth
    x = synth.normal_outliers(ROWS, COLS, seed=11, std=1.0, p=0.01, factor=100.0, tensor=0).copy()
    x[45, 7] = 0x7FC0          # a NaN in group 2 (rank 1's part)
    x[3, 100] = 0x7F80         # +Inf in group 0 (rank 0's part)
    return x


def _local_offsets(r0, r1):
    return [min(max(o, r0), r1) - r0 for o in GLOBAL_OFF]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        from mxfp8_quantization_amax_gb300 import sharded
        x = _input()
        r0, r1 = (0, SPLIT) if rank == 0 else (SPLIT, ROWS)
        part = np.ascontiguousarray(x[r0:r1]).reshape(-1)
        off = _local_offsets(r0, r1)
        bits = [oracle.amax_bits(part, off[g] * COLS, off[g + 1] * COLS) for g in range(len(off) - 1)]
        amax = torch.tensor(np.array(bits, dtype=np.uint32).view(np.float32))
        sharded.allreduce_amax_(amax)
        gbits = amax.numpy().view(np.uint32)
        qp = np.zeros(part.size, dtype=np.uint8)
        scales = []
        for g in range(len(off) - 1):
            s, _ = oracle.per_tensor_scale(int(gbits[g]), FMT, MARGIN)
            oracle.cast(part, s, FMT, off[g] * COLS, off[g + 1] * COLS, out=qp, nthreads=1)
            scales.append(np.float32(s))
        q.put((rank, qp, gbits.copy(), np.array(scales, dtype=np.float32)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_sharded_current_scaling_equals_whole_tensor():
    import oracle
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = dict((r, (qp, a, s)) for r, qp, a, s in (q.get(timeout=120) for _ in range(world)))
    for p in procs:
        p.join(120)
        assert p.exitcode == 0

    whole = oracle.current_scaling(_input(), FMT, MARGIN, offsets=GLOBAL_OFF, nthreads=1)
    want_amax_bits = whole["amax"].view(np.uint32)
    assert np.isnan(whole["amax"][2]) and np.isinf(whole["amax"][0])
    for r in range(world):
        qp, abits, scales = got[r]
        r0, r1 = (0, SPLIT) if r == 0 else (SPLIT, ROWS)
        assert np.array_equal(qp, whole["q"][r0 * COLS:r1 * COLS])
        assert np.array_equal(abits, want_amax_bits)
        assert np.array_equal(scales.view(np.uint32), whole["scale"].view(np.uint32))
