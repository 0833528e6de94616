"""Helpers for the GPU parity tests: host <-> device copies of the seeded
inputs and guarded output buffers (canary bytes on both sides of every
output catch stray writes, since no memory checker runs on the GPU machine)."""
import numpy as np
import torch

GUARD = 4096
CANARY = 0xA5


def require_cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import mxfp8_quantization_amax_gb300 as fq
    fq.build()
    return fq


def dev(a: np.ndarray) -> torch.Tensor:
    """numpy -> CUDA tensor: uint16 arrays become bfloat16 (same bits)."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(a).cuda()


def host(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu()
    if t.dtype == torch.int64:
        return t.numpy().view(np.uint64)
    return t.numpy()


class Guarded:
    """A uint8/float/int64 CUDA buffer with canary bytes around it."""

    def __init__(self, shape, dtype=torch.uint8, device="cuda"):
        n = int(np.prod(shape)) if len(shape) else 1
        esz = torch.tensor([], dtype=dtype).element_size()
        self.nbytes = n * esz
        self.raw = torch.full((GUARD + self.nbytes + GUARD,), CANARY, dtype=torch.uint8, device=device)
        self.t = self.raw[GUARD:GUARD + self.nbytes].view(dtype).view(*shape) if n else \
            torch.empty(shape, dtype=dtype, device=device)

    def check(self):
        head = self.raw[:GUARD]
        tail = self.raw[GUARD + self.nbytes:]
        assert bool((head == CANARY).all()), "write before the output buffer"
        assert bool((tail == CANARY).all()), "write after the output buffer"


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)
