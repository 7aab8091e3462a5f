"""Small helpers for the GPU tests: host <-> device copies of bit patterns, canary guard bands."""
from __future__ import annotations

import numpy as np
import torch

DEV = "cuda:0"


def bf16_to_dev(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits, np.uint16).view(np.int16)).view(torch.bfloat16).to(DEV)


def dev_to_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def f16_dev_to_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def f16_bits_to_dev(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits, np.uint16).view(np.int16)).view(torch.float16).to(DEV)


class Guarded:
    """A device buffer with canary bands before and after the payload (16-byte aligned payload)."""

    PAD = 256  # bytes on each side
    CANARY = 0xA5

    def __init__(self, shape, dtype: torch.dtype):
        self.shape, self.dtype = tuple(shape), dtype
        nbytes = int(np.prod(self.shape)) * torch.empty((), dtype=dtype).element_size()
        self.nbytes = nbytes
        self.raw = torch.full((nbytes + 2 * self.PAD,), self.CANARY, dtype=torch.uint8, device=DEV)
        self.t = self.raw[self.PAD:self.PAD + nbytes].view(dtype).view(self.shape)

    def canaries_intact(self) -> bool:
        raw = self.raw.cpu().numpy()
        return bool(np.all(raw[:self.PAD] == self.CANARY) and np.all(raw[self.PAD + self.nbytes:] == self.CANARY))
