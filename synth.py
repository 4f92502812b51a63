"""Seeded synthetic rank buffers shared by the tests, the smoke check and the bench.

This module draws random inputs and nothing else: it holds none of the relay method's
arithmetic, so both the CUDA path and the CPU oracle can be fed from it.

Recipe: the input of active rank ``r`` in workload ``c`` is drawn from a torch
``Generator`` seeded with ``1000 * c + r``; fp32 and bf16 values are N(0, 1) (bf16 is
the fp32 draw rounded to nearest-even by torch), int32 values are uniform on
[-2**20, 2**20].  Helpers receive no input.
"""
from __future__ import annotations

import numpy as np
import torch

DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16, "i32": torch.int32}
ESIZE = {"f32": 4, "bf16": 2, "i32": 4}


def seed(config: int, rank: int) -> int:
    return 1000 * config + rank


def rank_input(config: int, rank: int, numel: int, dtype: str, device="cpu") -> torch.Tensor:
    """One active rank's input, drawn on ``device`` (CPU or CUDA generator)."""
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(seed(config, rank))
    if dtype == "i32":
        return torch.randint(-(2 ** 20), 2 ** 20 + 1, (numel,), generator=g, device=dev,
                             dtype=torch.int32)
    x = torch.randn(numel, generator=g, device=dev, dtype=torch.float32)
    return x if dtype == "f32" else x.to(torch.bfloat16)


def rank_inputs(config: int, A: int, numel: int, dtype: str, device="cpu"):
    return [rank_input(config, r, numel, dtype, device) for r in range(A)]


def to_numpy(t: torch.Tensor) -> np.ndarray:
    """Host copy as numpy; bf16 becomes its raw uint16 bit pattern."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def poison_(t: torch.Tensor, byte: int = 0xA5) -> torch.Tensor:
    """Fill a buffer with a recognisable byte pattern (scratch and canaries)."""
    t.view(torch.uint8).fill_(byte)
    return t
