"""Shared plumbing for the GPU parity tests (no GEMM arithmetic here)."""
from __future__ import annotations

import numpy as np
import torch

from async_pipelines_gb300 import workloads


def bits_of(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor (any device) -> numpy uint16 bit patterns."""
    return workloads.bf16_bits(t.detach().cpu())


def to_dev(t):
    return None if t is None else t.cuda()


def sample_rows(M: int, L: int, n_random: int, seed: int, tile: int = 128) -> np.ndarray:
    """Global row ids l*M + i: the first/last row of every batch, the rows on
    both sides of every 8th tile boundary, the last tile's rows, and
    `n_random` seeded random rows."""
    rows = set()
    for l in range(L):
        base = l * M
        rows.update({base, base + M - 1})
        for b in range(tile, M, tile * 8):
            rows.update({base + b - 1, base + b})
        last = (M - 1) // tile * tile
        rows.update(base + i for i in range(last, M, max(1, (M - last) // 8)))
    rng = np.random.default_rng(seed)
    rows.update(int(r) for r in rng.integers(0, L * M, size=n_random))
    return np.array(sorted(rows), dtype=np.int64)
