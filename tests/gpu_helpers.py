"""Shared plumbing for the GPU parity tests (no GEMM arithmetic here)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from async_pipelines_gb300 import workloads
from tests.numerics import assert_gemm_close


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


def check_every_row(d_bits: np.ndarray, A, B, C, M: int, N: int, K: int, L: int,
                    alpha: float, beta: float, what: str, chunk: int = 512):
    """Every element of a GPU result (bf16 bits, L*M x N) against the oracle,
    in slabs of `chunk` output rows so that the fp64 reference of a
    full-size workload is never held whole."""
    d_bits = np.asarray(d_bits).reshape(L * M, N)
    Ab, Bb = bits_of(A), bits_of(B)
    Cb = None if C is None else bits_of(C)
    for r0 in range(0, L * M, chunk):
        rows = np.arange(r0, min(r0 + chunk, L * M), dtype=np.int64)
        ref = oracle.gemm_rows(Ab, Bb, Cb, M, N, K, L, alpha, beta, rows=rows)
        assert_gemm_close(d_bits[rows], ref, K, f"{what}, rows {rows[0]}..{rows[-1]}")
