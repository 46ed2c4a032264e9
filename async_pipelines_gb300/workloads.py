"""Seeded synthetic workloads for the warp-specialized GEMM.

This module only *draws* inputs; it holds none of the GEMM arithmetic, so the
CPU oracle and the CUDA path can both take their inputs from here without
sharing any of the computation they are compared on.

Every workload is the dense GEMM ``D[l] = alpha * A[l] @ B[l] + beta * C[l]``
with bf16 operands, named by what it is and its sizes:

* A is row-major ``L x M x K`` (K contiguous, "K-major").
* B is column-major ``K x N`` per batch, i.e. stored ``L x N x K`` with K
  contiguous, so both operands are K-major (the operand layout of the SM90
  cooperative kernel page and of the SM100 mainloop on the discussion page).
* C and D are row-major ``L x M x N``; batches are packed.

Distributions (readings where the cited sources are silent, stated once here):

* ``uniform``: fp32 ``torch.rand * 2 - 1`` (so ``[-1, 1)``), rounded to bf16
  round-to-nearest-even.
* ``normal(s)``: fp32 ``torch.randn * s`` (``s`` is the standard deviation),
  rounded to bf16.
* A and B come from one ``torch.Generator`` seeded with the workload's seed,
  A drawn first; C from a second generator seeded with ``seed + 100``.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    L: int
    ab_dist: tuple          # ("uniform",) or ("normal", std)
    c_dist: Optional[tuple]  # None means no C (beta must be 0)
    alpha: float
    beta: float
    seed: int
    streamout: bool = False

    @property
    def flops(self) -> int:
        """Algorithmic FLOPs, 2*M*N*K*L (no padding of ragged tiles)."""
        return 2 * self.M * self.N * self.K * self.L

    def algorithmic_bytes(self) -> int:
        """Compulsory HBM bytes: A + B (+ C if read) + D (+ staging)."""
        b = 2 * self.L * (self.M * self.K + self.N * self.K + self.M * self.N)
        if self.c_dist is not None and self.beta != 0.0:
            b += 2 * self.L * self.M * self.N
        if self.streamout:
            b += 2 * staging_elems(self.M, self.N, self.L)
        return b


# Stream-out hands finished output tiles over at this granularity.
STAGING_TILE = 128


def staging_tiles(M: int, N: int, L: int) -> int:
    """Number of 128x128 stream-out tiles, L * ceil(M/128) * ceil(N/128)."""
    t = STAGING_TILE
    return L * ((M + t - 1) // t) * ((N + t - 1) // t)


def staging_elems(M: int, N: int, L: int) -> int:
    return staging_tiles(M, N, L) * STAGING_TILE * STAGING_TILE


WORKLOADS = {
    w.name: w
    for w in [
        Workload("gemm_256x256x256", 256, 256, 256, 1,
                 ("uniform",), None, 1.0, 0.0, seed=1),
        Workload("gemm_4096x4096x4096", 4096, 4096, 4096, 1,
                 ("uniform",), None, 1.0, 0.0, seed=2),
        Workload("gemm_8192x8192x8192_alpha_beta", 8192, 8192, 8192, 1,
                 ("uniform",), ("normal", 1.0), 1.5, 0.5, seed=3),
        Workload("gemm_batched4_5000x3000x4000_ragged", 5000, 3000, 4000, 4,
                 ("normal", 0.5), ("uniform",), 1.0, 1.0, seed=4),
        Workload("gemm_streamout_8192x8192x4096", 8192, 8192, 4096, 1,
                 ("uniform",), None, 1.0, 0.0, seed=5, streamout=True),
    ]
}

# The single-GPU headline workload: the 8192^3 GEMM with the full C epilogue.
HEADLINE = "gemm_8192x8192x8192_alpha_beta"
STREAMOUT = "gemm_streamout_8192x8192x4096"

# Informational shapes beside the five above (measured, not parity configs):
# a skinny GEMM bound by writing D.
EXTRA_WORKLOADS = {
    w.name: w
    for w in [
        Workload("gemm_8192x8192x64_skinny", 8192, 8192, 64, 1,
                 ("uniform",), None, 1.0, 0.0, seed=6),
    ]
}
SKINNY = "gemm_8192x8192x64_skinny"


def workload(name: str) -> Workload:
    """A workload of either table by name."""
    return WORKLOADS[name] if name in WORKLOADS else EXTRA_WORKLOADS[name]


def _draw(gen: torch.Generator, shape, dist) -> torch.Tensor:
    if dist[0] == "uniform":
        x = torch.rand(shape, generator=gen, dtype=torch.float32) * 2.0 - 1.0
    elif dist[0] == "normal":
        x = torch.randn(shape, generator=gen, dtype=torch.float32) * float(dist[1])
    elif dist[0] == "int":
        lo, hi = int(dist[1]), int(dist[2])
        x = torch.randint(lo, hi + 1, shape, generator=gen).to(torch.float32)
    else:
        raise ValueError(f"unknown distribution {dist!r}")
    return x.to(torch.bfloat16)


def make_inputs(M: int, N: int, K: int, L: int, ab_dist, c_dist, seed: int):
    """Returns CPU bf16 tensors A (L,M,K), B (L,N,K), C (L,M,N) or None."""
    g = torch.Generator().manual_seed(seed)
    A = _draw(g, (L, M, K), ab_dist)
    B = _draw(g, (L, N, K), ab_dist)
    C = None
    if c_dist is not None:
        gc = torch.Generator().manual_seed(seed + 100)
        C = _draw(gc, (L, M, N), c_dist)
    return A, B, C


def workload_inputs(w: Workload):
    return make_inputs(w.M, w.N, w.K, w.L, w.ab_dist, w.c_dist, w.seed)


def bf16_bits(t: torch.Tensor):
    """Raw bf16 bit patterns of a CPU tensor as a numpy uint16 array."""
    import numpy as np
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)
