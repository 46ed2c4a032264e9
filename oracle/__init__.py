"""CPU oracle for the warp-specialized GEMM (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The product library never does; the two
share no code. The arithmetic lives in ``gemm_ref.cpp`` (plain fp64 triple
loop, the definition ``D = alpha*A*B + beta*C`` written out); this module only
compiles it and marshals numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(_HERE, "gemm_ref.cpp")
LIB = os.path.join(_HERE, "libgemm_ref.so")

_lib = None


def compile_oracle(src: str = SRC, out: str = LIB) -> str:
    """Compiles the oracle with plain -O2 (no fast-math, so fp64 is IEEE)."""
    cmd = ["g++", "-std=c++17", "-O2", "-fno-fast-math", "-ffp-contract=off",
           "-fPIC", "-shared", "-pthread", src, "-o", out]
    subprocess.run(cmd, check=True)
    return out


def _needs_build() -> bool:
    return (not os.path.exists(LIB)) or os.path.getmtime(LIB) < os.path.getmtime(SRC)


def load(path: Optional[str] = None):
    """Loads (building first if stale) the oracle library; returns the CDLL."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        if _needs_build():
            compile_oracle()
        _lib = _bind(ctypes.CDLL(LIB))
    return _lib


def _bind(lib):
    f = lib.oracle_gemm_rows
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                  ctypes.c_int64, ctypes.c_int64, ctypes.c_float,
                  ctypes.c_float, ctypes.c_void_p, ctypes.c_int64,
                  ctypes.c_int]
    return lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def gemm_rows(A: np.ndarray, B: np.ndarray, C: Optional[np.ndarray],
              M: int, N: int, K: int, L: int, alpha: float, beta: float,
              rows: Optional[Sequence[int]] = None, threads: int = 0,
              lib=None) -> np.ndarray:
    """fp64 reference rows of ``alpha*A@B + beta*C``.

    A: uint16 bf16 bits, L*M*K (row-major); B: uint16, L*N*K (each batch is
    column-major K x N, i.e. N x K with K contiguous); C: uint16 L*M*N or
    None. ``rows`` are global row ids ``l*M + i`` (default: every row). The
    result has shape ``(len(rows), N)``.
    """
    lib = lib or load()
    A = np.ascontiguousarray(A, dtype=np.uint16).reshape(-1)
    B = np.ascontiguousarray(B, dtype=np.uint16).reshape(-1)
    if C is not None:
        C = np.ascontiguousarray(C, dtype=np.uint16).reshape(-1)
    if rows is None:
        rows = np.arange(L * M, dtype=np.int64)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    out = np.zeros((rows.size, N), dtype=np.float64)
    if threads <= 0:
        threads = len(os.sched_getaffinity(0))
    rc = lib.oracle_gemm_rows(_ptr(A), _ptr(B), _ptr(C), _ptr(out), M, N, K, L,
                              float(alpha), float(beta), _ptr(rows),
                              rows.size, int(threads))
    if rc != 0:
        raise ValueError(f"oracle_gemm_rows rejected its arguments (rc={rc})")
    return out


def gemm(A, B, C, M, N, K, L, alpha, beta, threads: int = 0, lib=None):
    """Full fp64 reference, shape (L, M, N)."""
    return gemm_rows(A, B, C, M, N, K, L, alpha, beta, None, threads,
                     lib).reshape(L, M, N)
