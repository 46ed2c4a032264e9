"""Pins the CPU oracle to things other than itself (no GPU needed).

Each test fixes the oracle against mathematics the GEMM definition
D = alpha*A*B + beta*C determines on its own: closed forms (identity B,
all-ones operands, alpha = 0), exact rational arithmetic on tiny shapes,
exact integer matrix products, linearity, and a hand-worked example. Together
they catch a dropped term, a wrong sign, a swapped or transposed operand and a
wrong batch stride (``test_oracle_mutants.py`` plants exactly those mistakes).
"""
from __future__ import annotations

import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from async_pipelines_gb300 import workloads
from tests.numerics import bf16_bits_to_f64, f64_to_bf16_bits

HERE = os.path.dirname(os.path.abspath(__file__))


def bits(t: torch.Tensor) -> np.ndarray:
    return workloads.bf16_bits(t)


def rand_bits(shape, seed, dist=("uniform",)):
    g = torch.Generator().manual_seed(seed)
    return bits(workloads._draw(g, shape, dist))


# ---------------------------------------------------------------- closed forms

@pytest.mark.parametrize("n", [1, 5, 64, 130])
def test_identity_b_returns_a(n):
    """B = I (K = N): every output element equals the A element exactly."""
    M, L = 37, 2
    A = rand_bits((L, M, n), 11)
    eye = torch.eye(n, dtype=torch.bfloat16).expand(L, n, n).contiguous()
    ref = oracle.gemm(A, bits(eye), None, M, n, n, L, 1.0, 0.0)
    np.testing.assert_array_equal(ref, bf16_bits_to_f64(A).reshape(L, M, n))


@pytest.mark.parametrize("K", [1, 7, 256, 4000, 4096])
def test_all_ones_gives_k(K):
    """All-ones A and B: each element is exactly K (K is exact in bf16 here)."""
    M, N, L = 3, 5, 2
    ones_a = np.full(L * M * K, 0x3F80, dtype=np.uint16)   # bf16 1.0
    ones_b = np.full(L * N * K, 0x3F80, dtype=np.uint16)
    ref = oracle.gemm(ones_a, ones_b, None, M, N, K, L, 1.0, 0.0)
    assert np.all(ref == float(K))


def test_alpha_zero_is_beta_c():
    M, N, K, L = 9, 17, 33, 3
    A, B = rand_bits((L, M, K), 1), rand_bits((L, N, K), 2)
    C = rand_bits((L, M, N), 3, ("normal", 1.0))
    beta = 0.5
    ref = oracle.gemm(A, B, C, M, N, K, L, 0.0, beta)
    np.testing.assert_array_equal(ref, beta * bf16_bits_to_f64(C).reshape(L, M, N))


def test_beta_zero_never_reads_c():
    """beta == 0 skips C: NaNs in C do not appear, and C may be absent."""
    M, N, K, L = 4, 6, 8, 1
    A, B = rand_bits((L, M, K), 4), rand_bits((L, N, K), 5)
    nan_c = np.full(L * M * N, 0x7FC0, dtype=np.uint16)     # bf16 NaN
    with_nan = oracle.gemm(A, B, nan_c, M, N, K, L, 1.0, 0.0)
    without = oracle.gemm(A, B, None, M, N, K, L, 1.0, 0.0)
    assert np.isfinite(with_nan).all()
    np.testing.assert_array_equal(with_nan, without)


def test_k_zero_gives_beta_c():
    M, N, L = 5, 8, 2
    C = rand_bits((L, M, N), 6)
    ref = oracle.gemm(np.zeros(0, np.uint16), np.zeros(0, np.uint16), C,
                      M, N, 0, L, 1.0, 2.0)
    np.testing.assert_array_equal(ref, 2.0 * bf16_bits_to_f64(C).reshape(L, M, N))


# -------------------------------------------------- exact arithmetic, by brute force

def _exact(Af, Bf, Cf, M, N, K, L, alpha, beta):
    """Rational GEMM on tiny shapes: every input is a dyadic rational."""
    out = [[[Fraction(0)] * N for _ in range(M)] for _ in range(L)]
    for l in range(L):
        for i in range(M):
            for j in range(N):
                s = sum((Fraction(float(Af[l, i, k])) * Fraction(float(Bf[l, j, k]))
                         for k in range(K)), Fraction(0))
                v = Fraction(float(alpha)) * s
                if beta != 0:
                    v += Fraction(float(beta)) * Fraction(float(Cf[l, i, j]))
                out[l][i][j] = v
    return out


@pytest.mark.parametrize("seed", range(12))
def test_bruteforce_rational(seed):
    """Tiny shapes against exact rationals, within fp64 summation error.

    The bound is the textbook one for a recursive sum of K products plus the
    scaling and the C term: (K + 2) * 2**-53 * (|alpha| sum|a b| + |beta c|).
    """
    rng = np.random.default_rng(seed)
    M, N, K = (int(x) for x in rng.integers(1, 9, size=3))
    L = int(rng.integers(1, 3))
    alpha = float(np.float32(rng.choice([1.0, 1.5, -0.75, 3.0])))
    beta = float(np.float32(rng.choice([0.0, 0.5, -2.0, 1.0])))
    A = rand_bits((L, M, K), 100 + seed, ("normal", 1.0))
    B = rand_bits((L, N, K), 200 + seed, ("normal", 1.0))
    C = rand_bits((L, M, N), 300 + seed) if beta != 0 else None
    Af = bf16_bits_to_f64(A).reshape(L, M, K)
    Bf = bf16_bits_to_f64(B).reshape(L, N, K)
    Cf = bf16_bits_to_f64(C).reshape(L, M, N) if C is not None else None
    ref = oracle.gemm(A, B, C, M, N, K, L, alpha, beta)
    exact = _exact(Af, Bf, Cf, M, N, K, L, alpha, beta)
    for l in range(L):
        for i in range(M):
            for j in range(N):
                mag = abs(alpha) * sum(abs(Af[l, i, k] * Bf[l, j, k]) for k in range(K))
                if beta != 0:
                    mag += abs(beta * Cf[l, i, j])
                bound = (K + 2) * 2.0 ** -53 * mag
                err = abs(Fraction(ref[l, i, j]) - exact[l][i][j])
                assert err <= Fraction(bound), (l, i, j, ref[l, i, j], float(exact[l][i][j]))


def test_integer_inputs_exact_vs_integer_matmul():
    """Integer-valued inputs in [-4, 4]: the fp64 oracle is exact, so it must
    equal the exact integer product taken by numpy's int64 matmul, with B read
    as the column-major K x N operand (B_kn[l, k, j] = B_stored[l, j, k])."""
    M, N, K, L = 37, 29, 50, 3
    g = torch.Generator().manual_seed(7)
    A = workloads._draw(g, (L, M, K), ("int", -4, 4))
    B = workloads._draw(g, (L, N, K), ("int", -4, 4))
    C = workloads._draw(g, (L, M, N), ("int", -4, 4))
    ref = oracle.gemm(bits(A), bits(B), bits(C), M, N, K, L, 2.0, -3.0)
    Ai = A.to(torch.int64).numpy()
    Bi = B.to(torch.int64).numpy()
    Ci = C.to(torch.int64).numpy()
    expect = 2 * np.matmul(Ai, np.transpose(Bi, (0, 2, 1))) - 3 * Ci
    np.testing.assert_array_equal(ref, expect.astype(np.float64))


def test_linearity_in_alpha_beta():
    M, N, K, L = 21, 19, 40, 2
    A, B = rand_bits((L, M, K), 8), rand_bits((L, N, K), 9)
    C = rand_bits((L, M, N), 10, ("normal", 1.0))
    d = oracle.gemm(A, B, C, M, N, K, L, 1.5, 0.5)
    ab = oracle.gemm(A, B, None, M, N, K, L, 1.0, 0.0)
    c = oracle.gemm(A, B, C, M, N, K, L, 0.0, 1.0)
    np.testing.assert_allclose(d, 1.5 * ab + 0.5 * c, rtol=1e-14, atol=1e-14)


def test_rows_subset_matches_full():
    M, N, K, L = 33, 12, 20, 3
    A, B = rand_bits((L, M, K), 12), rand_bits((L, N, K), 13)
    C = rand_bits((L, M, N), 14)
    full = oracle.gemm(A, B, C, M, N, K, L, 1.0, 1.0).reshape(L * M, N)
    rows = [0, 5, 32, 33, 70, L * M - 1]
    part = oracle.gemm_rows(A, B, C, M, N, K, L, 1.0, 1.0, rows=rows, threads=3)
    np.testing.assert_array_equal(part, full[rows])


def test_thread_count_does_not_change_result():
    M, N, K, L = 40, 16, 64, 1
    A, B = rand_bits((L, M, K), 15), rand_bits((L, N, K), 16)
    one = oracle.gemm(A, B, None, M, N, K, L, 1.0, 0.0, threads=1)
    many = oracle.gemm(A, B, None, M, N, K, L, 1.0, 0.0, threads=7)
    np.testing.assert_array_equal(one, many)


# ---------------------------------------------------------------- hand-worked

def load_handworked():
    path = os.path.join(HERE, "golden", "gemm_handworked_2x3x4.txt")
    rows = {"A": [], "B": [], "C": [], "D": []}
    scal = {}
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            if key in rows:
                rows[key].append([float(v) for v in vals])
            else:
                scal[key] = float(vals[0])
    A = np.array(rows["A"])            # M x K
    Bkn = np.array(rows["B"])          # K x N as printed
    C = np.array(rows["C"])
    D = np.array(rows["D"])
    return A, Bkn, C, D, scal["alpha"], scal["beta"]


def test_handworked_fixture():
    A, Bkn, C, D, alpha, beta = load_handworked()
    M, K = A.shape
    N = Bkn.shape[1]
    ref = oracle.gemm(f64_to_bf16_bits(A), f64_to_bf16_bits(Bkn.T.copy()),
                      f64_to_bf16_bits(C), M, N, K, 1, alpha, beta)
    np.testing.assert_array_equal(ref[0], D)


# ---------------------------------------------------------------- arguments

def test_rejects_missing_c_with_nonzero_beta():
    A = np.zeros(4, np.uint16)
    with pytest.raises(ValueError):
        oracle.gemm(A, A, None, 2, 2, 1, 1, 1.0, 1.0)


def test_rejects_row_out_of_range():
    A = np.zeros(4, np.uint16)
    with pytest.raises(ValueError):
        oracle.gemm_rows(A, A, None, 2, 2, 1, 1, 1.0, 0.0, rows=[2])
