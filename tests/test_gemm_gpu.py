"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Tolerance (per element): |d - ref| <= ulp_bf16(ref) + 1e-3 * sqrt(K / 64).
Integer-valued inputs make the fp32 accumulation exact, so there the bf16
result must equal the oracle rounded to bf16 bit for bit.
"""
from __future__ import annotations

import os
import numpy as np
import pytest
import torch

import oracle
from async_pipelines_gb300 import gemm_ws, workloads
from tests.gpu_helpers import bits_of, check_every_row, sample_rows, to_dev
from tests.numerics import assert_gemm_close, f64_to_bf16_bits
from tests.test_oracle import load_handworked

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gw():
    g = gemm_ws.GemmWS(0)
    yield g
    assert g.query_status() == gemm_ws.OK
    g.close()


@pytest.fixture(scope="module", params=[2, 1], ids=["cta_pair", "cta_single"])
def gw_each(request):
    """A handle per tile configuration, chosen at create time by the
    environment: CTA-pair 256x256 tiles (the default) and single-CTA 128x256
    tiles."""
    cg = request.param
    keys = ("GEMM_WS_CTA_GROUP",)
    old = {k: os.environ.get(k) for k in keys}
    os.environ["GEMM_WS_CTA_GROUP"] = str(cg)
    try:
        g = gemm_ws.GemmWS(0)
    finally:
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    yield g
    assert g.query_status() == gemm_ws.OK
    g.close()


def run_case(gw, M, N, K, L, alpha, beta, ab=("uniform",), cd=None, seed=0, rows=None,
             streamout=False):
    """Runs one GEMM on the GPU; returns (D bits, oracle rows, rows or None)."""
    A, B, C = workloads.make_inputs(M, N, K, L, ab, cd, seed)
    Ad, Bd, Cd = to_dev(A), to_dev(B), to_dev(C)
    D = torch.empty(L, M, N, dtype=torch.bfloat16, device="cuda")
    gw.run(Ad, Bd, Cd, D, alpha, beta)
    torch.cuda.synchronize()
    ref = oracle.gemm_rows(bits_of(A), bits_of(B), None if C is None else bits_of(C),
                           M, N, K, L, alpha, beta, rows=rows)
    d = bits_of(D).reshape(L * M, N)
    if rows is not None:
        d = d[rows]
    return d, ref


# ------------------------------------------------------------------ exact cases

def test_handworked_fixture(gw_each):
    """The hand-worked 2x3x4 example, zero-padded to K = N = 8 (16-byte rows)."""
    A, Bkn, C, Dexp, alpha, beta = load_handworked()
    M, K = A.shape
    N = Bkn.shape[1]
    Ap = np.zeros((M, 8)); Ap[:, :K] = A
    Bp = np.zeros((8, 8)); Bp[:N, :K] = Bkn.T          # stored N x K
    Cp = np.zeros((M, 8)); Cp[:, :N] = C
    t = lambda x: torch.from_numpy(f64_to_bf16_bits(x).astype(np.int16)).view(
        torch.bfloat16).reshape(1, *x.shape).cuda()
    D = torch.empty(1, M, 8, dtype=torch.bfloat16, device="cuda")
    gw_each.run(t(Ap), t(Bp), t(Cp), D, alpha, beta)
    torch.cuda.synchronize()
    got = bits_of(D).reshape(M, 8)
    np.testing.assert_array_equal(got[:, :N], f64_to_bf16_bits(Dexp))
    np.testing.assert_array_equal(got[:, N:], 0)


@pytest.mark.parametrize("M,N,K,L", [
    (128, 256, 64, 1),      # exactly one tile, one k-block
    (300, 520, 200, 2),     # ragged M, N, K; several tiles; batches
    (1, 8, 8, 1),           # smallest legal problem
    (2048, 2048, 128, 1),   # more tiles than SMs: persistent loop, ring wraps
])
def test_integer_inputs_bit_exact(gw_each, M, N, K, L):
    A, B, C = workloads.make_inputs(M, N, K, L, ("int", -4, 4), ("int", -4, 4), seed=M + K)
    D = torch.empty(L, M, N, dtype=torch.bfloat16, device="cuda")
    gw_each.run(to_dev(A), to_dev(B), to_dev(C), D, 2.0, -3.0)
    torch.cuda.synchronize()
    ref = oracle.gemm(bits_of(A), bits_of(B), bits_of(C), M, N, K, L, 2.0, -3.0)
    np.testing.assert_array_equal(bits_of(D).reshape(L, M, N), f64_to_bf16_bits(ref))


@pytest.mark.parametrize("M,N,K,L", [
    (300, 520, 200, 2),     # ragged M and N (N not a multiple of 64), batches
    (4000, 4104, 96, 2),    # half-width tail units, ragged N edge inside a 64-column block
    (130, 8, 64, 1),        # N narrower than one 64-column block
    (8192, 1024, 64, 1),    # skinny: many units per cluster, blocks in flight back to back
])
def test_wide_d_stores_bit_exact(gw_each, M, N, K, L):
    """beta == 0 and K <= 512: D leaves in 32 x 64 blocks (128-byte swizzle).
    Integer inputs make the result exact, so it must match bit for bit,
    including the columns and rows the TMA store clips at ragged edges."""
    A, B, _ = workloads.make_inputs(M, N, K, L, ("int", -4, 4), None, seed=N + K)
    D = torch.full((L, M, N), 5.0, dtype=torch.bfloat16, device="cuda")
    gw_each.run(to_dev(A), to_dev(B), None, D, 0.5, 0.0)
    torch.cuda.synchronize()
    ref = oracle.gemm(bits_of(A), bits_of(B), None, M, N, K, L, 0.5, 0.0)
    np.testing.assert_array_equal(bits_of(D).reshape(L, M, N), f64_to_bf16_bits(ref))


# ------------------------------------------------------------------ small shapes

@pytest.mark.parametrize("M,N,K,L,alpha,beta", [
    (256, 256, 256, 1, 1.0, 0.0),
    (200, 136, 72, 1, 1.0, 0.0),      # ragged edges, K not a multiple of 64
    (130, 264, 8, 3, 1.5, 0.5),       # K < 64, batches, C
    (64, 512, 56, 2, -1.25, 0.75),
    (513, 1032, 1000, 1, 1.0, 1.0),
    (4096, 4096, 128, 1, 1.0, 0.0),   # 512 tiles: several tiles per CTA
    (4000, 4104, 96, 2, 1.0, 0.5),    # tail tiles split into halves, ragged N edge in a half
])
def test_small_shapes_match_oracle(gw_each, M, N, K, L, alpha, beta):
    cd = ("normal", 1.0) if beta != 0 else None
    d, ref = run_case(gw_each, M, N, K, L, alpha, beta, cd=cd, seed=17)
    assert_gemm_close(d, ref, K, f"{M}x{N}x{K}x{L}")


def test_k_zero_gives_beta_c(gw_each):
    M, N, L = 200, 264, 2
    C = workloads.make_inputs(M, N, 0, L, ("uniform",), ("uniform",), 3)[2]
    D = torch.full((L, M, N), 7.0, dtype=torch.bfloat16, device="cuda")
    A = torch.empty(L, M, 0, dtype=torch.bfloat16, device="cuda")
    B = torch.empty(L, N, 0, dtype=torch.bfloat16, device="cuda")
    gw_each.run(A, B, C.cuda(), D, 1.0, 0.5)
    torch.cuda.synchronize()
    ref = oracle.gemm(np.zeros(0, np.uint16), np.zeros(0, np.uint16), bits_of(C),
                      M, N, 0, L, 1.0, 0.5)
    assert_gemm_close(bits_of(D), ref, 0, "K=0")


def test_beta_zero_ignores_nan_c(gw_each):
    M, N, K, L = 192, 256, 128, 1
    A, B, _ = workloads.make_inputs(M, N, K, L, ("uniform",), None, 5)
    C = torch.full((L, M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    D = torch.empty(L, M, N, dtype=torch.bfloat16, device="cuda")
    gw_each.run(A.cuda(), B.cuda(), C, D, 1.0, 0.0)
    torch.cuda.synchronize()
    ref = oracle.gemm(bits_of(A), bits_of(B), None, M, N, K, L, 1.0, 0.0)
    assert_gemm_close(bits_of(D), ref, K, "beta=0 with NaN C")


def test_in_place_d_is_c(gw_each):
    M, N, K, L = 320, 392, 96, 2
    A, B, C = workloads.make_inputs(M, N, K, L, ("uniform",), ("normal", 1.0), 9)
    D = C.clone().cuda()
    gw_each.run(A.cuda(), B.cuda(), D, D, 1.0, -1.0)
    torch.cuda.synchronize()
    ref = oracle.gemm(bits_of(A), bits_of(B), bits_of(C), M, N, K, L, 1.0, -1.0)
    assert_gemm_close(bits_of(D), ref, K, "D is C")


def test_empty_problem_is_a_no_op(gw):
    D = torch.full((1, 0, 8), 1.0, dtype=torch.bfloat16, device="cuda")
    A = torch.empty(1, 0, 8, dtype=torch.bfloat16, device="cuda")
    B = torch.empty(1, 8, 8, dtype=torch.bfloat16, device="cuda")
    gw.run(A, B, None, D, 1.0, 0.0)
    D2 = torch.full((2, 16, 8), 3.0, dtype=torch.bfloat16, device="cuda")
    B0 = torch.empty(2, 8, 8, dtype=torch.bfloat16, device="cuda")
    A0 = torch.empty(2, 16, 8, dtype=torch.bfloat16, device="cuda")
    # N == 0 problem: D has no elements; nothing launches
    rc = gemm_ws.gemm_ws_run(gw.handle, A0, B0, None, D2, 16, 0, 8, 2, 1.0, 0.0)
    assert rc == gemm_ws.OK
    torch.cuda.synchronize()
    assert torch.all(D2 == 3.0)


def test_repeated_runs_are_identical(gw_each):
    """Shakes out mbarrier phase bugs: many back-to-back launches, same bits."""
    M, N, K, L = 640, 1280, 320, 1
    A, B, _ = workloads.make_inputs(M, N, K, L, ("uniform",), None, 21)
    Ad, Bd = A.cuda(), B.cuda()
    first = torch.empty(L, M, N, dtype=torch.bfloat16, device="cuda")
    gw_each.run(Ad, Bd, None, first, 1.0, 0.0)
    D = torch.empty_like(first)
    for _ in range(30):
        gw_each.run(Ad, Bd, None, D, 1.0, 0.0)
    torch.cuda.synchronize()
    assert torch.equal(first.view(torch.int16), D.view(torch.int16))
    ref = oracle.gemm(bits_of(A), bits_of(B), None, M, N, K, L, 1.0, 0.0)
    assert_gemm_close(bits_of(D), ref, K, "repeat")


# ------------------------------------------------------------------ argument checks

def test_argument_errors_launch_nothing(gw):
    h = gw.handle
    A = torch.zeros(1, 64, 64, dtype=torch.bfloat16, device="cuda")
    B = torch.zeros(1, 64, 64, dtype=torch.bfloat16, device="cuda")
    D = torch.full((1, 64, 64), 5.0, dtype=torch.bfloat16, device="cuda")
    run = gemm_ws.gemm_ws_run
    assert run(h, A, B, None, D, 64, 64, 64, 1, 1.0, 1.0) == gemm_ws.ERR_INVALID_ARG  # C NULL
    assert run(h, A, B, None, D, -1, 64, 64, 1, 1.0, 0.0) == gemm_ws.ERR_INVALID_ARG
    assert run(h, A, B, None, None, 64, 64, 64, 1, 1.0, 0.0) == gemm_ws.ERR_INVALID_ARG
    assert run(h, A, B, None, A, 64, 64, 64, 1, 1.0, 0.0) == gemm_ws.ERR_INVALID_ARG  # D is A
    assert run(h, A, B, None, D, 64, 64, 60, 1, 1.0, 0.0) == gemm_ws.ERR_ALIGNMENT   # K % 8
    assert run(h, A, B, None, D, 64, 60, 64, 1, 1.0, 0.0) == gemm_ws.ERR_ALIGNMENT   # N % 8
    Dv = D.view(-1)[1:].view(-1)                                                    # 2-byte offset
    assert gemm_ws.load_library().gemm_ws_run(
        h, A.data_ptr(), B.data_ptr(), None, Dv.data_ptr(), 8, 8, 64, 1, 1.0, 0.0,
        torch.cuda.current_stream().cuda_stream) == gemm_ws.ERR_ALIGNMENT
    torch.cuda.synchronize()
    assert torch.all(D == 5.0)


# ------------------------------------------------------------------ full-size workloads

@pytest.mark.parametrize("name", [
    "gemm_256x256x256",
    "gemm_4096x4096x4096",
    "gemm_8192x8192x8192_alpha_beta",
    "gemm_batched4_5000x3000x4000_ragged",
])
def test_workload_parity(gw, name):
    """Each workload at full size, in the launch configuration the benchmark
    times (a default handle), every element against the oracle."""
    w = workloads.WORKLOADS[name]
    A, B, C = workloads.workload_inputs(w)
    D = torch.empty(w.L, w.M, w.N, dtype=torch.bfloat16, device="cuda")
    gw.run(to_dev(A), to_dev(B), to_dev(C), D, w.alpha, w.beta)
    torch.cuda.synchronize()
    check_every_row(bits_of(D), A, B, C, w.M, w.N, w.K, w.L, w.alpha, w.beta, name)


# ------------------------------------------------------------------ randomized and guarded

def _random_cases(n, seed):
    rng = np.random.default_rng(seed)
    for _ in range(n):
        M = int(rng.integers(1, 700))
        N = 8 * int(rng.integers(1, 90))
        K = 8 * int(rng.integers(0, 80))
        L = int(rng.integers(1, 4))
        alpha = float(np.float32(rng.choice([1.0, -0.5, 2.0, 0.75])))
        beta = float(np.float32(rng.choice([0.0, 0.0, 1.0, -1.5])))
        yield M, N, K, L, alpha, beta


@pytest.mark.parametrize("case", list(_random_cases(16, seed=2024)),
                         ids=lambda c: "x".join(str(v) for v in c[:4]))
def test_random_shapes_match_oracle(gw_each, case):
    """Seeded random problems: ragged M, N, K (including K = 0), batches,
    alpha/beta signs; every element checked against the oracle."""
    M, N, K, L, alpha, beta = case
    cd = ("uniform",) if beta != 0 else None
    d, ref = run_case(gw_each, M, N, K, L, alpha, beta, ab=("normal", 0.5), cd=cd,
                      seed=M * 7 + N + K)
    assert_gemm_close(d, ref, K, f"{M}x{N}x{K}x{L}")


def _random_auto_cases(n, seed):
    """Shapes that reach every path the default handle picks per problem:
    short K (single-CTA tiles), long K on few tiles (split pieces), and the
    rest (CTA pairs, with half-width tail tiles)."""
    rng = np.random.default_rng(seed)
    for i in range(n):
        kind = i % 3
        if kind == 0:     # short K
            M, N, K = int(rng.integers(1, 3000)), 8 * int(rng.integers(1, 400)), 8 * int(rng.integers(1, 64))
        elif kind == 1:   # few tiles, long K
            M, N, K = int(rng.integers(1, 900)), 8 * int(rng.integers(1, 110)), 8 * int(rng.integers(512, 2500))
        else:             # many tiles
            M, N, K = int(rng.integers(1500, 5000)), 8 * int(rng.integers(190, 600)), 8 * int(rng.integers(130, 400))
        L = int(rng.integers(1, 3))
        alpha = float(np.float32(rng.choice([1.0, -0.5, 2.0])))
        beta = float(np.float32(rng.choice([0.0, 1.0, -1.5])))
        yield M, N, K, L, alpha, beta


@pytest.mark.parametrize("case", list(_random_auto_cases(12, seed=77)),
                         ids=lambda c: "x".join(str(v) for v in c[:4]))
def test_random_shapes_default_handle(gw, case):
    """Seeded random problems on a default handle (tile configuration and
    split chosen per problem); sampled rows (every tile edge plus random
    rows) against the oracle."""
    M, N, K, L, alpha, beta = case
    cd = ("uniform",) if beta != 0 else None
    rows = sample_rows(M, L, 16, seed=K + N)
    d, ref = run_case(gw, M, N, K, L, alpha, beta, ab=("normal", 0.5), cd=cd,
                      seed=M * 5 + N + K, rows=rows)
    assert_gemm_close(d, ref, K, f"{M}x{N}x{K}x{L}")


def test_d_neighbours_are_never_written(gw_each):
    """D lives inside a larger buffer; the elements before and after it (and
    hence outside the ragged M x N edges of the TMA stores) keep their canary
    values."""
    M, N, K, L = 333, 264, 72, 2
    A, B, C = workloads.make_inputs(M, N, K, L, ("uniform",), ("uniform",), seed=90)
    pad = 4096
    buf = torch.full((pad + L * M * N + pad,), 123.0, dtype=torch.bfloat16, device="cuda")
    D = buf[pad:pad + L * M * N].view(L, M, N)
    gw_each.run(A.cuda(), B.cuda(), C.cuda(), D, 1.0, 1.0)
    torch.cuda.synchronize()
    assert torch.all(buf[:pad] == 123.0) and torch.all(buf[pad + L * M * N:] == 123.0)
    ref = oracle.gemm(bits_of(A), bits_of(B), bits_of(C), M, N, K, L, 1.0, 1.0)
    assert_gemm_close(bits_of(D), ref, K, "guarded D")


def test_create_rejects_a_missing_device():
    with pytest.raises(gemm_ws.GemmWSError) as e:
        gemm_ws.GemmWS(torch.cuda.device_count())
    assert e.value.status == gemm_ws.ERR_INVALID_ARG


def test_oversized_dimensions_are_rejected(gw):
    A = torch.zeros(1, 8, 8, dtype=torch.bfloat16, device="cuda")
    rc = gemm_ws.gemm_ws_run(gw.handle, A, A, None, A.clone(), 1 << 31, 8, 8, 1, 1.0, 0.0)
    assert rc == gemm_ws.ERR_INVALID_ARG
    # L*M*N = 2^42 elements, beyond the 2^40 limit: rejected by the size check,
    # before any pointer is used (the buffers here are far smaller)
    rc = gemm_ws.gemm_ws_run(gw.handle, A, A, None, A.clone(), 1 << 21, 1 << 21, 8, 1, 1.0, 0.0)
    assert rc == gemm_ws.ERR_INVALID_ARG
