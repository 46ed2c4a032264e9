"""Split-K parity: problems with few output tiles and a long K.

When the output has at most half as many tiles as the GPU has persistent
clusters, the library cuts each tile's K range into pieces that run on
separate clusters. Every piece parks its fp32 partial in the handle's
workspace, chunk by chunk (32 x 32), and counts each chunk in; the piece
whose write completes a chunk's count adds that chunk's partials (in piece
order, so the bits do not depend on which piece it was) and runs the
alpha/beta epilogue for it. These tests check that the launch plan really
splits, compare with the oracle, and check that back-to-back launches and
graph replays (whose chunk counters the kernel returns to zero) stay correct.
"""
from __future__ import annotations

import os

import numpy as np
import pytest
import torch

import oracle
from async_pipelines_gb300 import gemm_ws, workloads
from tests.debug_helpers import debug_handle, launch_shape
from tests.gpu_helpers import bits_of, sample_rows, to_dev
from tests.numerics import assert_gemm_close, f64_to_bf16_bits

pytestmark = pytest.mark.gpu

CONFIGS = [(2, 0), (1, 0), (2, 1)]
IDS = ["cta_pair", "cta_single", "cta_pair_multicast"]


def _handle(cg, mc):
    keys = ("GEMM_WS_CTA_GROUP", "GEMM_WS_MULTICAST")
    old = {k: os.environ.get(k) for k in keys}
    os.environ["GEMM_WS_CTA_GROUP"] = str(cg)
    os.environ["GEMM_WS_MULTICAST"] = str(mc)
    try:
        return gemm_ws.GemmWS(0)
    finally:
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


@pytest.fixture(scope="module", params=CONFIGS, ids=IDS)
def cfg(request):
    cg, mc = request.param
    g = _handle(cg, mc)
    plan = debug_handle(cta_group=cg, multicast=mc)
    yield g, plan
    assert g.query_status() == gemm_ws.OK
    g.close()
    plan.close()


def ksplit_of(plan, M, N, K, L, streamout=False):
    return launch_shape(plan, M, N, K, L, streamout=streamout)[3]


# Shapes with few tiles and long K. Full oracle where it finishes in seconds;
# sampled rows (every tile's edges plus random rows) otherwise.
CASES = [
    # M, N, K, L, alpha, beta, full
    (256, 256, 8192, 1, 1.0, 0.0, True),         # one tile, many pieces
    (200, 296, 4096, 3, 1.5, 0.5, True),         # ragged M, N; batches; C
    (1000, 776, 20000, 1, -0.75, 1.25, False),   # ragged everything, K not a stage multiple
    (1024, 1024, 32768, 1, 1.0, -0.5, False),    # the long-K square shape
    (128, 8, 2048, 1, 2.0, 0.0, True),           # smallest split: 2 pieces
]


@pytest.mark.parametrize("M,N,K,L,alpha,beta,full", CASES,
                         ids=[f"{c[0]}x{c[1]}x{c[2]}x{c[3]}" for c in CASES])
def test_split_k_matches_oracle(cfg, M, N, K, L, alpha, beta, full):
    g, plan = cfg
    assert ksplit_of(plan, M, N, K, L) > 1
    cd = ("normal", 1.0) if beta != 0 else None
    A, B, C = workloads.make_inputs(M, N, K, L, ("uniform",), cd, seed=M + N + K)
    D = torch.empty(L, M, N, dtype=torch.bfloat16, device="cuda")
    g.run(to_dev(A), to_dev(B), to_dev(C), D, alpha, beta)
    torch.cuda.synchronize()
    rows = None if full else sample_rows(M, L, 24, seed=K)
    ref = oracle.gemm_rows(bits_of(A), bits_of(B), None if C is None else bits_of(C),
                           M, N, K, L, alpha, beta, rows=rows)
    d = bits_of(D).reshape(L * M, N)
    if rows is not None:
        d = d[rows]
    assert_gemm_close(d, ref, K, f"split-K {M}x{N}x{K}x{L}")


def test_split_k_integer_inputs_bit_exact(cfg):
    """Integer inputs keep every partial and their sum exact in fp32, so the
    summation of the pieces must give the oracle's bf16 bits exactly."""
    g, plan = cfg
    M, N, K, L = 384, 520, 12288, 1
    assert ksplit_of(plan, M, N, K, L) > 1
    A, B, C = workloads.make_inputs(M, N, K, L, ("int", -3, 3), ("int", -4, 4), seed=77)
    D = torch.empty(L, M, N, dtype=torch.bfloat16, device="cuda")
    g.run(to_dev(A), to_dev(B), to_dev(C), D, 1.0, 2.0)
    torch.cuda.synchronize()
    rows = sample_rows(M, L, 32, seed=5)
    ref = oracle.gemm_rows(bits_of(A), bits_of(B), bits_of(C), M, N, K, L, 1.0, 2.0, rows=rows)
    np.testing.assert_array_equal(bits_of(D).reshape(L * M, N)[rows], f64_to_bf16_bits(ref))


def test_split_k_counters_reset_between_launches(cfg):
    """Different data back to back: a counter left non-zero by one launch
    would make the next launch's wrong piece (or none) finish the tile."""
    g, plan = cfg
    M, N, K, L = 256, 512, 6144, 1
    assert ksplit_of(plan, M, N, K, L) > 1
    D = torch.empty(L, M, N, dtype=torch.bfloat16, device="cuda")
    for seed in (101, 102, 103):
        A, B, _ = workloads.make_inputs(M, N, K, L, ("uniform",), None, seed=seed)
        D.fill_(float("nan"))
        g.run(A.cuda(), B.cuda(), None, D, 1.0, 0.0)
        torch.cuda.synchronize()
        ref = oracle.gemm(bits_of(A), bits_of(B), None, M, N, K, L, 1.0, 0.0)
        assert_gemm_close(bits_of(D), ref, K, f"launch with seed {seed}")


def test_split_k_is_deterministic(cfg):
    """The pieces are summed in a fixed order: the same bits every launch,
    whichever piece happened to finish last."""
    g, plan = cfg
    M, N, K, L = 512, 512, 16384, 1
    assert ksplit_of(plan, M, N, K, L) > 1
    A, B, C = workloads.make_inputs(M, N, K, L, ("normal", 1.0), ("normal", 1.0), seed=88)
    Ad, Bd, Cd = A.cuda(), B.cuda(), C.cuda()
    first = torch.empty(L, M, N, dtype=torch.bfloat16, device="cuda")
    g.run(Ad, Bd, Cd, first, 0.5, 0.25)
    D = torch.empty_like(first)
    for _ in range(20):
        g.run(Ad, Bd, Cd, D, 0.5, 0.25)
        torch.cuda.synchronize()
        assert torch.equal(first.view(torch.int16), D.view(torch.int16))


def test_split_k_replays_from_a_graph(cfg):
    g, plan = cfg
    M, N, K, L = 320, 264, 8192, 2
    assert ksplit_of(plan, M, N, K, L) > 1
    A, B, C = workloads.make_inputs(M, N, K, L, ("uniform",), ("uniform",), seed=64)
    Ad, Bd, Cd = A.cuda(), B.cuda(), C.cuda()
    eager = torch.empty(L, M, N, dtype=torch.bfloat16, device="cuda")
    g.run(Ad, Bd, Cd, eager, 1.0, 1.0)
    D = torch.zeros_like(eager)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        for _ in range(2):
            g.run(Ad, Bd, Cd, D, 1.0, 1.0, stream=s)
    for _ in range(3):
        D.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(D.view(torch.int16), eager.view(torch.int16))
    ref = oracle.gemm(bits_of(A), bits_of(B), bits_of(C), M, N, K, L, 1.0, 1.0)
    assert_gemm_close(bits_of(D), ref, K, "graph replay")


def test_split_k_beta_zero_ignores_nan_c(cfg):
    g, plan = cfg
    M, N, K, L = 256, 256, 4096, 1
    assert ksplit_of(plan, M, N, K, L) > 1
    A, B, _ = workloads.make_inputs(M, N, K, L, ("uniform",), None, 7)
    C = torch.full((L, M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    D = torch.empty(L, M, N, dtype=torch.bfloat16, device="cuda")
    g.run(A.cuda(), B.cuda(), C, D, 1.0, 0.0)
    torch.cuda.synchronize()
    ref = oracle.gemm(bits_of(A), bits_of(B), None, M, N, K, L, 1.0, 0.0)
    assert_gemm_close(bits_of(D), ref, K, "split-K, beta=0, NaN C")


def test_plan_keeps_whole_tiles_where_it_should(cfg):
    """No split for stream-out (its consumer takes each tile where it is
    computed), for short K, or once the tiles alone fill half the GPU."""
    _, plan = cfg
    assert ksplit_of(plan, 1024, 1024, 32768, 1, streamout=True) == 1
    assert ksplit_of(plan, 1024, 1024, 1024, 1) == 1
    assert ksplit_of(plan, 8192, 8192, 8192, 1) == 1
    assert ksplit_of(plan, 256, 256, 0, 1) == 1
    cs, clusters, units, ks = launch_shape(plan, 256, 256, 65536, 1, streamout=False)
    assert 2 <= ks <= 32 and units % ks == 0 and units == clusters
