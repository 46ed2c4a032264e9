"""Stream-K parity: tiles whose K range is cut into pieces on several clusters.

The library cuts the K range of the last tiles (all tiles, when there are at
most half as many as clusters; else the tiles of a last, at most half-full
wave) into equal pieces, each run by its own cluster as its last unit. With
two pieces, the piece whose epilogue warp arrives second adds the other's
fp32 partial (written to the handle's workspace and flagged) and runs the
alpha/beta epilogue itself; with more, every piece writes its partial and a
reduction kernel that the call launches after the GEMM adds them. Either way
the pieces are added in piece order (the same bits on every run, and the
same bits from both fix-ups), and no piece waits for one that has not
started. These tests check that the launch plan really splits, compare with
the oracle, and check that back-to-back launches, graph replays, work on
another stream and the public kernel count stay correct.
GEMM_WS_STREAM_K=2 splits shapes the cost model would run whole, down to
one-stage pieces, so that many pieces, ragged K and a whole-tile part before
the split tiles are covered at sizes the oracle checks quickly.
"""
from __future__ import annotations

import os

import numpy as np
import pytest
import torch

import oracle
from async_pipelines_gb300 import gemm_ws, workloads
from tests.debug_helpers import debug_handle, launch_shape, split_plan
from tests.gpu_helpers import bits_of, sample_rows, to_dev
from tests.numerics import assert_gemm_close, f64_to_bf16_bits

pytestmark = pytest.mark.gpu

CONFIGS = [2, 1]
IDS = ["cta_pair", "cta_single"]


def _handle(cg, stream_k, lib=None, inline=1):
    keys = ("GEMM_WS_CTA_GROUP", "GEMM_WS_STREAM_K", "GEMM_WS_SK_INLINE")
    old = {k: os.environ.get(k) for k in keys}
    os.environ["GEMM_WS_CTA_GROUP"] = str(cg)
    os.environ["GEMM_WS_STREAM_K"] = str(stream_k)
    os.environ["GEMM_WS_SK_INLINE"] = str(inline)
    try:
        return gemm_ws.GemmWS(0, lib=lib)
    finally:
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


@pytest.fixture(scope="module", params=CONFIGS, ids=IDS)
def cfg(request):
    """(auto handle, forced handle, debug handles for their plans)."""
    cg = request.param
    auto, forced = _handle(cg, 1), _handle(cg, 2)
    lib = gemm_ws.load_debug_library()
    plan_auto = _handle(cg, 1, lib)
    plan_forced = _handle(cg, 2, lib)
    yield auto, forced, plan_auto, plan_forced
    for g in (auto, forced):
        assert g.query_status() == gemm_ws.OK
    for g in (auto, forced, plan_auto, plan_forced):
        g.close()


def sk_tiles(plan, M, N, K, L, streamout=False):
    return launch_shape(plan, M, N, K, L, streamout=streamout)[3]


def run_and_check(g, M, N, K, L, alpha, beta, seed, full, what, ab=("uniform",)):
    cd = ("normal", 1.0) if beta != 0 else None
    A, B, C = workloads.make_inputs(M, N, K, L, ab, cd, seed=seed)
    D = torch.empty(L, M, N, dtype=torch.bfloat16, device="cuda")
    g.run(to_dev(A), to_dev(B), to_dev(C), D, alpha, beta)
    torch.cuda.synchronize()
    rows = None if full else sample_rows(M, L, 24, seed=K + seed)
    ref = oracle.gemm_rows(bits_of(A), bits_of(B), None if C is None else bits_of(C),
                           M, N, K, L, alpha, beta, rows=rows)
    d = bits_of(D).reshape(L * M, N)
    if rows is not None:
        d = d[rows]
    assert_gemm_close(d, ref, K, what)


# Few tiles and long K: the cost model itself picks stream-K (every tile).
AUTO_CASES = [
    # M, N, K, L, alpha, beta, full
    (256, 256, 8192, 1, 1.0, 0.0, True),         # one tile, many pieces
    (200, 296, 16384, 3, 1.5, 0.5, False),       # ragged M, N; batches; C
    (1000, 776, 20000, 1, -0.75, 1.25, False),   # ragged everything, K not a stage multiple
    (1024, 1024, 32768, 1, 1.0, -0.5, False),    # the long-K square shape
    (128, 8, 16384, 1, 2.0, 0.0, True),          # smallest tile, long K
]


@pytest.mark.parametrize("M,N,K,L,alpha,beta,full", AUTO_CASES,
                         ids=[f"{c[0]}x{c[1]}x{c[2]}x{c[3]}" for c in AUTO_CASES])
def test_few_tiles_long_k_matches_oracle(cfg, M, N, K, L, alpha, beta, full):
    auto, _, plan, _ = cfg
    assert sk_tiles(plan, M, N, K, L) > 0
    run_and_check(auto, M, N, K, L, alpha, beta, M + N + K, full, f"stream-K {M}x{N}x{K}x{L}")


# Forced: whole-tile waves then a split last wave (more tiles than clusters),
# pieces of a few stages, ragged K, batches.
FORCED_CASES = [
    (4096, 2560, 512, 1, 1.0, 0.0, False),       # whole-tile waves, then the stream-K region
    (1536, 1280, 1024, 1, 1.25, -0.5, False),    # one partial wave: 2-3 pieces per tile
    (1000, 776, 3000, 2, 1.0, 1.0, False),       # ragged M, N, K (last k-block 56 deep), batches
    (9000, 1032, 320, 1, -1.0, 0.5, False),      # short pieces, ragged N
    (384, 512, 256, 2, 1.0, 0.0, True),          # two-stage tiles
]


@pytest.mark.parametrize("M,N,K,L,alpha,beta,full", FORCED_CASES,
                         ids=[f"{c[0]}x{c[1]}x{c[2]}x{c[3]}" for c in FORCED_CASES])
def test_forced_stream_k_matches_oracle(cfg, M, N, K, L, alpha, beta, full):
    _, forced, _, plan = cfg
    assert sk_tiles(plan, M, N, K, L) > 0
    run_and_check(forced, M, N, K, L, alpha, beta, 7 * M + K, full,
                  f"forced stream-K {M}x{N}x{K}x{L}")


def test_stream_k_integer_inputs_bit_exact(cfg):
    """Integer inputs keep every partial and their sum exact in fp32, so the
    sum of the pieces must give the oracle's bf16 bits exactly."""
    auto, forced, plan_auto, plan_forced = cfg
    for g, plan, (M, N, K, L) in ((auto, plan_auto, (384, 520, 12288, 1)),
                                  (forced, plan_forced, (2048, 1024, 1536, 1))):
        assert sk_tiles(plan, M, N, K, L) > 0
        A, B, C = workloads.make_inputs(M, N, K, L, ("int", -3, 3), ("int", -4, 4), seed=77)
        D = torch.empty(L, M, N, dtype=torch.bfloat16, device="cuda")
        g.run(to_dev(A), to_dev(B), to_dev(C), D, 1.0, 2.0)
        torch.cuda.synchronize()
        rows = sample_rows(M, L, 32, seed=5)
        ref = oracle.gemm_rows(bits_of(A), bits_of(B), bits_of(C), M, N, K, L, 1.0, 2.0,
                               rows=rows)
        np.testing.assert_array_equal(bits_of(D).reshape(L * M, N)[rows], f64_to_bf16_bits(ref))


def test_stream_k_workspace_reused_between_launches(cfg):
    """Different data back to back through the same partial workspace: each
    launch's reduction must read that launch's partials, never a previous
    launch's."""
    auto, forced, plan_auto, plan_forced = cfg
    for g, plan, (M, N, K, L) in ((auto, plan_auto, (256, 512, 6144, 1)),
                                  (forced, plan_forced, (1280, 1536, 768, 1))):
        assert sk_tiles(plan, M, N, K, L) > 0
        D = torch.empty(L, M, N, dtype=torch.bfloat16, device="cuda")
        for seed in (101, 102, 103):
            A, B, _ = workloads.make_inputs(M, N, K, L, ("uniform",), None, seed=seed)
            D.fill_(float("nan"))
            g.run(A.cuda(), B.cuda(), None, D, 1.0, 0.0)
            torch.cuda.synchronize()
            rows = sample_rows(M, L, 16, seed=seed)
            ref = oracle.gemm_rows(bits_of(A), bits_of(B), None, M, N, K, L, 1.0, 0.0, rows=rows)
            assert_gemm_close(bits_of(D).reshape(L * M, N)[rows], ref, K, f"seed {seed}")


def test_stream_k_is_deterministic(cfg):
    """The pieces are summed in a fixed order: the same bits every launch,
    whichever piece happened to finish first."""
    auto, forced, plan_auto, plan_forced = cfg
    for g, plan, (M, N, K, L) in ((auto, plan_auto, (512, 512, 16384, 1)),
                                  (forced, plan_forced, (2048, 1024, 1024, 1))):
        assert sk_tiles(plan, M, N, K, L) > 0
        A, B, C = workloads.make_inputs(M, N, K, L, ("normal", 1.0), ("normal", 1.0), seed=88)
        Ad, Bd, Cd = A.cuda(), B.cuda(), C.cuda()
        first = torch.empty(L, M, N, dtype=torch.bfloat16, device="cuda")
        g.run(Ad, Bd, Cd, first, 0.5, 0.25)
        D = torch.empty_like(first)
        for _ in range(20):
            g.run(Ad, Bd, Cd, D, 0.5, 0.25)
            torch.cuda.synchronize()
            assert torch.equal(first.view(torch.int16), D.view(torch.int16))


def test_stream_k_replays_from_a_graph(cfg):
    auto, forced, plan_auto, plan_forced = cfg
    for g, plan, (M, N, K, L) in ((auto, plan_auto, (320, 264, 8192, 2)),
                                  (forced, plan_forced, (1024, 2048, 1024, 1))):
        assert sk_tiles(plan, M, N, K, L) > 0
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
        rows = sample_rows(M, L, 16, seed=3)
        ref = oracle.gemm_rows(bits_of(A), bits_of(B), bits_of(C), M, N, K, L, 1.0, 1.0,
                               rows=rows)
        assert_gemm_close(bits_of(D).reshape(L * M, N)[rows], ref, K, "graph replay")


def test_stream_k_beta_zero_ignores_nan_c_and_in_place(cfg):
    _, forced, _, plan = cfg
    M, N, K, L = 1536, 1024, 2048, 1
    assert sk_tiles(plan, M, N, K, L) > 0
    A, B, C = workloads.make_inputs(M, N, K, L, ("uniform",), ("normal", 1.0), 7)
    Cnan = torch.full((L, M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    D = torch.empty(L, M, N, dtype=torch.bfloat16, device="cuda")
    forced.run(A.cuda(), B.cuda(), Cnan, D, 1.0, 0.0)
    torch.cuda.synchronize()
    rows = sample_rows(M, L, 16, seed=9)
    ref = oracle.gemm_rows(bits_of(A), bits_of(B), None, M, N, K, L, 1.0, 0.0, rows=rows)
    assert_gemm_close(bits_of(D).reshape(L * M, N)[rows], ref, K, "beta=0, NaN C")
    DC = C.clone().cuda()   # D is C: each chunk's C is read before its D is written
    forced.run(A.cuda(), B.cuda(), DC, DC, 1.0, -1.0)
    torch.cuda.synchronize()
    ref = oracle.gemm_rows(bits_of(A), bits_of(B), bits_of(C), M, N, K, L, 1.0, -1.0, rows=rows)
    assert_gemm_close(bits_of(DC).reshape(L * M, N)[rows], ref, K, "in place")


def test_plan_keeps_whole_tiles_where_it_should(cfg):
    """No stream-K for stream-out (its consumer takes each tile where it is
    computed) or for short K."""
    auto, forced, plan_auto, plan_forced = cfg
    for plan in (plan_auto, plan_forced):
        assert sk_tiles(plan, 1024, 1024, 32768, 1, streamout=True) == 0
        assert sk_tiles(plan, 256, 256, 0, 1) == 0
    assert sk_tiles(plan_auto, 1024, 1024, 1024, 1) == 0


@pytest.mark.parametrize("M,N,K,L,inline", [(512, 512, 16384, 1, 0), (1536, 1536, 8192, 1, 1)],
                         ids=["reduction_kernel", "in_kernel"])
def test_split_gemm_beside_kernels_on_another_stream(cfg, M, N, K, L, inline):
    """No piece waits for one that has not started (a piece that adds
    another's partial waits only for a piece that already arrived), so a
    split GEMM is correct (and ends with status OK) while other work on
    another stream holds SMs: cuBLAS GEMMs keep a second stream busy for the
    whole call (bounded: a fixed number of library calls). Both fix-ups: the
    reduction kernel (16 pieces per tile) and the in-kernel one (2)."""
    auto, _, plan, _ = cfg
    assert sk_tiles(plan, M, N, K, L) > 0
    assert split_plan(plan, M, N, K, L)[1] == inline
    A, B, C = workloads.make_inputs(M, N, K, L, ("uniform",), ("normal", 1.0), seed=55)
    Ad, Bd, Cd = A.cuda(), B.cuda(), C.cuda()
    X = torch.randn(4096, 4096, device="cuda", dtype=torch.bfloat16)
    Y = torch.empty_like(X)
    side = torch.cuda.Stream()
    D = torch.empty(L, M, N, dtype=torch.bfloat16, device="cuda")
    results = []
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(200):
            torch.matmul(X, X, out=Y)
    for _ in range(10):
        D.fill_(float("nan"))
        auto.run(Ad, Bd, Cd, D, 1.0, 0.5)
        results.append(D.clone())
    torch.cuda.synchronize()
    assert auto.query_status() == gemm_ws.OK
    rows = sample_rows(M, L, 32, seed=4)
    ref = oracle.gemm_rows(bits_of(A), bits_of(B), bits_of(C), M, N, K, L, 1.0, 0.5, rows=rows)
    for n, R in enumerate(results):
        assert torch.equal(R.view(torch.int16), results[0].view(torch.int16)), n
    assert_gemm_close(bits_of(results[0]).reshape(L * M, N)[rows], ref, K, "beside other kernels")


def test_kernels_per_run_matches_the_plan(cfg):
    """The public launch count: 2 exactly where the plan splits tiles into
    more than two pieces (the GEMM and the reduction), 1 otherwise (two
    pieces are added inside the GEMM), 0 for empty problems."""
    auto, forced, plan_auto, plan_forced = cfg
    shapes = [(256, 256, 8192, 1), (1024, 1024, 1024, 1), (8192, 8192, 8192, 1),
              (4096, 4096, 4096, 1), (200, 296, 16384, 3), (4096, 2560, 512, 1),
              (1536, 1536, 8192, 1)]
    seen = set()
    for g, plan in ((auto, plan_auto), (forced, plan_forced)):
        for M, N, K, L in shapes:
            pieces, inline = split_plan(plan, M, N, K, L)
            split = sk_tiles(plan, M, N, K, L) > 0
            assert inline == (split and pieces == 2), (M, N, K, L)
            want = 2 if split and not inline else 1
            if split:
                seen.add(inline)
            assert g.kernels_per_run(M, N, K, L) == want, (M, N, K, L)
            assert g.kernels_per_run(M, N, K, L, streamout=True) == 1
        assert g.kernels_per_run(0, 64, 64, 1) == 0
    assert seen == {0, 1}   # both fix-ups occur among these shapes


def _in_kernel_cases(cg):
    # Forced plans whose split tiles have exactly two pieces: M x N tiles
    # between a third and a half of the cluster count (76 CTA pairs / 152
    # single CTAs); ragged edges and C included.
    if cg == 2:
        return [(1536, 1536, 4096, 1, 1.0, 0.0), (1400, 1480, 3000, 1, 1.5, -0.5)]
    return [(1024, 2048, 4096, 1, 1.0, 0.0), (1000, 1960, 3000, 1, 1.5, -0.5)]


def test_in_kernel_fixup_equals_reduction_kernel(cfg):
    """Two-piece tiles: the in-kernel fix-up and the reduction kernel add the
    same two partials in the same order, so D is bit-identical, and both
    match the oracle; the fix-up words return to zero (a second launch is
    again bit-identical)."""
    auto, forced, plan_auto, plan_forced = cfg
    cg = launch_shape(plan_forced, 1536, 1536, 4096, 1, streamout=False)[0]
    sep = _handle(cg, 2, inline=0)
    sep_plan = _handle(cg, 2, gemm_ws.load_debug_library(), inline=0)
    try:
        for (M, N, K, L, alpha, beta) in _in_kernel_cases(cg):
            assert sk_tiles(plan_forced, M, N, K, L) > 0
            assert split_plan(plan_forced, M, N, K, L) == (2, 1), (M, N, K, L)
            assert split_plan(sep_plan, M, N, K, L) == (2, 0), (M, N, K, L)
            assert forced.kernels_per_run(M, N, K, L) == 1
            assert sep.kernels_per_run(M, N, K, L) == 2
            cd = ("normal", 1.0) if beta != 0 else None
            A, B, C = workloads.make_inputs(M, N, K, L, ("uniform",), cd, seed=M + K)
            Ad, Bd, Cd = to_dev(A), to_dev(B), to_dev(C)
            outs = []
            for g in (forced, sep, forced):
                D = torch.full((L, M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
                g.run(Ad, Bd, Cd, D, alpha, beta)
                outs.append(D)
            torch.cuda.synchronize()
            for D in outs[1:]:
                assert torch.equal(D.view(torch.int16), outs[0].view(torch.int16)), (M, N, K, L)
            rows = sample_rows(M, L, 24, seed=K)
            ref = oracle.gemm_rows(bits_of(A), bits_of(B), None if C is None else bits_of(C),
                                   M, N, K, L, alpha, beta, rows=rows)
            assert_gemm_close(bits_of(outs[0]).reshape(L * M, N)[rows], ref, K,
                              f"in-kernel fix-up {M}x{N}x{K}")
        assert sep.query_status() == gemm_ws.OK
    finally:
        sep.close()
        sep_plan.close()
