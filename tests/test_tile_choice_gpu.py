"""Per-problem tile configuration and the debug phase stamps (GPU).

A handle created without GEMM_WS_CTA_GROUP picks single-CTA 128 x 256 tiles
for short K (K <= 512) and for small problems with K <= 1024 (at most two
waves of CTA-pair tiles), CTA pairs otherwise; both choices must give the
oracle's results. The phase stamps of the debug build must be ordered.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import pytest
import torch

import oracle
from async_pipelines_gb300 import gemm_ws, workloads
from tests.debug_helpers import launch_shape
from tests.gpu_helpers import bits_of, sample_rows
from tests.numerics import assert_gemm_close, f64_to_bf16_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def auto_debug():
    keys = ("GEMM_WS_CTA_GROUP", "GEMM_WS_STREAM_K")
    old = {k: os.environ.pop(k, None) for k in keys}
    try:
        g = gemm_ws.GemmWS(0, lib=gemm_ws.load_debug_library())
    finally:
        for k, v in old.items():
            if v is not None:
                os.environ[k] = v
    yield g
    assert g.query_status() == gemm_ws.OK
    g.close()


@pytest.mark.parametrize("M,N,K,L,cs", [
    (8192, 8192, 64, 1, 1),      # short K: single CTAs
    (256, 256, 256, 1, 1),
    (2048, 2048, 1024, 1, 1),    # small problem, K = 1024
    (8192, 8192, 1024, 1, 2),    # many pair tiles
    (4096, 4096, 4096, 1, 2),    # long K
    (8192, 8192, 8192, 1, 2),
])
def test_tile_configuration_choice(auto_debug, M, N, K, L, cs):
    assert launch_shape(auto_debug, M, N, K, L, streamout=False)[0] == cs


@pytest.mark.parametrize("M,N,K,L", [(1000, 2056, 192, 2), (2048, 1536, 1024, 1)])
def test_single_cta_choice_matches_oracle(auto_debug, M, N, K, L):
    assert launch_shape(auto_debug, M, N, K, L, streamout=False)[0] == 1
    A, B, C = workloads.make_inputs(M, N, K, L, ("uniform",), ("normal", 1.0), seed=M + K)
    D = torch.empty(L, M, N, dtype=torch.bfloat16, device="cuda")
    auto_debug.run(A.cuda(), B.cuda(), C.cuda(), D, 1.25, -0.5)
    torch.cuda.synchronize()
    rows = sample_rows(M, L, 24, seed=K)
    ref = oracle.gemm_rows(bits_of(A), bits_of(B), bits_of(C), M, N, K, L, 1.25, -0.5, rows=rows)
    assert_gemm_close(bits_of(D).reshape(L * M, N)[rows], ref, K, f"{M}x{N}x{K}x{L}")


def test_phase_stamps_are_ordered(auto_debug):
    """Per CTA: entry <= start of work <= exit, all within the launch."""
    M, N, K, L = 1024, 1024, 2048, 1
    cs, clusters, _, _ = launch_shape(auto_debug, M, N, K, L, streamout=False)
    ph = torch.zeros(clusters * cs * 8, dtype=torch.int64, device="cuda")
    lib = auto_debug.lib
    assert lib.gemm_ws_debug_phases(auto_debug.handle, ctypes.c_void_p(ph.data_ptr())) == 0
    A, B, _ = workloads.make_inputs(M, N, K, L, ("uniform",), None, seed=3)
    D = torch.empty(L, M, N, dtype=torch.bfloat16, device="cuda")
    auto_debug.run(A.cuda(), B.cuda(), None, D, 1.0, 0.0)
    torch.cuda.synchronize()
    assert lib.gemm_ws_debug_phases(auto_debug.handle, None) == 0
    p = ph.view(clusters * cs, 8).cpu().numpy().astype(np.int64)
    assert np.all(p[:, 0] > 0)
    assert np.all(p[:, 0] <= p[:, 1]) and np.all(p[:, 1] <= p[:, 2])
    assert p[:, 2].max() - p[:, 0].min() < 10_000_000   # well under 10 ms


@pytest.mark.parametrize("M,N,K,L", [
    (256, 256, 256, 1),    # two single-CTA tiles -> eight 64-column quarters
    (300, 200, 520, 2),    # ragged: the last quarter of each tile straddles N or lies past it
    (130, 72, 64, 1),      # N inside the first quarter; three quarters outside N
    (1000, 776, 1024, 1),  # 32 tiles, 128 quarter units (a 4x wider launch than halves)
])
def test_quarter_units_bit_exact(auto_debug, M, N, K, L):
    """Problems with at most a quarter as many tiles as clusters run every
    tile as four 64-column units; integer inputs make the result exact, so
    it must equal the oracle's bf16 bits, ragged edges included."""
    cs, clusters, units, sk = launch_shape(auto_debug, M, N, K, L, streamout=False)
    tiles = L * -(-M // (128 * cs)) * -(-N // 256)
    assert sk == 0 and units == 4 * tiles and clusters == 4 * tiles
    A, B, C = workloads.make_inputs(M, N, K, L, ("int", -3, 3), ("int", -4, 4), seed=M + N)
    for beta, Cd in ((0.0, None), (1.5, C.cuda())):
        D = torch.full((L, M, N), 9.0, dtype=torch.bfloat16, device="cuda")
        auto_debug.run(A.cuda(), B.cuda(), Cd, D, 2.0, beta)
        torch.cuda.synchronize()
        ref = oracle.gemm(bits_of(A), bits_of(B), None if beta == 0 else bits_of(C),
                          M, N, K, L, 2.0, beta)
        np.testing.assert_array_equal(bits_of(D).reshape(L, M, N), f64_to_bf16_bits(ref))
    # stream-out keeps 128-column units
    assert launch_shape(auto_debug, M, N, K, L, streamout=True)[2] < 4 * tiles
