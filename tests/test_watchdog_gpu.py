"""The watchdog, tested without faulting the GPU.

The debug build's fault switch makes the stream-out consumer warp take no
tile, so the epilogue's wait for a free shared-memory slot is a wait on a
barrier that nothing will ever complete. The run must end on its own within
its bounded waits, report GEMM_WS_ERR_TIMEOUT through the status query, and
leave the device usable: the next normal run on the same handle is correct.
"""
from __future__ import annotations

import time

import pytest
import torch

import oracle
from async_pipelines_gb300 import gemm_ws, workloads
from tests.debug_helpers import configure, debug_handle
from tests.gpu_helpers import bits_of, sample_rows
from tests.numerics import assert_gemm_close
from tests.test_streamout_gpu import check_staging

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("cta_group", [2, 1])
def test_consumer_that_takes_no_tile_times_out_then_recovers(cta_group):
    g = debug_handle(cta_group=cta_group, timeout_ms=200)
    # Several units per cluster, the first a whole 256-column tile: every
    # epilogue warp needs more shared-memory slots than its ring holds, so it
    # must wait for the consumer to release one.
    M, N, K, L = 4096, 4096, 64, 1
    A, B, _ = workloads.make_inputs(M, N, K, L, ("uniform",), None, seed=41)
    Ad, Bd = A.cuda(), B.cuda()
    T = gemm_ws.gemm_ws_streamout_tiles(M, N, L)
    staging = torch.empty(T * 128 * 128, dtype=torch.bfloat16, device="cuda")
    flags = torch.empty(2 * T, dtype=torch.int32, device="cuda")
    D = torch.empty(L, M, N, dtype=torch.bfloat16, device="cuda")

    configure(g, fault=1)
    t0 = time.perf_counter()
    g.run_streamout(Ad, Bd, None, D, staging, flags, 1.0, 0.0)
    status = g.query_status()
    elapsed = time.perf_counter() - t0
    assert status == gemm_ws.ERR_TIMEOUT, gemm_ws.status_string(status)
    assert elapsed < 20.0
    assert g.query_status() == gemm_ws.OK          # reading cleared the word
    assert int(flags[1::2].sum().item()) == 0      # no tile was flagged ready

    configure(g, fault=0)
    g.run_streamout(Ad, Bd, None, D, staging, flags, 1.0, 0.0)
    assert g.query_status() == gemm_ws.OK
    ref = oracle.gemm(bits_of(A), bits_of(B), None, M, N, K, L, 1.0, 0.0)
    assert_gemm_close(bits_of(D), ref, K, "after recovery")
    check_staging(D, staging, flags)
    g.close()


@pytest.mark.parametrize("cta_group", [2, 1])
def test_split_piece_that_never_flags_times_out_then_recovers(cta_group):
    """The in-kernel fix-up's one cross-CTA wait, under the watchdog: with the
    debug build's fault 2 the piece that arrives first writes its partial
    but never sets its written flag, so the other piece's bounded wait must
    end the launch with GEMM_WS_ERR_TIMEOUT. The status query clears the
    fix-up words that the aborted launch left part-way, and the next two
    runs on the same handle are correct and bit-identical."""
    from tests.debug_helpers import split_plan
    g = debug_handle(cta_group=cta_group, timeout_ms=200)
    # 36 pair tiles (72 single-CTA tiles) with K = 8192: every tile in two
    # pieces, fixed up inside the GEMM.
    M, N, K, L = (1536, 1536, 8192, 1) if cta_group == 2 else (1024, 2304, 8192, 1)
    assert split_plan(g, M, N, K, L) == (2, 1)
    A, B, C = workloads.make_inputs(M, N, K, L, ("uniform",), ("normal", 1.0), seed=43)
    Ad, Bd, Cd = A.cuda(), B.cuda(), C.cuda()
    D = torch.empty(L, M, N, dtype=torch.bfloat16, device="cuda")

    configure(g, fault=2)
    t0 = time.perf_counter()
    g.run(Ad, Bd, Cd, D, 1.5, -0.5)
    status = g.query_status()
    assert status == gemm_ws.ERR_TIMEOUT, gemm_ws.status_string(status)
    assert time.perf_counter() - t0 < 20.0
    assert g.query_status() == gemm_ws.OK

    configure(g, fault=0)
    outs = []
    for _ in range(2):
        D.fill_(float("nan"))
        g.run(Ad, Bd, Cd, D, 1.5, -0.5)
        assert g.query_status() == gemm_ws.OK
        outs.append(D.clone())
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    rows = sample_rows(M, L, 24, seed=5)
    ref = oracle.gemm_rows(bits_of(A), bits_of(B), bits_of(C), M, N, K, L, 1.5, -0.5, rows=rows)
    assert_gemm_close(bits_of(outs[0]).reshape(L * M, N)[rows], ref, K, "after recovery")
    g.close()
