"""CUDA-graph capture of the C-ABI calls.

A call launches exactly one kernel and allocates nothing, so it can be
captured into a CUDA graph and replayed (launch overhead then disappears for
small problems). Replays must give the same bits as eager calls; for the
stream-out call, every replay must deliver every tile exactly once again
(the kernel clears the flags it publishes and returns its sequence counter
to zero at the end, so nothing on the host has to run between replays).
"""
from __future__ import annotations

import pytest
import torch

from async_pipelines_gb300 import gemm_ws, workloads
from tests.test_streamout_gpu import check_staging

pytestmark = pytest.mark.gpu


def test_run_replays_from_a_graph():
    M, N, K, L = 640, 1024, 384, 2
    A, B, C = workloads.make_inputs(M, N, K, L, ("uniform",), ("normal", 1.0), seed=61)
    Ad, Bd, Cd = A.cuda(), B.cuda(), C.cuda()
    g = gemm_ws.GemmWS(0)
    eager = torch.empty(L, M, N, dtype=torch.bfloat16, device="cuda")
    g.run(Ad, Bd, Cd, eager, 1.25, -0.5)
    D = torch.zeros_like(eager)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        for _ in range(3):
            g.run(Ad, Bd, Cd, D, 1.25, -0.5, stream=s)
    for _ in range(4):
        D.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(D.view(torch.int16), eager.view(torch.int16))
    assert g.query_status() == gemm_ws.OK
    g.close()


def test_streamout_replays_from_a_graph():
    M, N, K, L = 768, 1280, 256, 1
    A, B, _ = workloads.make_inputs(M, N, K, L, ("uniform",), None, seed=62)
    Ad, Bd = A.cuda(), B.cuda()
    g = gemm_ws.GemmWS(0)
    T = gemm_ws.gemm_ws_streamout_tiles(M, N, L)
    staging = torch.empty(T * 128 * 128, dtype=torch.bfloat16, device="cuda")
    flags = torch.empty(2 * T, dtype=torch.int32, device="cuda")
    D = torch.empty(L, M, N, dtype=torch.bfloat16, device="cuda")
    g.run_streamout(Ad, Bd, None, D, staging, flags, 1.0, 0.0)   # eager, first
    torch.cuda.synchronize()
    eager = D.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        g.run_streamout(Ad, Bd, None, D, staging, flags, 1.0, 0.0, stream=s)
    for _ in range(4):
        staging.fill_(-7.0)
        flags.fill_(-1)
        D.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(D.view(torch.int16), eager.view(torch.int16))
        check_staging(D, staging, flags)
    assert g.query_status() == gemm_ws.OK
    g.close()
