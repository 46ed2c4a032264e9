"""The allocation-free stream-out entry point, against the handle-based one.

gemm_ws_run_streamout_noalloc serves callers that may not call cudaMalloc
(inside another allocator's hook, under a framework that owns all device
memory); it keeps its scratch in a fixed array inside the library. This file
is collected last so that a failure here comes after every other test ran; it
passes alone in a fresh process as well.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from async_pipelines_gb300 import gemm_ws, workloads
from tests.gpu_helpers import bits_of
from tests.numerics import assert_gemm_close, bf16_bits_to_f64
from tests.test_streamout_gpu import check_staging

pytestmark = pytest.mark.gpu


def test_noalloc_matches_handle_entry_point_twice_in_a_row():
    M, N, K, L, alpha, beta = 384, 1032, 200, 2, 1.5, 0.5
    A, B, C = workloads.make_inputs(M, N, K, L, ("uniform",), ("normal", 1.0), seed=77)
    Ad, Bd, Cd = A.cuda(), B.cuda(), C.cuda()
    T = gemm_ws.gemm_ws_streamout_tiles(M, N, L)

    g = gemm_ws.GemmWS(0)
    D_ref = torch.empty(L, M, N, dtype=torch.bfloat16, device="cuda")
    st_ref = torch.empty(T * 128 * 128, dtype=torch.bfloat16, device="cuda")
    fl_ref = torch.empty(2 * T, dtype=torch.int32, device="cuda")
    g.run_streamout(Ad, Bd, Cd, D_ref, st_ref, fl_ref, alpha, beta)
    assert g.query_status() == gemm_ws.OK
    g.close()
    ref = bf16_bits_to_f64(bits_of(D_ref))

    for call in range(2):
        D = torch.full((L, M, N), 9.0, dtype=torch.bfloat16, device="cuda")
        staging = torch.full((T * 128 * 128,), -3.0, dtype=torch.bfloat16, device="cuda")
        flags = torch.full((2 * T,), 0x7A7A7A7A, dtype=torch.int32, device="cuda")
        rc = gemm_ws.gemm_ws_run_streamout_noalloc(Ad, Bd, Cd, D, M, N, K, L, alpha, beta,
                                                   staging, flags)
        assert rc == gemm_ws.OK, gemm_ws.status_string(rc)
        torch.cuda.synchronize()
        assert_gemm_close(bits_of(D), ref, K, f"no-alloc call {call}")
        # same tile configuration and schedule as the handle: the same bits
        assert np.array_equal(bits_of(D), bits_of(D_ref)), f"no-alloc call {call}"
        check_staging(D, staging, flags)


def test_noalloc_rejects_bad_arguments_without_launching():
    D = torch.full((1, 64, 64), 4.0, dtype=torch.bfloat16, device="cuda")
    A = torch.zeros(1, 64, 64, dtype=torch.bfloat16, device="cuda")
    flags = torch.zeros(2, dtype=torch.int32, device="cuda")
    rc = gemm_ws.gemm_ws_run_streamout_noalloc(A, A, None, D, 64, 64, 64, 1, 1.0, 0.0,
                                               None, flags)
    assert rc == gemm_ws.ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.all(D == 4.0)
