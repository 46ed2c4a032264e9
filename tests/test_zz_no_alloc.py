"""The allocation-free stream-out entry point, against the handle-based one.

gemm_ws_run_streamout_noalloc serves callers that may not call cudaMalloc
(inside another allocator's hook, under a framework that owns all device
memory); it keeps its scratch in a fixed array inside the library. This file
is collected last so that a failure here comes after every other test ran; it
passes alone in a fresh process as well.
"""
from __future__ import annotations

import ctypes
import time

import numpy as np
import pytest
import torch

import oracle
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


def test_noalloc_timeout_shows_as_unflagged_tiles_then_recovers():
    """A caller of the allocation-free entry point has no handle to query, so
    a watchdog timeout must show in the flags: with the debug build's fault
    (the stream-out consumer takes no tile, so the epilogue waits for a slot
    that is never released) the call ends on its own, every ready word is 0,
    and the next two normal calls are correct."""
    lib = gemm_ws.load_debug_library()
    dev = torch.cuda.current_device()
    M, N, K, L = 4096, 4096, 64, 1
    A, B, _ = workloads.make_inputs(M, N, K, L, ("uniform",), None, seed=47)
    Ad, Bd = A.cuda(), B.cuda()
    T = gemm_ws.gemm_ws_streamout_tiles(M, N, L)
    D = torch.empty(L, M, N, dtype=torch.bfloat16, device="cuda")
    staging = torch.empty(T * 128 * 128, dtype=torch.bfloat16, device="cuda")
    flags = torch.full((2 * T,), 0x5A5A5A5A, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream

    def call():
        return lib.gemm_ws_run_streamout_noalloc(
            Ad.data_ptr(), Bd.data_ptr(), None, D.data_ptr(), M, N, K, L, 1.0, 0.0,
            staging.data_ptr(), flags.data_ptr(), ctypes.c_void_p(stream))

    assert lib.gemm_ws_debug_noalloc_configure(dev, 1, 200) == gemm_ws.OK
    try:
        t0 = time.perf_counter()
        assert call() == gemm_ws.OK
        torch.cuda.synchronize()
        assert time.perf_counter() - t0 < 20.0
        assert int(flags[1::2].ne(0).sum().item()) == 0    # no tile flagged ready
    finally:
        assert lib.gemm_ws_debug_noalloc_configure(dev, 0, 0) == gemm_ws.OK
    ref = oracle.gemm(bits_of(A), bits_of(B), None, M, N, K, L, 1.0, 0.0)
    for n in range(2):
        D.fill_(float("nan"))
        assert call() == gemm_ws.OK
        torch.cuda.synchronize()
        assert_gemm_close(bits_of(D), ref, K, f"no-alloc call {n} after the timeout")
        check_staging(D, staging, flags)
