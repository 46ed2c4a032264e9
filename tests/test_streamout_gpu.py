"""GPU tests of the epilogue -> consumer-warp tile stream-out.

The staging buffer is checked bit for bit against D itself (not the oracle):
slot s must hold, row-major 128 x 128, the output tile whose flag says s,
with zeros outside M and N; the sequence numbers must be a permutation of
0..T-1 and every ready word must be 1. D itself is checked against the oracle.
"""
from __future__ import annotations

import os
import numpy as np
import pytest
import torch

import oracle
from async_pipelines_gb300 import gemm_ws, workloads
from tests.gpu_helpers import bits_of, check_every_row
from tests.numerics import assert_gemm_close

pytestmark = pytest.mark.gpu
T_EDGE = 128


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


def check_staging(D: torch.Tensor, staging: torch.Tensor, flags: torch.Tensor):
    """Every tile delivered exactly once, bit-exact, zero-padded at the edges."""
    L, M, N = D.shape
    tm, tn = -(-M // T_EDGE), -(-N // T_EDGE)
    T = L * tm * tn
    f = flags[: 2 * T].cpu().numpy().astype(np.int64).reshape(T, 2)
    assert np.all(f[:, 1] == 1), "a tile was not flagged ready"
    seq = f[:, 0]
    assert np.array_equal(np.sort(seq), np.arange(T)), "sequence numbers are not 0..T-1"
    # Pad D to whole tiles, then cut it into T row-major 128 x 128 tiles.
    Dp = torch.zeros(L, tm * T_EDGE, tn * T_EDGE, dtype=torch.bfloat16, device=D.device)
    Dp[:, :M, :N] = D
    tiles = Dp.view(L, tm, T_EDGE, tn, T_EDGE).permute(0, 1, 3, 2, 4).reshape(T, T_EDGE, T_EDGE)
    st = staging[: T * T_EDGE * T_EDGE].view(T, T_EDGE, T_EDGE)
    expect = tiles[torch.from_numpy(np.argsort(seq)).to(D.device)]
    # bit-exact everywhere, except that -0.0 and +0.0 are both "0" in the padding
    same = st.view(torch.int16) == expect.view(torch.int16)
    zero_pad = (st == 0) & (expect == 0)
    assert bool(torch.all(same | zero_pad)), "staging differs from D"


@pytest.mark.parametrize("M,N,K,L,beta", [
    (128, 128, 64, 1, 0.0),     # one stream-out tile; half of one output tile
    (300, 392, 136, 2, 0.0),    # ragged M and N, batches
    (256, 2904, 64, 1, 0.5),    # N edge where a 256-wide tile holds one 128 stream-out tile
    (1024, 2048, 192, 1, 0.0),  # 128 output tiles, several per CTA
    (4096, 4096, 64, 1, 0.0),   # more tiles than one wave: the last ones run as halves
])
def test_streamout_small(gw_each, M, N, K, L, beta):
    cd = ("uniform",) if beta != 0 else None
    A, B, C = workloads.make_inputs(M, N, K, L, ("uniform",), cd, seed=M + N)
    Ad, Bd = A.cuda(), B.cuda()
    Cd = C.cuda() if C is not None else None
    T = gemm_ws.gemm_ws_streamout_tiles(M, N, L)
    # canaries after the staging and flag regions catch writes past T slots
    staging = torch.full((T * T_EDGE * T_EDGE + 4096,), -2.0, dtype=torch.bfloat16, device="cuda")
    flags = torch.full((2 * T + 64,), 0x5A5A5A5A, dtype=torch.int32, device="cuda")
    D = torch.empty(L, M, N, dtype=torch.bfloat16, device="cuda")
    gw_each.run_streamout(Ad, Bd, Cd, D, staging, flags, 1.0, beta)
    torch.cuda.synchronize()
    ref = oracle.gemm(bits_of(A), bits_of(B), None if C is None else bits_of(C),
                      M, N, K, L, 1.0, beta)
    assert_gemm_close(bits_of(D), ref, K, "streamout D")
    check_staging(D, staging, flags)
    assert torch.all(staging[T * T_EDGE * T_EDGE:] == -2.0), "wrote past the staging slots"
    assert torch.all(flags[2 * T:] == 0x5A5A5A5A), "wrote past the flags"


def test_streamout_matches_plain_run(gw_each):
    """Stream-out leaves D identical to a plain run, bit for bit (when the
    plain run's plan keeps whole K ranges, as by default at this shape: a
    plan that splits K sums in another fp32 order)."""
    M, N, K, L = 512, 1024, 256, 1
    if gw_each.kernels_per_run(M, N, K, L) != 1:
        pytest.skip("the plain plan splits K here (GEMM_WS_STREAM_K forces it)")
    A, B, _ = workloads.make_inputs(M, N, K, L, ("uniform",), None, 33)
    Ad, Bd = A.cuda(), B.cuda()
    D0 = torch.empty(L, M, N, dtype=torch.bfloat16, device="cuda")
    D1 = torch.empty_like(D0)
    T = gemm_ws.gemm_ws_streamout_tiles(M, N, L)
    staging = torch.empty(T * T_EDGE * T_EDGE, dtype=torch.bfloat16, device="cuda")
    flags = torch.empty(2 * T, dtype=torch.int32, device="cuda")
    gw_each.run(Ad, Bd, None, D0, 1.0, 0.0)
    for _ in range(5):   # flags and counter are reset by every call
        gw_each.run_streamout(Ad, Bd, None, D1, staging, flags, 1.0, 0.0)
    torch.cuda.synchronize()
    assert torch.equal(D0.view(torch.int16), D1.view(torch.int16))
    check_staging(D1, staging, flags)


def test_streamout_workload(gw):
    """The 8192 x 8192 x 4096 stream-out workload at full size: staging
    bit-exact against D, and every element of D against the oracle."""
    w = workloads.WORKLOADS[workloads.STREAMOUT]
    A, B, _ = workloads.workload_inputs(w)
    Ad, Bd = A.cuda(), B.cuda()
    T = gemm_ws.gemm_ws_streamout_tiles(w.M, w.N, w.L)
    staging = torch.empty(T * T_EDGE * T_EDGE, dtype=torch.bfloat16, device="cuda")
    flags = torch.empty(2 * T, dtype=torch.int32, device="cuda")
    D = torch.empty(w.L, w.M, w.N, dtype=torch.bfloat16, device="cuda")
    gw.run_streamout(Ad, Bd, None, D, staging, flags, w.alpha, w.beta)
    torch.cuda.synchronize()
    check_staging(D, staging, flags)
    check_every_row(bits_of(D), A, B, None, w.M, w.N, w.K, w.L, w.alpha, w.beta,
                    "streamout workload")
