"""Overlap of the tile handoff with compute, and correct handoff, on the
8192 x 8192 x 4096 stream-out workload (debug build timestamps).

For every persistent CTA (group) and every tile it computes, the debug build
stamps the global time at which the tile's accumulator was complete (seen by
the epilogue) and at which the consumer warp had published the tile's last
stream-out flag. Overlap means the handoff of tile i is done while the MMA
is still working on later tiles: tile i must be published before the
accumulator of tile i+2 completes (the MMA warp can only be one tile ahead of
the epilogue, since there are two accumulators). The staging buffer must
still match D bit for bit, every tile flagged exactly once.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from async_pipelines_gb300 import gemm_ws, workloads
from tests.debug_helpers import configure, debug_handle, launch_shape
from tests.test_streamout_gpu import check_staging

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("cta_group", [2, 1])
def test_streamout_overlaps_mma(cta_group):
    w = workloads.WORKLOADS[workloads.STREAMOUT]
    g = debug_handle(cta_group=cta_group)
    cg, clusters, tiles, sk_tiles = launch_shape(g, w.M, w.N, w.K, w.L)   # cg: CTAs per cluster
    assert sk_tiles == 0
    assert cg == cta_group
    trace = torch.zeros(tiles * cg * 2, dtype=torch.int64, device="cuda")
    configure(g, fault=0, trace_ptr=trace.data_ptr())
    A, B, _ = workloads.workload_inputs(w)
    Ad, Bd = A.cuda(), B.cuda()
    T = gemm_ws.gemm_ws_streamout_tiles(w.M, w.N, w.L)
    staging = torch.empty(T * 128 * 128, dtype=torch.bfloat16, device="cuda")
    flags = torch.empty(2 * T, dtype=torch.int32, device="cuda")
    D = torch.empty(w.L, w.M, w.N, dtype=torch.bfloat16, device="cuda")
    g.run_streamout(Ad, Bd, None, D, staging, flags, w.alpha, w.beta)
    assert g.query_status() == gemm_ws.OK
    configure(g, fault=0)
    g.close()
    check_staging(D, staging, flags)

    tr = trace.cpu().numpy().reshape(tiles, cg, 2)
    assert np.all(tr > 0), "a tile part was never stamped"
    strict = total = 0
    for c in range(clusters):
        seq = np.arange(c, tiles, clusters)
        for r in range(cg):
            acc, pub = tr[seq, r, 0], tr[seq, r, 1]
            assert np.all(np.diff(acc) > 0), "accumulators completed out of order"
            assert np.all(pub >= acc), "published before the accumulator was complete"
            assert np.all(pub[:-2] < acc[2:]), f"cluster {c} rank {r}: handoff trails compute"
            strict += int(np.sum(pub[:-1] < acc[1:]))
            total += len(seq) - 1
    # Most tiles are even published before the NEXT accumulator completes.
    print(f"published before the next tile's accumulator: {strict}/{total}")
    assert strict >= 0.5 * total
