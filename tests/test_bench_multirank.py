"""The benchmark's multi-rank plumbing on CPU: two gloo ranks.

GEMM replicas share nothing on the data path; across ranks the benchmark
only synchronises (barrier) and takes the slowest rank's time (all-reduce
MAX), then counts every rank's work. Those pieces run here with the gloo
backend and world size 2, exactly as the NCCL path uses them on GPUs.
"""
from __future__ import annotations

import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        assert (r, w, local) == (rank, world, rank)
        bench.barrier(w)
        ms = [1.25, 2.5][rank]
        slowest = bench.max_over_ranks(ms, w, device="cpu")
        out.put((rank, slowest, bench.job_throughput(1e12, w, slowest)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_sum_the_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, slowest, tflops in got:
        assert slowest == 2.5
        # 2 ranks x 1e12 FLOP in 2.5 ms
        assert tflops == pytest.approx(2 * 1e12 / 2.5e-3 / 1e12)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.0, 1) == 3.0
    bench.barrier(1)
    assert bench.job_throughput(2e12, 1, 1.0) == pytest.approx(2000.0)
