"""The benchmark's multi-rank plumbing on CPU: two gloo ranks.

GEMM replicas share nothing on the data path; across ranks the benchmark
only synchronises (barrier) and takes the slowest rank's time (all-reduce
MAX), then counts every rank's work. Those pieces run here with the gloo
backend and world size 2, exactly as the NCCL path uses them on GPUs. So
does the launcher of its own that `bench.py --gpus N` uses when no torchrun
started it: N spawned processes with the rank variables set.
"""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys

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


def _probe(argv):
    """Body of each rank started by bench.spawn_ranks (CPU, gloo)."""
    rank, world, local = bench.dist_env()
    bench.init_ranks(world)            # gloo: this machine has no CUDA
    try:
        bench.barrier(world)
        slowest = bench.max_over_ranks([4.0, 1.5, 3.0][rank], world, device="cpu")
        with open(os.path.join(argv[0], f"rank{rank}.json"), "w") as f:
            json.dump({"rank": rank, "world": world, "local": local, "slowest": slowest}, f)
    finally:
        import torch.distributed as d
        d.destroy_process_group()


def test_spawned_ranks_rendezvous_without_an_outer_launcher(tmp_path):
    """--gpus N without torchrun: bench.spawn_ranks starts N processes with
    RANK = LOCAL_RANK = r and WORLD_SIZE = N that form one process group."""
    rc = bench.spawn_ranks(3, [str(tmp_path)], target=_probe, timeout_s=120)
    assert rc == 0
    got = sorted(json.loads((tmp_path / f"rank{r}.json").read_text())["rank"] for r in range(3))
    assert got == [0, 1, 2]
    for r in range(3):
        rec = json.loads((tmp_path / f"rank{r}.json").read_text())
        assert (rec["world"], rec["local"], rec["slowest"]) == (3, r, 4.0)


def _fails(argv):
    raise SystemExit(3 if os.environ["RANK"] == "1" else 0)


def test_spawned_ranks_report_the_worst_exit_code():
    assert bench.spawn_ranks(2, [], target=_fails, timeout_s=60) == 3


def test_bench_gpus_two_spawns_two_ranks_and_rank0_prints_one_line():
    """The command line the driver uses for N GPUs, minus torchrun: the
    reference arm (CPU only) runs on two self-started ranks and only rank 0
    prints its JSON line."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {k: v for k, v in os.environ.items()
           if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT")}
    out = subprocess.run(
        [sys.executable, os.path.join(root, "bench.py"), "--gpus", "2", "--impl", "reference",
         "--steps", "1", "--warmup", "3", "--cpu-budget", "1"],
        cwd=root, env=env, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2
