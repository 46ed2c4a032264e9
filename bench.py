"""Benchmark of the persistent warp-specialized bf16 GEMM on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With --gpus N > 1 and no outer launcher (no WORLD_SIZE in the environment)
the script starts N rank processes itself, one per GPU; under torchrun it
uses the launcher's ranks.

One step = one GEMM D = alpha*A*B + beta*C over the 8192^3 workload (A, B
uniform[-1,1), C normal(0,1), alpha 1.5, beta 0.5), inputs resident in HBM.
Every step's inputs (512 MiB) exceed the 129 MB L2, so L2 is not flushed.

Printed (rank 0, one JSON line): whole-job TFLOP/s (all ranks; replicas on N
GPUs, weak scaling), the fraction of the measured dense bf16 peak, the
end-to-end figure through the C ABI with host buffers, the stream-out
overhead on the 8192 x 8192 x 4096 workload, the roofline record of the GEMM
kernel, SM clocks sampled during the timed region, a fixed-length sustained
leg (back-to-back launches for at least half a second, under the power cap,
with its own clock record), and the CPU oracle timed on a bounded sample of
the same workload on this host's cores.

`--impl reference` times that CPU oracle as the reference arm.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import socket
import statistics
import subprocess
import sys
import tempfile
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from async_pipelines_gb300 import workloads  # noqa: E402

METRIC = ("bf16 GEMM TFLOP/s & % of GB300 dense bf16 peak (8192³); "
          "stream-out overhead %")
UNIT = "TFLOP/s"
NOMINAL_BF16_TFLOPS = 2250.0
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# Timed regions at least this long are compared with the sustained peak.
SUSTAINED_MIN_S = 0.25
# Length of the sustained leg: back-to-back launches timed as one region.
SUSTAINED_LEG_S = 0.6
KERNEL_SOURCES = ["async_pipelines_gb300/csrc/gemm_ws.cu",
                  "async_pipelines_gb300/csrc/gemm_ws_kernel.cuh",
                  "async_pipelines_gb300/csrc/ptx.cuh"]
# DRAM bytes per launch of the GEMM kernel from one ncu capture, keyed by the
# workload, with the hash of the kernel sources the capture was taken with.
# A stale hash reports traffic as null.
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


def kernel_hash() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def traffic_for(workload: str):
    if not os.path.exists(TRAFFIC_FILE):
        return None
    with open(TRAFFIC_FILE) as f:
        rec = json.load(f).get(workload)
    if not rec or rec.get("kernel_hash") != kernel_hash():
        return None
    return rec.get("dram_bytes_per_launch")


# ------------------------------------------------------------------ distributed

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_process(rank: int, world: int, port: int, argv, target):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      LOCAL_WORLD_SIZE=str(world))
    (target or main)(argv)


def spawn_ranks(world: int, argv, target=None, timeout_s: float = 3600.0) -> int:
    """Runs `target(argv)` (default: this script's main) in `world` fresh
    processes on this node, rank r with RANK = LOCAL_RANK = r and a
    rendezvous on 127.0.0.1, as torchrun would. Returns the worst exit code."""
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    port = _free_port()
    procs = [ctx.Process(target=_rank_process, args=(r, world, port, argv, target))
             for r in range(world)]
    for p in procs:
        p.start()
    deadline = time.monotonic() + timeout_s
    for p in procs:
        p.join(timeout=max(1.0, deadline - time.monotonic()))
    codes = []
    for p in procs:
        if p.is_alive():   # a rank that never finished: stop it, report failure
            p.terminate()
            p.join(timeout=10)
            codes.append(1)
        else:
            codes.append(p.exitcode or 0)
    return max(codes)


def init_ranks(world: int):
    """Process group of the replicas: NCCL between GPUs, gloo without CUDA."""
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device: str = "cuda") -> float:
    """The largest of every rank's x (the slowest rank's time)."""
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_rank: float, world: int, ms_slowest: float) -> float:
    """Whole-job TFLOP/s: all ranks' work over the slowest rank's time."""
    return world * flops_per_rank / (ms_slowest * 1e-3) / 1e12


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.out.flush()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        with open(self.out.name) as f:
            lines = [ln.strip() for ln in f if ln.strip()]
        os.unlink(self.out.name)
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        # samples under load: the timed region keeps the GPU busy throughout
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "power_w_max": max(power), "samples": len(sm), "reasons": sorted(reasons)}


# ------------------------------------------------------------------ CPU oracle

class OracleSampler:
    """Times the CPU oracle on bounded row samples of workload `w`.

    Inputs are drawn once; the oracle's rate is calibrated once on all cores;
    each sample is then a set of whole output rows (each row is 2*N*K FLOPs),
    evenly spread over the output, sized to take about `seconds`."""

    def __init__(self, w: workloads.Workload):
        import numpy as np
        self.np = np
        self.w = w
        self.cores = len(os.sched_getaffinity(0))
        A, B, C = workloads.workload_inputs(w)
        self.Ab, self.Bb = workloads.bf16_bits(A), workloads.bf16_bits(B)
        self.Cb = workloads.bf16_bits(C) if C is not None else None
        rows = self.np.arange(self.cores, dtype=self.np.int64)
        _, dt = self._time(rows)
        self.rows_per_s = self.cores / max(dt, 1e-6)

    def _time(self, rows):
        import oracle
        w = self.w
        t0 = time.perf_counter()
        oracle.gemm_rows(self.Ab, self.Bb, self.Cb, w.M, w.N, w.K, w.L, w.alpha, w.beta,
                         rows=rows, threads=self.cores)
        return len(rows), time.perf_counter() - t0

    def sample(self, seconds: float):
        """Returns (TFLOP/s, seconds, description) of one timed sample."""
        w = self.w
        n = int(min(w.M * w.L, max(self.cores, seconds * self.rows_per_s)))
        n = max(self.cores, (n // self.cores) * self.cores)
        rows = self.np.linspace(0, w.M * w.L - 1, n).astype(self.np.int64)
        n, dt = self._time(rows)
        flops = 2.0 * n * w.N * w.K
        desc = (f"{n} of {w.M * w.L} output rows of {w.name} "
                f"({flops / 1e9:.1f} GFLOP, {dt:.2f} s, fp64 triple loop, {self.cores} threads)")
        return flops / dt / 1e12, dt, desc


# ------------------------------------------------------------------ GPU arm

def time_launches(fn, steps: int, stream) -> float:
    """Mean ms per call of `fn` over `steps` calls, CUDA events on `stream`."""
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for _ in range(steps):
        fn()
    end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end) / steps


def time_scrubbed(fn, runs: int, stream, scrub) -> float:
    """Median ms of single calls of `fn`, each one after a write of `scrub`
    (256 MiB, twice the L2), so that no call finds its inputs in L2. CUDA
    events on `stream` bracket the call alone, not the scrub."""
    pairs = []
    for i in range(runs):
        scrub.fill_(i & 0xFF)
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(stream)
        fn()
        end.record(stream)
        pairs.append((start, end))
    torch.cuda.synchronize()
    ms = sorted(s.elapsed_time(e) for s, e in pairs)
    return ms[len(ms) // 2]


def time_e2e_serial(g, w, Ah, Bh, Ch, Ad, Bd, Cd, D, stream, warmup, steps, world):
    """ms per step of copy-in, GEMM, copy-out, one after another on one stream."""
    Dh = torch.empty(D.shape, dtype=D.dtype).pin_memory()

    def step():
        Ad.copy_(Ah, non_blocking=True)
        Bd.copy_(Bh, non_blocking=True)
        Cd.copy_(Ch, non_blocking=True)
        g.run(Ad, Bd, Cd, D, w.alpha, w.beta)
        Dh.copy_(D, non_blocking=True)

    for _ in range(max(1, warmup)):
        step()
    barrier(world)
    return time_launches(step, steps, stream)


def time_e2e_pipelined(g, w, Ah, Bh, Ch, dev, comp, warmup, steps, world, one_copy_stream=False,
                       copy_streams=1):
    """ms per step with copy-in of step i+1 and copy-out of step i-1 overlapping
    the GEMM of step i (two device buffer sets, events between the streams).
    one_copy_stream: both copy directions on the same stream(s), so they
    overlap the GEMMs but not each other (on some hosts the two directions at
    once are slower than one after the other). copy_streams: every copy split
    into that many chunks, each on its own stream (per direction)."""
    bufs = [tuple(torch.empty(t.shape, dtype=t.dtype, device=dev) for t in (Ah, Bh, Ch))
            + (torch.empty(w.L, w.M, w.N, dtype=torch.bfloat16, device=dev),)
            for _ in range(2)]
    Dh = [torch.empty(w.L, w.M, w.N, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    cin = [torch.cuda.Stream(device=dev) for _ in range(copy_streams)]
    cout = cin if one_copy_stream else [torch.cuda.Stream(device=dev) for _ in range(copy_streams)]
    copy_lanes = cin if one_copy_stream else cin + cout
    ev = {k: [[torch.cuda.Event() for _ in range(copy_streams)] for _ in range(2)]
          for k in ("in", "out")}
    ev_gemm = [torch.cuda.Event() for _ in range(2)]

    def chunk(t, j):
        f = t.view(-1)
        c = (f.numel() + copy_streams - 1) // copy_streams
        return f[j * c:(j + 1) * c]

    def copy_in(i):
        b = i % 2
        for j, st in enumerate(cin):
            with torch.cuda.stream(st):
                if i >= 2:
                    st.wait_event(ev_gemm[b])      # step i-2 no longer reads buffer set b
                for dst, src in zip(bufs[b][:3], (Ah, Bh, Ch)):
                    chunk(dst, j).copy_(chunk(src, j), non_blocking=True)
                ev["in"][b][j].record(st)

    def compute(i):
        b = i % 2
        Ad, Bd, Cd, Dd = bufs[b]
        for j in range(copy_streams):
            comp.wait_event(ev["in"][b][j])
            if i >= 2:
                comp.wait_event(ev["out"][b][j])   # step i-2's D has been read back
        g.run(Ad, Bd, Cd, Dd, w.alpha, w.beta, stream=comp)
        ev_gemm[b].record(comp)

    def copy_out(i):
        b = i % 2
        for j, st in enumerate(cout):
            with torch.cuda.stream(st):
                st.wait_event(ev_gemm[b])
                chunk(Dh[b], j).copy_(chunk(bufs[b][3], j), non_blocking=True)
                ev["out"][b][j].record(st)

    def run(n):
        # issue order in(0), in(1), gemm(0), out(0), in(2), gemm(1), out(1), ...:
        # on a shared copy stream the copy-in of step i+1 then sits ahead of
        # the copy-out of step i, so both overlap the GEMM of step i.
        for st in copy_lanes:
            st.wait_stream(comp)
        for i in range(n + 1):
            if i < n:
                copy_in(i)
            if i >= 1:
                compute(i - 1)
                copy_out(i - 1)
        for st in copy_lanes:
            comp.wait_stream(st)

    run(max(2, warmup))
    torch.cuda.synchronize()
    barrier(world)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(comp)
    run(steps)
    end.record(comp)
    torch.cuda.synchronize()
    return start.elapsed_time(end) / steps


def other_workloads(g, dev, stream, steps: int = 30):
    """Informational figures for the other workloads (not the headline):
    TFLOP/s of the 4096^3 and ragged batched GEMMs, launch-to-launch latency
    of the 256^3 GEMM (latency-bound), and the HBM bandwidth of a skinny
    8192 x 8192 x 64 GEMM (bound by writing D), per call and replayed from a
    CUDA graph."""
    out = {}
    # Both of these fit in L2 (96 MiB of operands at 4096^3), so they are
    # also timed with the L2 scrubbed before every call.
    scrubbed = ("gemm_256x256x256", "gemm_4096x4096x4096")
    scrub = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    cases = [(workloads.WORKLOADS["gemm_256x256x256"], "us"),
             (workloads.WORKLOADS["gemm_4096x4096x4096"], "tflops"),
             (workloads.WORKLOADS["gemm_batched4_5000x3000x4000_ragged"], "tflops"),
             (workloads.EXTRA_WORKLOADS[workloads.SKINNY], "gbs")]
    for w, kind in cases:
        A, B, C = workloads.workload_inputs(w)
        Ad, Bd = A.to(dev), B.to(dev)
        Cd = C.to(dev) if C is not None else None
        D = torch.empty(w.L, w.M, w.N, dtype=torch.bfloat16, device=dev)
        step = lambda: g.run(Ad, Bd, Cd, D, w.alpha, w.beta)
        for _ in range(3):
            step()
        ms = time_launches(step, steps, stream)
        rec = {"ms_per_launch": round(ms, 5)}
        if kind == "us":
            rec["us_per_launch"] = round(ms * 1e3, 2)
            # The same calls captured once in a CUDA graph and replayed: the
            # device time per GEMM without the per-call host path.
            rec["us_per_gemm_graph_replay"] = round(graph_replay_us(g, Ad, Bd, Cd, D, w, dev), 2)
        if kind in ("tflops", "us"):
            rec["tflops"] = round(w.flops / (ms * 1e-3) / 1e12, 2)
        if w.name in scrubbed:
            cold = time_scrubbed(step, 20, stream, scrub)
            rec["l2_scrubbed"] = {"ms_median_of_20": round(cold, 5),
                                  "us": round(cold * 1e3, 2),
                                  "tflops": round(w.flops / (cold * 1e-3) / 1e12, 2)}
        if kind == "gbs":
            rec["gbs"] = round(w.algorithmic_bytes() / (ms * 1e-3) / 1e9, 1)
            rec["algorithmic_bytes"] = w.algorithmic_bytes()
            # The same GEMM replayed from a CUDA graph: device time without
            # the per-call host path between launches.
            us = graph_replay_us(g, Ad, Bd, Cd, D, w, dev)
            rec["us_per_gemm_graph_replay"] = round(us, 2)
            rec["gbs_graph_replay"] = round(w.algorithmic_bytes() / (us * 1e-6) / 1e9, 1)
        out[w.name] = rec
        del A, B, C, Ad, Bd, Cd, D
    del scrub
    torch.cuda.empty_cache()
    return out


def graph_replay_us(g, Ad, Bd, Cd, D, w, dev, per_graph: int = 20, replays: int = 10) -> float:
    """Median device time per GEMM over replays of a CUDA graph holding
    `per_graph` back-to-back calls (CUDA events around each replay)."""
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(3):
            g.run(Ad, Bd, Cd, D, w.alpha, w.beta, stream=s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        for _ in range(per_graph):
            g.run(Ad, Bd, Cd, D, w.alpha, w.beta, stream=s)
    graph.replay()
    torch.cuda.synchronize()
    times = []
    for _ in range(replays):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        graph.replay()
        b.record()
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b) * 1e3 / per_graph)
    return statistics.median(times)


def run_ours(args, rank, world, local):
    from async_pipelines_gb300 import gemm_ws

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    g = gemm_ws.GemmWS(local)
    w = workloads.WORKLOADS[workloads.HEADLINE]
    A, B, C = workloads.workload_inputs(w)
    Ad, Bd, Cd = A.to(dev), B.to(dev), C.to(dev)
    D = torch.empty(w.L, w.M, w.N, dtype=torch.bfloat16, device=dev)
    step = lambda: g.run(Ad, Bd, Cd, D, w.alpha, w.beta)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    barrier(world)
    with ClockSampler(local) as clocks:
        torch.cuda.synchronize()
        barrier(world)
        ms_local = time_launches(step, args.steps, stream)
        barrier(world)
    ms = max_over_ranks(ms_local, world)
    kernels_per_step = g.kernels_per_run(w.M, w.N, w.K, w.L)
    status = g.query_status()
    if status != gemm_ws.OK:
        raise RuntimeError(f"device status after timing: {gemm_ws.status_string(status)}")
    tflops_rank = w.flops / (ms * 1e-3) / 1e12
    value = job_throughput(w.flops, world, ms)
    # Sustained leg: a fixed length of back-to-back launches (independent of
    # --steps) timed as one region, in the power-capped steady state that a
    # user of long GEMM streams sees, with its own clock record.
    n_sus = max(50, math.ceil(SUSTAINED_LEG_S / (ms * 1e-3)))
    barrier(world)
    with ClockSampler(local) as sus_clocks:
        torch.cuda.synchronize()
        ms_sus = max_over_ranks(time_launches(step, n_sus, stream), world)
    sustained = {"launches": n_sus, "seconds": round(n_sus * ms_sus * 1e-3, 3),
                 "ms_per_launch": round(ms_sus, 4),
                 "tflops": round(job_throughput(w.flops, world, ms_sus), 2),
                 "clocks": sus_clocks.summary()}
    # Informational: 20 single launches, each timed alone (events around one
    # call, synchronised between calls), median and best.
    singles = sorted(time_launches(step, 1, stream) for _ in range(20))
    single = {"n": len(singles), "median_ms": round(statistics.median(singles), 4),
              "best_ms": round(singles[0], 4),
              "median_tflops": round(w.flops / (statistics.median(singles) * 1e-3) / 1e12, 2),
              "best_tflops": round(w.flops / (singles[0] * 1e-3) / 1e12, 2)}

    # End to end through the C ABI with host buffers: every step copies its
    # inputs A, B, C in from pinned host memory and reads D back. The timed
    # loop is a 2-deep software pipeline (two device buffer sets, a copy-in
    # stream, the compute stream and a copy-out stream), so step i+1's copy-in
    # and step i-1's copy-out overlap step i's GEMM; all copies of all timed
    # steps are inside the timed region. The plain serial loop is reported too.
    Ah, Bh, Ch = A.pin_memory(), B.pin_memory(), C.pin_memory()
    e2e_steps = max(3, min(args.steps, 20))
    h2d = sum(t.numel() * t.element_size() for t in (Ah, Bh, Ch))
    d2h = 2 * w.L * w.M * w.N
    e2e_serial_ms = max_over_ranks(time_e2e_serial(g, w, Ah, Bh, Ch, Ad, Bd, Cd, D, stream,
                                                   args.warmup, e2e_steps, world), world)
    del Ad, Bd, Cd, D
    torch.cuda.empty_cache()
    e2e_pipe_ms = max_over_ranks(time_e2e_pipelined(g, w, Ah, Bh, Ch, dev, stream, args.warmup,
                                                    e2e_steps, world), world)
    torch.cuda.empty_cache()
    e2e_pipe1_ms = max_over_ranks(time_e2e_pipelined(g, w, Ah, Bh, Ch, dev, stream, args.warmup,
                                                     e2e_steps, world, one_copy_stream=True),
                                  world)
    torch.cuda.empty_cache()
    e2e_pipe8_ms = max_over_ranks(time_e2e_pipelined(g, w, Ah, Bh, Ch, dev, stream, args.warmup,
                                                     e2e_steps, world, copy_streams=8),
                                  world)
    # The reported end-to-end figure is the fastest of the schedules (every
    # one copies every step's inputs in and its result out inside the timed
    # region); all are listed.
    e2e_schedules = {
        "serial: copy-in, GEMM, copy-out on one stream": e2e_serial_ms,
        "2-deep pipeline: copy-in / GEMM / copy-out streams": e2e_pipe_ms,
        "2-deep pipeline: one copy stream for both directions / GEMM stream": e2e_pipe1_ms,
        "2-deep pipeline: every copy in 8 chunks on 8 streams per direction / GEMM stream":
            e2e_pipe8_ms,
    }
    e2e_schedule, e2e_ms = min(e2e_schedules.items(), key=lambda kv: kv[1])
    del Ah, Bh, Ch
    torch.cuda.empty_cache()

    # Stream-out overhead: same inputs, interleaved plain / stream-out runs.
    so = workloads.WORKLOADS[workloads.STREAMOUT]
    As, Bs, _ = workloads.workload_inputs(so)
    As, Bs = As.to(dev), Bs.to(dev)
    Ds = torch.empty(so.L, so.M, so.N, dtype=torch.bfloat16, device=dev)
    T = gemm_ws.gemm_ws_streamout_tiles(so.M, so.N, so.L)
    staging = torch.empty(T * 128 * 128, dtype=torch.bfloat16, device=dev)
    flags = torch.empty(2 * T, dtype=torch.int32, device=dev)
    plain = lambda: g.run(As, Bs, None, Ds, so.alpha, so.beta)
    streamed = lambda: g.run_streamout(As, Bs, None, Ds, staging, flags, so.alpha, so.beta)
    for _ in range(3):
        plain()
        streamed()
    t_plain, t_so = [], []
    for _ in range(max(20, args.overhead_reps)):
        t_plain.append(time_launches(plain, 1, stream))
        t_so.append(time_launches(streamed, 1, stream))
    mp, ms_so = statistics.median(t_plain), statistics.median(t_so)
    overhead = (ms_so - mp) / mp * 100.0
    status = g.query_status()
    if status != gemm_ws.OK:
        raise RuntimeError(f"device status after stream-out: {gemm_ws.status_string(status)}")
    del As, Bs, Ds, staging, flags
    torch.cuda.empty_cache()
    others = other_workloads(g, dev, stream)
    g.close()

    if rank != 0:
        return
    peaks, peak_src = load_peaks()
    peak = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    peak_sus = peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
    # The roofline denominator matches how the kernel was timed: launches
    # back to back for a quarter of a second or more run in the power-capped
    # regime of the sustained library measurement (a seconds-long loop);
    # shorter timed regions compare with the burst figure.
    timed_s = ms * args.steps / 1e3
    regime = "sustained" if timed_s >= SUSTAINED_MIN_S else "burst"
    roof_peak = peak_sus if regime == "sustained" else peak
    sustained["peak_sustained"] = peak_sus
    sustained["frac_of_sustained"] = round(
        w.flops / (sustained["ms_per_launch"] * 1e-3) / 1e12 / peak_sus, 4)
    cpu = None
    if not args.no_cpu_baseline:
        sampler = OracleSampler(w)
        v, _, desc = sampler.sample(args.cpu_budget)
        cpu = {"value": v, "unit": UNIT, "cores": sampler.cores, "kind": "oracle",
               "sample": desc}
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded uniform/normal bf16, no dataset)",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "L": w.L,
                   "alpha": w.alpha, "beta": w.beta, "accumulate": "fp32", "out": "bf16",
                   "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (512 MiB per step), no flush"},
        "pct_of_nominal_2250_tflops": round(100.0 * tflops_rank / NOMINAL_BF16_TFLOPS, 2),
        "pct_of_measured_bf16_burst": round(100.0 * tflops_rank / peak, 2),
        "single_launch": single,
        "sustained": sustained,
        "streamout_overhead_pct": round(overhead, 2),
        "streamout": {"workload": so.name, "plain_ms_median": round(mp, 4),
                      "streamout_ms_median": round(ms_so, 4), "reps": len(t_plain),
                      "plain_tflops": round(so.flops / (mp * 1e-3) / 1e12, 2)},
        "e2e": {"value": round(world * w.flops / (e2e_ms * 1e-3) / 1e12, 2), "unit": UNIT,
                "ms_per_step": round(e2e_ms, 4),
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "schedule": e2e_schedule,
                "schedules_ms_per_step": {k: round(v, 4) for k, v in e2e_schedules.items()},
                "serial_value": round(world * w.flops / (e2e_serial_ms * 1e-3) / 1e12, 2),
                "serial_ms_per_step": round(e2e_serial_ms, 4)},
        # this library's kernels in the timed region (the GEMM, and the
        # reduction where the plan splits the last wave's tiles into pieces)
        "gpu_launches": args.steps * kernels_per_step,
        "kernels_per_step": kernels_per_step,
        "pct_of_measured_bf16_sustained": round(
            100.0 * tflops_rank / peaks.get("bf16_tflops_sustained", peak), 2),
        "roofline": {"bound": "tensor", "achieved": round(tflops_rank, 2), "peak": roof_peak,
                     "unit": "TFLOP/s", "frac": round(tflops_rank / roof_peak, 4),
                     "peak_source": f"{peak_src} bf16 {regime} (cuBLAS 8192^3); timed region "
                                    f"{timed_s:.2f} s of back-to-back launches",
                     "frac_of_burst": round(tflops_rank / peak, 4),
                     "traffic": traffic_for(w.name),
                     "algorithmic_bytes_per_launch": w.algorithmic_bytes(),
                     "kernel": "gws::gemm_ws_kernel"},
        "other_workloads": others,
        "clocks": clocks.summary(),
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)


def run_kernel_only(args, local):
    """Only the GEMM launches of one workload (warmup + steps), for profilers."""
    from async_pipelines_gb300 import gemm_ws

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    g = gemm_ws.GemmWS(local)
    w = workloads.workload(args.workload or workloads.HEADLINE)
    A, B, C = workloads.workload_inputs(w)
    Ad, Bd = A.to(dev), B.to(dev)
    Cd = C.to(dev) if C is not None else None
    D = torch.empty(w.L, w.M, w.N, dtype=torch.bfloat16, device=dev)
    if w.streamout:
        T = gemm_ws.gemm_ws_streamout_tiles(w.M, w.N, w.L)
        staging = torch.empty(T * 128 * 128, dtype=torch.bfloat16, device=dev)
        flags = torch.empty(2 * T, dtype=torch.int32, device=dev)
        step = lambda: g.run_streamout(Ad, Bd, Cd, D, staging, flags, w.alpha, w.beta)
    else:
        step = lambda: g.run(Ad, Bd, Cd, D, w.alpha, w.beta)
    for _ in range(args.warmup):
        step()
    ms = time_launches(step, args.steps, torch.cuda.current_stream())
    status = g.query_status()
    g.close()
    if status != gemm_ws.OK:
        raise RuntimeError(f"device status: {gemm_ws.status_string(status)}")
    print(json.dumps({"workload": w.name, "ms_per_launch": round(ms, 4),
                      "tflops": round(w.flops / (ms * 1e-3) / 1e12, 2)}), flush=True)


def run_vs_library(args, local):
    """Library cross-check (not the product path): the headline GEMM through
    this library and through torch.addmm (cuBLAS) with the same alpha/beta
    epilogue, timed in interleaved rounds of --steps launches each on one
    GPU, so both see the same power and clock state. Prints one JSON line."""
    from async_pipelines_gb300 import gemm_ws

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    g = gemm_ws.GemmWS(local)
    w = workloads.WORKLOADS[workloads.HEADLINE]
    A, B, C = workloads.workload_inputs(w)
    Ad, Bd, Cd = A.to(dev), B.to(dev), C.to(dev)
    D = torch.empty(w.L, w.M, w.N, dtype=torch.bfloat16, device=dev)
    ours = lambda: g.run(Ad, Bd, Cd, D, w.alpha, w.beta)
    lib = lambda: torch.addmm(Cd[0], Ad[0], Bd[0].t(), beta=w.beta, alpha=w.alpha, out=D[0])
    res = {"gemm_ws": [], "torch.addmm": []}
    for rnd in range(args.rounds):
        order = [("gemm_ws", ours), ("torch.addmm", lib)]
        for name, fn in (order if rnd % 2 == 0 else order[::-1]):
            for _ in range(args.warmup):
                fn()
            ms = time_launches(fn, args.steps, stream)
            res[name].append(w.flops / (ms * 1e-3) / 1e12)
    status = g.query_status()
    g.close()
    if status != gemm_ws.OK:
        raise RuntimeError(f"device status: {gemm_ws.status_string(status)}")
    out = {k: {"tflops_median": round(statistics.median(v), 1),
               "tflops_rounds": [round(x, 1) for x in v]} for k, v in res.items()}
    print(json.dumps({"workload": w.name, "steps_per_round": args.steps, "rounds": args.rounds,
                      "interleaved": True, **out}), flush=True)


def run_reference(args, rank, world, local):
    """The reference arm: the CPU oracle as it stands, timed on this host's
    cores, on bounded row samples of the headline workload; the whole run
    (W warm-up + K timed samples) takes about --cpu-budget seconds."""
    if rank != 0:
        return
    w = workloads.WORKLOADS[workloads.HEADLINE]
    sampler = OracleSampler(w)
    per_step = args.cpu_budget / max(1, args.steps + args.warmup)
    for _ in range(args.warmup):
        sampler.sample(per_step)
    vals, secs, desc = [], 0.0, ""
    for _ in range(args.steps):
        v, dt, desc = sampler.sample(per_step)
        vals.append(v)
        secs += dt
    value = statistics.median(vals)
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(1000.0 * secs / max(1, args.steps), 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded uniform/normal bf16, no dataset)",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "L": w.L,
                   "alpha": w.alpha, "beta": w.beta},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": sampler.cores, "kind": "oracle",
                         "sample": f"per step: {desc}"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-budget", type=float, default=15.0,
                    help="seconds of CPU oracle work: the baseline sample, or the whole "
                         "reference arm")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--overhead-reps", type=int, default=300,
                    help="interleaved plain / stream-out launch pairs for the overhead median")
    ap.add_argument("--kernel-only", action="store_true",
                    help="launch only the GEMM of --workload (for profilers); no contract line")
    ap.add_argument("--workload", choices=sorted(workloads.WORKLOADS) + sorted(workloads.EXTRA_WORKLOADS),
                    default=None)
    ap.add_argument("--vs-library", action="store_true",
                    help="interleaved rounds against torch.addmm (cuBLAS) on the headline "
                         "workload; a cross-check, no contract line")
    ap.add_argument("--rounds", type=int, default=6)
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # No outer launcher: start one rank per GPU here.
        sys.exit(spawn_ranks(args.gpus, sys.argv[1:] if argv is None else argv))
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world, local)
        return
    if args.kernel_only:
        run_kernel_only(args, local)
        return
    if args.vs_library:
        run_vs_library(args, local)
        return
    if world > 1:
        torch.cuda.set_device(local)
    init_ranks(world)
    try:
        run_ours(args, rank, world, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
