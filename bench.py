"""Benchmark of the persistent warp-specialized bf16 GEMM on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one GEMM D = alpha*A*B + beta*C over the 8192^3 workload (A, B
uniform[-1,1), C normal(0,1), alpha 1.5, beta 0.5), inputs resident in HBM.
Every step's inputs (512 MiB) exceed the 129 MB L2, so L2 is not flushed.

Printed (rank 0, one JSON line): whole-job TFLOP/s (all ranks; replicas on N
GPUs, weak scaling), the fraction of the measured dense bf16 peak, the
end-to-end figure through the C ABI with host buffers, the stream-out
overhead on the 8192 x 8192 x 4096 workload, the roofline record of the GEMM
kernel, SM clocks sampled during the timed region, and the CPU oracle timed
on a bounded sample of the same workload on this host's cores.

`--impl reference` times that CPU oracle as the reference arm.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
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


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


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

def oracle_sample(w: workloads.Workload, budget_s: float):
    """Times the CPU oracle on a bounded row sample of workload `w`.

    Returns (TFLOP/s, cores, description). The sample is whole output rows
    (each row is 2*N*K FLOPs), sized from a one-row probe to take about
    `budget_s` seconds on every core of this host."""
    import numpy as np
    import oracle

    cores = len(os.sched_getaffinity(0))
    A, B, C = workloads.workload_inputs(w)
    Ab, Bb = workloads.bf16_bits(A), workloads.bf16_bits(B)
    Cb = workloads.bf16_bits(C) if C is not None else None
    probe = np.array([0], dtype=np.int64)
    t0 = time.perf_counter()
    oracle.gemm_rows(Ab, Bb, Cb, w.M, w.N, w.K, w.L, w.alpha, w.beta, rows=probe, threads=1)
    per_row_1core = time.perf_counter() - t0
    nrows = int(max(cores, min(w.M * w.L, budget_s * cores / max(per_row_1core, 1e-6))))
    nrows = max(cores, (nrows // cores) * cores)
    rows = np.linspace(0, w.M * w.L - 1, nrows).astype(np.int64)
    t0 = time.perf_counter()
    oracle.gemm_rows(Ab, Bb, Cb, w.M, w.N, w.K, w.L, w.alpha, w.beta, rows=rows, threads=cores)
    dt = time.perf_counter() - t0
    flops = 2.0 * nrows * w.N * w.K
    desc = (f"{nrows} of {w.M * w.L} output rows of {w.name} "
            f"({flops / 1e9:.1f} GFLOP, {dt:.1f} s, fp64 triple loop)")
    return flops / dt / 1e12, cores, desc, dt


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
    status = g.query_status()
    if status != gemm_ws.OK:
        raise RuntimeError(f"device status after timing: {gemm_ws.status_string(status)}")
    tflops_rank = w.flops / (ms * 1e-3) / 1e12
    value = world * w.flops / (ms * 1e-3) / 1e12

    # End to end through the C ABI with host buffers: pinned host inputs are
    # copied in and D is read back inside every timed step.
    Ah, Bh, Ch = A.pin_memory(), B.pin_memory(), C.pin_memory()
    Dh = torch.empty(D.shape, dtype=D.dtype).pin_memory()

    def e2e_step():
        Ad.copy_(Ah, non_blocking=True)
        Bd.copy_(Bh, non_blocking=True)
        Cd.copy_(Ch, non_blocking=True)
        g.run(Ad, Bd, Cd, D, w.alpha, w.beta)
        Dh.copy_(D, non_blocking=True)

    for _ in range(max(1, args.warmup)):
        e2e_step()
    e2e_steps = max(3, min(args.steps, 20))
    barrier(world)
    e2e_ms = max_over_ranks(time_launches(e2e_step, e2e_steps, stream), world)
    h2d = sum(t.numel() * t.element_size() for t in (Ah, Bh, Ch))
    d2h = Dh.numel() * Dh.element_size()

    # Stream-out overhead: same inputs, interleaved plain / stream-out runs.
    so = workloads.WORKLOADS[workloads.STREAMOUT]
    del Ah, Bh, Ch, Dh, Ad, Bd, Cd, D
    torch.cuda.empty_cache()
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
    g.close()

    if rank != 0:
        return
    peaks, peak_src = load_peaks()
    peak = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    cpu = None
    if not args.no_cpu_baseline:
        v, cores, desc, _ = oracle_sample(w, args.cpu_budget)
        cpu = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc}
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
        "streamout_overhead_pct": round(overhead, 2),
        "streamout": {"workload": so.name, "plain_ms_median": round(mp, 4),
                      "streamout_ms_median": round(ms_so, 4), "reps": len(t_plain),
                      "plain_tflops": round(so.flops / (mp * 1e-3) / 1e12, 2)},
        "e2e": {"value": round(world * w.flops / (e2e_ms * 1e-3) / 1e12, 2), "unit": UNIT,
                "ms_per_step": round(e2e_ms, 4),
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": args.steps,
        "roofline": {"bound": "tensor", "achieved": round(tflops_rank, 2), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(tflops_rank / peak, 4),
                     "peak_source": f"{peak_src} bf16 burst (cuBLAS 8192^3)",
                     "traffic": traffic_for(w.name),
                     "algorithmic_bytes_per_launch": w.algorithmic_bytes(),
                     "kernel": "gws::gemm_ws_kernel"},
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
    w = workloads.WORKLOADS[args.workload or workloads.HEADLINE]
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


def run_reference(args, rank, world, local):
    """The reference arm: the CPU oracle, timed on this host's cores."""
    if rank != 0:
        return
    w = workloads.WORKLOADS[workloads.HEADLINE]
    per_step = max(1.0, args.cpu_budget / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_sample(w, per_step)
    vals, secs = [], 0.0
    desc, cores = "", 0
    for _ in range(args.steps):
        v, cores, desc, dt = oracle_sample(w, per_step)
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
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-budget", type=float, default=15.0,
                    help="seconds of CPU oracle work for the baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--overhead-reps", type=int, default=30)
    ap.add_argument("--kernel-only", action="store_true",
                    help="launch only the GEMM of --workload (for profilers); no contract line")
    ap.add_argument("--workload", choices=sorted(workloads.WORKLOADS), default=None)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world, local)
        return
    if args.kernel_only:
        run_kernel_only(args, local)
        return
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    try:
        run_ours(args, rank, world, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
