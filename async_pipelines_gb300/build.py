"""Builds the CUDA library in-tree with nvcc for sm_103a (GB300).

One translation unit, one -gencode; the shared library links the CUDA
runtime statically and reaches the driver's tensor-map encoder through the
runtime's driver-entry-point query, so it needs no libcuda at link time.
"""
from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libgemm_ws.so")
# Debug build: the same sources with the test hooks of include/gemm_ws_debug.h
# (fault injection for the watchdog, per-tile timestamps). Tests only.
DEBUG_LIB = os.path.join(PKG, "libgemm_ws_debug.so")
SOURCES = [os.path.join(CSRC, "gemm_ws.cu")]
DEPS = SOURCES + [os.path.join(CSRC, f) for f in ("ptx.cuh", "gemm_ws_kernel.cuh")] + [
    os.path.join(INCLUDE, "gemm_ws.h"), os.path.join(INCLUDE, "gemm_ws_debug.h")]

ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")


def stale(out: str = LIB) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in DEPS if os.path.exists(d))


def _cmd(out: str, extra=(), verbose: bool = False):
    cmd = [nvcc(), ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
           f"-I{INCLUDE}", "-o", out, *extra, *SOURCES]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    return cmd


def build(out: str = LIB, extra=(), verbose: bool = False, debug: bool = True) -> str:
    """Builds the production library (and, by default, the debug library) in
    parallel nvcc processes."""
    procs = [subprocess.Popen(_cmd(out, extra, verbose))]
    if debug:
        procs.append(subprocess.Popen(_cmd(DEBUG_LIB, ("-DGEMM_WS_DEBUG", *extra))))
    codes = [p.wait() for p in procs]
    if any(codes):
        raise subprocess.CalledProcessError(max(codes), "nvcc")
    return out


def ensure_built() -> str:
    if stale() or stale(DEBUG_LIB):
        build()
    return LIB


if __name__ == "__main__":
    build(verbose=True)
    print(LIB)
