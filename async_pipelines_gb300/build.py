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
SOURCES = [os.path.join(CSRC, "gemm_ws.cu")]
DEPS = SOURCES + [os.path.join(CSRC, f) for f in ("ptx.cuh", "gemm_ws_kernel.cuh")] + [
    os.path.join(INCLUDE, "gemm_ws.h")]

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


def build(out: str = LIB, extra=(), verbose: bool = False) -> str:
    cmd = [nvcc(), ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
           f"-I{INCLUDE}", "-o", out, *extra, *SOURCES]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.run(cmd, check=True)
    return out


def ensure_built() -> str:
    if stale():
        build()
    return LIB


if __name__ == "__main__":
    build(verbose=True)
    print(LIB)
