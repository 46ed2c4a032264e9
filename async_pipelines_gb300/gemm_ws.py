"""Python binding of the C ABI in include/gemm_ws.h (argument marshalling only).

Every step of the GEMM runs in the CUDA library; this module passes tensor
pointers, sizes and the current CUDA stream through ctypes. PyTorch provides
device memory and streams. There is no fallback: if the library is missing or
the device is not a GB300, the calls raise.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import build as _build

OK = 0
ERR_INVALID_ARG = 1
ERR_ALIGNMENT = 2
ERR_UNSUPPORTED = 3
ERR_CUDA = 4
ERR_TIMEOUT = 5

EXPORTS = (
    "gemm_ws_create", "gemm_ws_destroy", "gemm_ws_run", "gemm_ws_run_streamout",
    "gemm_ws_query_status", "gemm_ws_last_cuda_error", "gemm_ws_status_string",
    "gemm_ws_streamout_tiles", "gemm_ws_run_streamout_noalloc", "gemm_ws_kernels_per_run",
)

STAGING_TILE = 128

_lib = None


class GemmWSError(RuntimeError):
    def __init__(self, status: int, what: str, cuda_error: int = 0):
        self.status = status
        self.cuda_error = cuda_error
        msg = f"{what}: {status_string(status)} (status {status})"
        if cuda_error:
            msg += f", CUDA error {cuda_error}"
        super().__init__(msg)


def library_path() -> str:
    return _build.LIB


def load_library(path: Optional[str] = None):
    """Loads the CUDA library. Raises if it has not been built."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or library_path()
    if not os.path.exists(p):
        raise RuntimeError(
            f"gemm_ws CUDA library not found at {p}; build it with "
            "`python -m async_pipelines_gb300.build` (needs nvcc)")
    lib = ctypes.CDLL(p)
    vp, i64, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float
    lib.gemm_ws_create.argtypes = [ctypes.POINTER(vp), ctypes.c_int]
    lib.gemm_ws_destroy.argtypes = [vp]
    lib.gemm_ws_run.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, f32, f32, vp]
    lib.gemm_ws_run_streamout.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, f32, f32,
                                          vp, vp, vp]
    lib.gemm_ws_run_streamout_noalloc.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, f32, f32,
                                                  vp, vp, vp]
    lib.gemm_ws_query_status.argtypes = [vp, vp]
    lib.gemm_ws_last_cuda_error.argtypes = [vp]
    lib.gemm_ws_status_string.argtypes = [ctypes.c_int]
    lib.gemm_ws_status_string.restype = ctypes.c_char_p
    lib.gemm_ws_streamout_tiles.argtypes = [i64, i64, i64]
    lib.gemm_ws_streamout_tiles.restype = i64
    lib.gemm_ws_kernels_per_run.argtypes = [vp, i64, i64, i64, i64, ctypes.c_int]
    lib.gemm_ws_kernels_per_run.restype = ctypes.c_int
    for name in ("gemm_ws_create", "gemm_ws_destroy", "gemm_ws_run", "gemm_ws_run_streamout",
                 "gemm_ws_query_status", "gemm_ws_last_cuda_error",
                 "gemm_ws_run_streamout_noalloc"):
        getattr(lib, name).restype = ctypes.c_int
    if path is None:
        _lib = lib
    return lib


DEBUG_EXPORTS = ("gemm_ws_debug_configure", "gemm_ws_debug_launch_shape",
                 "gemm_ws_debug_schedule", "gemm_ws_debug_phases",
                 "gemm_ws_debug_noalloc_configure")

_debug_lib = None


def load_debug_library():
    """The debug build (test hooks of include/gemm_ws_debug.h). Tests only."""
    global _debug_lib
    if _debug_lib is None:
        lib = load_library(_build.DEBUG_LIB)
        lib.gemm_ws_debug_configure.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]
        lib.gemm_ws_debug_configure.restype = ctypes.c_int
        ip = ctypes.POINTER(ctypes.c_int)
        lib.gemm_ws_debug_launch_shape.argtypes = [ctypes.c_void_p, ctypes.c_int64,
                                                   ctypes.c_int64, ctypes.c_int64,
                                                   ctypes.c_int64, ctypes.c_int, ip, ip, ip, ip, ip, ip]
        lib.gemm_ws_debug_launch_shape.restype = ctypes.c_int
        i64 = ctypes.c_int64
        lib.gemm_ws_debug_schedule.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_int, i64, i64, i64, i64,
                                               ctypes.c_int, ctypes.c_void_p, i64,
                                               ctypes.POINTER(i64), ip]
        lib.gemm_ws_debug_schedule.restype = ctypes.c_int
        lib.gemm_ws_debug_phases.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
        lib.gemm_ws_debug_phases.restype = ctypes.c_int
        lib.gemm_ws_debug_noalloc_configure.argtypes = [ctypes.c_int, ctypes.c_int,
                                                        ctypes.c_longlong]
        lib.gemm_ws_debug_noalloc_configure.restype = ctypes.c_int
        _debug_lib = lib
    return _debug_lib


def status_string(status: int) -> str:
    return load_library().gemm_ws_status_string(int(status)).decode()


def gemm_ws_streamout_tiles(M: int, N: int, L: int) -> int:
    return int(load_library().gemm_ws_streamout_tiles(M, N, L))


# ------------------------------------------------------------------ C-ABI names

def gemm_ws_create(device: int = 0) -> ctypes.c_void_p:
    h = ctypes.c_void_p()
    rc = load_library().gemm_ws_create(ctypes.byref(h), int(device))
    if rc != OK:
        raise GemmWSError(rc, "gemm_ws_create")
    return h


def gemm_ws_destroy(h) -> None:
    load_library().gemm_ws_destroy(h)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream) -> int:
    """The raw cudaStream_t of `stream` (default: the current torch stream)."""
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def gemm_ws_run(h, A, B, C, D, M, N, K, L, alpha, beta, stream=None) -> int:
    """Raw call: tensors (or None for C) passed as device pointers. Returns the status."""
    return load_library().gemm_ws_run(h, _ptr(A), _ptr(B), _ptr(C), _ptr(D), M, N, K, L,
                                      float(alpha), float(beta), _stream(stream))


def gemm_ws_run_streamout(h, A, B, C, D, M, N, K, L, alpha, beta, staging, flags,
                          stream=None) -> int:
    return load_library().gemm_ws_run_streamout(
        h, _ptr(A), _ptr(B), _ptr(C), _ptr(D), M, N, K, L, float(alpha), float(beta),
        _ptr(staging), _ptr(flags), _stream(stream))


def gemm_ws_run_streamout_noalloc(A, B, C, D, M, N, K, L, alpha, beta, staging, flags,
                                  stream=None) -> int:
    """Stream-out GEMM on the current device with no handle and no device
    allocation (its scratch is a fixed array inside the library)."""
    return load_library().gemm_ws_run_streamout_noalloc(
        _ptr(A), _ptr(B), _ptr(C), _ptr(D), M, N, K, L, float(alpha), float(beta),
        _ptr(staging), _ptr(flags), _stream(stream))


def gemm_ws_query_status(h, stream=None) -> int:
    return load_library().gemm_ws_query_status(h, _stream(stream))


def gemm_ws_last_cuda_error(h) -> int:
    return load_library().gemm_ws_last_cuda_error(h)


# ------------------------------------------------------------------ tensor API

_BF16 = torch.bfloat16


def _check_operands(A, B, C, D):
    for t in (A, B, D) if C is None else (A, B, C, D):
        if t.dtype is not _BF16 or not t.is_cuda or not t.is_contiguous():
            raise ValueError("A, B, C and D must be contiguous bf16 CUDA tensors")
    if A.dim() != 3 or B.dim() != 3 or D.dim() != 3:
        raise ValueError("A (L,M,K), B (L,N,K) and D (L,M,N) must be 3-D")
    L, M, K = A.shape
    if B.shape[0] != L or B.shape[2] != K:
        raise ValueError("B must be (L, N, K)")
    N = B.shape[1]
    if tuple(D.shape) != (L, M, N) or (C is not None and tuple(C.shape) != (L, M, N)):
        raise ValueError("C and D must be (L, M, N)")
    return M, N, K, L


class GemmWS:
    """Owns one library handle on one CUDA device.

    `lib` selects the loaded library (default: the production build; tests
    pass the debug build from `load_debug_library()`)."""

    def __init__(self, device: int = 0, lib=None):
        self.device = int(device)
        self.lib = lib or load_library()
        h = ctypes.c_void_p()
        rc = self.lib.gemm_ws_create(ctypes.byref(h), self.device)
        if rc != OK:
            raise GemmWSError(rc, "gemm_ws_create")
        self.handle = h

    def close(self):
        if self.handle is not None:
            self.lib.gemm_ws_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _raise(self, rc, what):
        if rc != OK:
            raise GemmWSError(rc, what, self.lib.gemm_ws_last_cuda_error(self.handle))

    def run(self, A, B, C, D, alpha=1.0, beta=0.0, stream=None):
        """D = alpha * A @ B^T-stored + beta * C on the current (or given) stream.

        A: (L, M, K), B: (L, N, K) (column-major K x N per batch), C/D: (L, M, N).
        """
        M, N, K, L = _check_operands(A, B, C, D)
        rc = self.lib.gemm_ws_run(self.handle, A.data_ptr(), B.data_ptr(),
                                  None if C is None else C.data_ptr(), D.data_ptr(), M, N, K, L,
                                  alpha, beta, _stream_handle(stream))
        if rc != OK:
            self._raise(rc, "gemm_ws_run")
        return D

    def run_streamout(self, A, B, C, D, staging, flags, alpha=1.0, beta=0.0, stream=None):
        M, N, K, L = _check_operands(A, B, C, D)
        T = gemm_ws_streamout_tiles(M, N, L)
        if staging.dtype != torch.bfloat16 or staging.numel() < T * STAGING_TILE ** 2:
            raise ValueError(f"staging must be bf16 with >= {T} * 128 * 128 elements")
        if flags.dtype != torch.int32 or flags.numel() < 2 * T:
            raise ValueError(f"flags must be int32 (read as uint32) with >= {2 * T} elements")
        rc = self.lib.gemm_ws_run_streamout(self.handle, _ptr(A), _ptr(B), _ptr(C), _ptr(D), M,
                                            N, K, L, float(alpha), float(beta), _ptr(staging),
                                            _ptr(flags), _stream(stream))
        self._raise(rc, "gemm_ws_run_streamout")
        return D

    def query_status(self, stream=None) -> int:
        return self.lib.gemm_ws_query_status(self.handle, _stream(stream))

    def kernels_per_run(self, M, N, K, L, streamout=False) -> int:
        """Kernels one run of this problem launches (1, or 2 with split pieces)."""
        n = self.lib.gemm_ws_kernels_per_run(self.handle, M, N, K, L, int(bool(streamout)))
        if n < 0:
            raise GemmWSError(-n, "gemm_ws_kernels_per_run")
        return n
