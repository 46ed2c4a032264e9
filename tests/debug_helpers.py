"""Debug-build plumbing for the watchdog and overlap tests."""
from __future__ import annotations

import contextlib
import ctypes
import os

from async_pipelines_gb300 import gemm_ws


@contextlib.contextmanager
def env(**kv):
    old = {k: os.environ.get(k) for k in kv}
    os.environ.update({k: str(v) for k, v in kv.items()})
    try:
        yield
    finally:
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


def debug_handle(cta_group: int = 2, timeout_ms: int = 1000) -> gemm_ws.GemmWS:
    """A handle on the debug build, created with the given tile configuration
    (CTA group) and per-wait watchdog limit."""
    lib = gemm_ws.load_debug_library()
    with env(GEMM_WS_CTA_GROUP=cta_group, GEMM_WS_TIMEOUT_MS=timeout_ms):
        return gemm_ws.GemmWS(0, lib=lib)


def launch_shape(g: gemm_ws.GemmWS, M: int, N: int, K: int, L: int, streamout: bool = True):
    """(CTAs per cluster, clusters, unit-id bound, stream-K tiles) of the handle's launch."""
    cg, cl, nu, ks = ctypes.c_int(), ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    rc = g.lib.gemm_ws_debug_launch_shape(g.handle, M, N, K, L, int(streamout), ctypes.byref(cg),
                                          ctypes.byref(cl), ctypes.byref(nu), ctypes.byref(ks),
                                          None, None)
    assert rc == gemm_ws.OK
    return cg.value, cl.value, nu.value, ks.value


def split_plan(g: gemm_ws.GemmWS, M: int, N: int, K: int, L: int):
    """(pieces per split tile, 1 if the GEMM kernel adds them itself / 0 if
    the reduction kernel does) of the handle's gemm_ws_run launch."""
    cg, cl, nu, ks, sp, si = (ctypes.c_int() for _ in range(6))
    rc = g.lib.gemm_ws_debug_launch_shape(g.handle, M, N, K, L, 0, ctypes.byref(cg),
                                          ctypes.byref(cl), ctypes.byref(nu), ctypes.byref(ks),
                                          ctypes.byref(sp), ctypes.byref(si))
    assert rc == gemm_ws.OK
    return sp.value, si.value


def configure(g: gemm_ws.GemmWS, fault: int, trace_ptr=None):
    rc = g.lib.gemm_ws_debug_configure(g.handle, fault,
                                       None if trace_ptr is None else ctypes.c_void_p(trace_ptr))
    assert rc == gemm_ws.OK
