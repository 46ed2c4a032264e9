"""CPU checks of the C ABI boundary: the library builds, loads and exports
every function that include/gemm_ws.h declares; pure-host entry points work
without a GPU; and the product package never reaches for the oracle."""
from __future__ import annotations

import ast
import os
import re

import pytest
import torch

from async_pipelines_gb300 import build, gemm_ws

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gemm_ws.h")


DEBUG_HEADER = os.path.join(ROOT, "include", "gemm_ws_debug.h")


def declared_functions(header=HEADER):
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gemm_ws_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    build.ensure_built()
    return gemm_ws.load_library()


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("gemm_ws_create", "gemm_ws_run", "gemm_ws_run_streamout",
                     "gemm_ws_destroy"):
        assert required in names


def test_library_exports_every_declared_function(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in gemm_ws.h but not exported"
    assert set(declared_functions()) == set(gemm_ws.EXPORTS)


def test_debug_hooks_only_in_the_debug_build(lib):
    import ctypes
    dbg = ctypes.CDLL(build.DEBUG_LIB)
    debug_names = [n for n in declared_functions(DEBUG_HEADER) if n.startswith("gemm_ws_debug")]
    assert set(debug_names) == set(gemm_ws.DEBUG_EXPORTS)
    for name in declared_functions() + debug_names:
        assert hasattr(dbg, name), name
    for name in debug_names:
        assert not hasattr(lib, name), f"{name} leaked into the production library"


def test_streamout_tile_count_is_host_arithmetic(lib):
    assert gemm_ws.gemm_ws_streamout_tiles(256, 256, 1) == 4
    assert gemm_ws.gemm_ws_streamout_tiles(5000, 3000, 4) == 4 * 40 * 24
    assert gemm_ws.gemm_ws_streamout_tiles(8192, 8192, 1) == 4096
    assert gemm_ws.gemm_ws_streamout_tiles(1, 1, 1) == 1
    assert gemm_ws.gemm_ws_streamout_tiles(0, 128, 1) == 0


def test_status_strings(lib):
    assert gemm_ws.status_string(gemm_ws.OK) == "ok"
    assert "timed out" in gemm_ws.status_string(gemm_ws.ERR_TIMEOUT)
    assert gemm_ws.status_string(99) == "unknown status"


def test_null_handle_is_rejected_without_a_gpu(lib):
    assert lib.gemm_ws_run(None, None, None, None, None, 8, 8, 8, 1, 1.0, 0.0, None) == \
        gemm_ws.ERR_INVALID_ARG
    assert lib.gemm_ws_query_status(None, None) == gemm_ws.ERR_INVALID_ARG
    assert lib.gemm_ws_destroy(None) == gemm_ws.OK


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU error path")
def test_create_without_gpu_fails_cleanly(lib):
    with pytest.raises(gemm_ws.GemmWSError):
        gemm_ws.gemm_ws_create(0)


def test_product_package_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "async_pipelines_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            path = os.path.join(dirpath, f)
            if f.endswith(".py"):
                tree = ast.parse(open(path).read())
                for node in ast.walk(tree):
                    if isinstance(node, ast.Import):
                        assert not any(a.name.split(".")[0] == "oracle" for a in node.names), path
                    if isinstance(node, ast.ImportFrom):
                        assert (node.module or "").split(".")[0] != "oracle", path
            if f.endswith((".cu", ".cuh", ".h", ".cpp")):
                assert "gemm_ref" not in open(path).read(), path
