"""CPU checks of the C ABI: the libraries build for sm_103a, load, and export
every function that include/*.h declares; host-side argument validation that
needs no GPU (null pointers, bad counts, size queries)."""
import ctypes
import os
import re

import pytest

from tests.gpu_util import ensure_built

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions(header):
    text = open(os.path.join(ROOT, "include", header)).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def libs():
    ensure_built()
    route = ctypes.CDLL(os.path.join(ROOT, "quantized_moe_expert_route_gb300", "libmoe_route.so"))
    synth_lib = ctypes.CDLL(os.path.join(ROOT, "synth", "libmoe_synth.so"))
    return route, synth_lib


def test_exports_every_declared_function(libs):
    route, synth_lib = libs
    names = declared_functions("moe_route.h")
    assert len(names) >= 10
    for n in names:
        assert hasattr(route, n), n
    for n in declared_functions("moe_synth.h"):
        assert hasattr(synth_lib, n), n
    import quantized_moe_expert_route_gb300 as M
    assert sorted(M.EXPORTED) == sorted(n for n in names)


def test_host_validation_without_gpu(libs):
    route, _ = libs
    route.moe_strerror.restype = ctypes.c_char_p
    assert route.moe_strerror(5) == b"workspace too small"
    route.moe_table_device_bytes.restype = ctypes.c_size_t
    assert route.moe_table_device_bytes(0) == 0
    assert route.moe_table_device_bytes(1025) == 0
    assert route.moe_table_device_bytes(512) >= 512 * 72
    route.moe_ffn_forward.restype = ctypes.c_int
    assert route.moe_ffn_forward(None, None, None, 1, 1, None, None, None, 0, None) == 1
    route.moe_route_topk.restype = ctypes.c_int
    # k > E and k = 0 are rejected on the host before any launch
    assert route.moe_route_topk(None, 1, 4, 5, 1, None, None, None, None) == 1
    assert route.moe_route_topk(None, 1, 4, 0, 1, None, None, None, None) == 1
    assert route.moe_route_topk(None, 1, 2048, 4, 1, None, None, None, None) == 8
    route.moe_bucket.restype = ctypes.c_int
    assert route.moe_bucket(None, 1, 0, 4, 0, 4, None, None, None, None, None, None) == 1
    # the path and GEMV-kernel queries refuse a missing table on the host
    route.moe_ffn_path.restype = ctypes.c_int
    assert route.moe_ffn_path(None, 1, 1, None) == -1
    route.moe_ffn_gemv_kernels.restype = ctypes.c_int
    assert route.moe_ffn_gemv_kernels(None, 1, 1) == -1
