"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every function include/megamoe.h declares, and the pure-host workspace query
applies the documented rules."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def B():
    from serving_route_gb300 import build
    build.build()
    import serving_route_gb300.binding as B
    return B


def header_functions():
    src = open(os.path.join(ROOT, "include", "megamoe.h")).read()
    return sorted(set(re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", src)))


def test_every_declared_symbol_is_exported(B):
    names = header_functions()
    assert len(names) >= 11
    lib = ctypes.CDLL(B.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(B.API_NAMES) == names


def test_header_constants_match_the_binding(B):
    """every #define MOE_* of the header has the same value in the binding"""
    src = open(os.path.join(ROOT, "include", "megamoe.h")).read()
    defs = dict(re.findall(r"#define\s+(MOE_\w+)\s+(0x[0-9a-fA-F]+|\d+)u?\b", src))
    assert len(defs) >= 15 and "MOE_FLAG_WATCHDOG_ROUTE_TEST" in defs
    for name, val in defs.items():
        assert getattr(B, name) == int(val, 0), name


def test_status_strings(B):
    assert B.status_str(B.MOE_OK) == "ok"
    assert "capacity" in B.status_str(B.MOE_ERR_CAPACITY)


@pytest.mark.parametrize("H,I,E,K,ok", [
    (7168, 2048, 256, 8, B_OK := 0), (512, 256, 8, 2, 0), (2048, 1408, 64, 6, 0),
    (100, 256, 8, 2, 2), (512, 200, 8, 2, 2), (512, 256, 8, 3, 2), (512, 256, 8, 10, 2),
    (512, 256, 0, 2, 2), (32768, 256, 8, 2, 2), (512, 256, 2048, 2, 2)])
def test_workspace_query_rules(B, H, I, E, K, ok):
    if ok == 0:
        ws, w = B.moe_workspace_query(H, I, E, K, 0, 1, 128)
        assert w >= E * 3 * H * I and ws > 0
    else:
        with pytest.raises(B.MoEError) as e:
            B.moe_workspace_query(H, I, E, K, 0, 1, 128)
        assert e.value.status == ok


def test_workspace_query_capacity_and_tactic(B):
    a = B.moe_workspace_query(7168, 2048, 256, 8, 0, 1, 8192, 1.0)
    b = B.moe_workspace_query(7168, 2048, 256, 8, 0, 8192, 8192, 1.0)
    assert a == b                              # expected_m never changes a buffer size
    c = B.moe_workspace_query(7168, 2048, 256, 8, 0, 1, 8192, 0.5)
    assert c[0] < a[0] and c[1] == a[1]        # capacity bounds the GEMM buffers only
    fused = B.moe_workspace_query(7168, 2048, 256, 8, B.MOE_FLAG_FUSE_FC1_EPILOGUE, 1, 8192)
    assert fused[0] < a[0]                     # no BF16 gate||up buffer when fused
    for bad in ((0, 128, 1.0), (1, 0, 1.0), (1, 128, 0.0), (1, 128, -1.0), (1, 128, 100.0)):
        with pytest.raises(B.MoEError):
            B.moe_workspace_query(512, 256, 8, 2, 0, *bad)
    # one or two GEMM launches: the forcing flags exclude each other, and
    # neither changes a buffer size
    f = B.MOE_FLAG_FUSE_FC1_EPILOGUE
    assert B.moe_workspace_query(7168, 2048, 256, 8, f | B.MOE_FLAG_SPLIT_GEMMS, 1, 8192) == fused
    assert B.moe_workspace_query(7168, 2048, 256, 8, f | B.MOE_FLAG_GEMMS_ONE_LAUNCH, 1, 8192) == fused
    with pytest.raises(B.MoEError):
        B.moe_workspace_query(512, 256, 8, 2, f | B.MOE_FLAG_SPLIT_GEMMS | B.MOE_FLAG_GEMMS_ONE_LAUNCH,
                              1, 128)
    # MXFP8 keeps one scale atom per K block instead of per four: larger
    # workspace and weight store, same for every other buffer
    mx = B.moe_workspace_query(7168, 2048, 256, 8, f | B.MOE_FLAG_MXFP8, 1, 8192)
    assert mx[0] > fused[0] and mx[1] > fused[1]


def test_null_arguments_rejected_without_cuda(B):
    L = B.lib()
    assert L.moe_workspace_query(None, 1, 1, 1.0, None, None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_stage_inputs(None, None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_forward(None, None, None, None, 1, None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_debug_views(None, None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_forward_plan(None, 1, None) == B.MOE_ERR_INVALID_ARG


def test_gemm_source_hash_ignores_comments_only():
    """bench.py keeps a recorded DRAM-traffic figure only while the GEMM code is
    unchanged; comments and whitespace do not count as code."""
    import bench
    a = 'int f(int x) { return x + 1; } // note\n/* block\n comment */ const char* s = "a // b";'
    b = 'int f(int x)  {\n  return x + 1;\n}\nconst char* s = "a // b";  // other note'
    c = 'int f(int x) { return x + 2; } const char* s = "a // b";'
    assert bench.strip_c_comments(a) == bench.strip_c_comments(b)
    assert bench.strip_c_comments(a) != bench.strip_c_comments(c)
    assert '"a // b"' in bench.strip_c_comments(a)
