"""ctypes binding of libmegamoe.so (include/megamoe.h): same names, argument
marshalling only.  Every step of the layer runs in the library's CUDA
kernels; there is no Python or CPU fallback -- if the library is missing the
import fails loudly.

Pointers are passed as Python ints (``tensor.data_ptr()``) and streams as
``torch.cuda.Stream.cuda_stream`` ints.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmegamoe.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_CAPACITY = 3
MOE_ERR_NOT_BOUND = 4
MOE_ERR_CUDA = 5
MOE_ERR_BAD_ROUTE = 6
MOE_ERR_DEVICE_TIMEOUT = 7
MOE_ERR_BAD_SCALE = 8
MOE_ERR_WORKSPACE = 9

MOE_DEV_ROUTE_RANGE = 0x01
MOE_DEV_ROUTE_DUP = 0x02
MOE_DEV_ROUTE_NONFINITE = 0x04
MOE_DEV_CAPACITY = 0x08
MOE_DEV_TIMEOUT = 0x10
MOE_DEV_BAD_SCALE = 0x20

MOE_FLAG_FUSE_FC1_EPILOGUE = 0x1
MOE_FLAG_CHECK_ROUTES = 0x2
MOE_FLAG_EMIT_FC1 = 0x4
MOE_FLAG_GEMM_SINGLE_CTA = 0x8
MOE_FLAG_GEMM_CTA_PAIR = 0x10
MOE_FLAG_WATCHDOG_TEST = 0x20
MOE_FLAG_SPLIT_GEMMS = 0x40
MOE_FLAG_GEMMS_ONE_LAUNCH = 0x80
MOE_FLAG_MXFP8 = 0x100
MOE_FLAG_WATCHDOG_ROUTE_TEST = 0x200
MOE_FLAG_PER_TENSOR = 0x400
MOE_FLAG_NO_SWAP_AB = 0x800
MOE_FLAG_COMBINE_IN_FC2 = 0x1000

# every function the header declares (checked against include/megamoe.h by a test)
API_NAMES = ("moe_workspace_query", "moe_create", "moe_quantize_weights", "moe_quantize_weights_mx",
             "moe_quantize_weights_pt", "moe_requantize_weights_nvfp4", "moe_bind_weights",
             "moe_set_activation_scales",
             "moe_stage_inputs", "moe_forward", "moe_read_status", "moe_debug_views",
             "moe_set_profile_events", "moe_set_sm_budget", "moe_forward_plan", "moe_route_noalloc",
             "moe_destroy", "moe_status_str")


class moe_dims(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("inter", ctypes.c_int32),
                ("num_experts", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("flags", ctypes.c_uint32)]


class moe_debug_view(ctypes.Structure):
    _fields_ = [("status", ctypes.c_void_p), ("counts", ctypes.c_void_p),
                ("offsets", ctypes.c_void_p), ("pad_offsets", ctypes.c_void_p),
                ("perm", ctypes.c_void_p), ("inv", ctypes.c_void_p), ("inv_pad", ctypes.c_void_p),
                ("a", ctypes.c_void_p), ("a_sf", ctypes.c_void_p), ("gu", ctypes.c_void_p),
                ("hq", ctypes.c_void_p), ("h_sf", ctypes.c_void_p), ("y", ctypes.c_void_p),
                ("rows_alloc", ctypes.c_int64), ("sf_atom_bytes", ctypes.c_int32),
                ("gemm_pair", ctypes.c_int32), ("gemm_ctas", ctypes.c_int32),
                ("pad_rows", ctypes.c_int32), ("route_coop_blocks", ctypes.c_int32)]


class moe_plan(ctypes.Structure):
    _fields_ = [("route_kernels", ctypes.c_int32), ("gemm_launches", ctypes.c_int32),
                ("swiglu_kernels", ctypes.c_int32), ("kernels", ctypes.c_int32),
                ("swap_ab_tokens", ctypes.c_int32), ("combine_in_fc2", ctypes.c_int32)]


class MoEError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_str(status)} ({status})")


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is not built: run __graft_entry__.build() "
                              "(there is no CPU fallback)")
        L = ctypes.CDLL(LIB_PATH)
        vp, i64, i32, st = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int
        L.moe_workspace_query.argtypes = [ctypes.POINTER(moe_dims), i64, i64, ctypes.c_float,
                                          ctypes.POINTER(ctypes.c_size_t),
                                          ctypes.POINTER(ctypes.c_size_t)]
        L.moe_create.argtypes = [ctypes.POINTER(moe_dims), i64, i64, ctypes.c_float, vp,
                                 ctypes.c_size_t, vp, ctypes.c_size_t, ctypes.POINTER(vp)]
        L.moe_quantize_weights.argtypes = [vp, i64, i32, i32, vp, vp, vp]
        L.moe_quantize_weights_mx.argtypes = [vp, i64, i32, i32, vp, vp, vp]
        L.moe_quantize_weights_pt.argtypes = [vp, i64, i32, i32, vp, vp, vp]
        L.moe_requantize_weights_nvfp4.argtypes = [vp, vp, vp, i64, i32, i32, vp, vp, vp]
        L.moe_set_activation_scales.argtypes = [vp, ctypes.c_float, ctypes.c_float, vp]
        L.moe_bind_weights.argtypes = [vp, vp, vp, vp, vp, vp]
        L.moe_stage_inputs.argtypes = [vp, vp]
        L.moe_forward.argtypes = [vp, vp, vp, vp, i64, vp]
        L.moe_read_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32), vp]
        L.moe_debug_views.argtypes = [vp, ctypes.POINTER(moe_debug_view)]
        L.moe_set_profile_events.argtypes = [vp, ctypes.POINTER(vp), i32]
        L.moe_set_sm_budget.argtypes = [vp, i32]
        L.moe_forward_plan.argtypes = [vp, i64, ctypes.POINTER(moe_plan)]
        L.moe_route_noalloc.argtypes = [vp, vp, i64, i32, i32, i32, vp, vp, vp, vp, vp, vp]
        L.moe_destroy.argtypes = [vp]
        L.moe_destroy.restype = None
        L.moe_status_str.argtypes = [st]
        L.moe_status_str.restype = ctypes.c_char_p
        for n in API_NAMES:
            if n not in ("moe_destroy", "moe_status_str"):
                getattr(L, n).restype = st
        _lib = L
    return _lib


def status_str(s: int) -> str:
    return lib().moe_status_str(s).decode()


def _check(s: int, where: str) -> None:
    if s != MOE_OK:
        raise MoEError(s, where)


def _dims(H: int, I: int, E: int, K: int, flags: int) -> moe_dims:
    return moe_dims(H, I, E, K, flags)


def moe_workspace_query(H, I, E, K, flags, expected_m, max_rows, capacity_factor=1.0):
    ws, w = ctypes.c_size_t(), ctypes.c_size_t()
    d = _dims(H, I, E, K, flags)
    _check(lib().moe_workspace_query(ctypes.byref(d), expected_m, max_rows, capacity_factor,
                                     ctypes.byref(ws), ctypes.byref(w)), "moe_workspace_query")
    return ws.value, w.value


def moe_create(H, I, E, K, flags, expected_m, max_rows, capacity_factor, d_ws, ws_bytes, d_w,
               w_bytes) -> int:
    h = ctypes.c_void_p()
    d = _dims(H, I, E, K, flags)
    _check(lib().moe_create(ctypes.byref(d), expected_m, max_rows, capacity_factor, d_ws, ws_bytes,
                            d_w, w_bytes, ctypes.byref(h)), "moe_create")
    return h.value


def moe_quantize_weights(d_w, num_mats, rows, cols, d_q, d_scale, stream) -> None:
    _check(lib().moe_quantize_weights(d_w, num_mats, rows, cols, d_q, d_scale, stream),
           "moe_quantize_weights")


def moe_quantize_weights_mx(d_w, num_mats, rows, cols, d_q, d_scale, stream) -> None:
    _check(lib().moe_quantize_weights_mx(d_w, num_mats, rows, cols, d_q, d_scale, stream),
           "moe_quantize_weights_mx")


def moe_quantize_weights_pt(d_w, num_mats, rows, cols, d_q, d_scale, stream) -> None:
    _check(lib().moe_quantize_weights_pt(d_w, num_mats, rows, cols, d_q, d_scale, stream),
           "moe_quantize_weights_pt")


def moe_requantize_weights_nvfp4(d_codes, d_block_scales, d_global_scales, num_mats, rows, cols, d_q,
                                 d_scale, stream) -> None:
    _check(lib().moe_requantize_weights_nvfp4(d_codes, d_block_scales, d_global_scales, num_mats, rows,
                                              cols, d_q, d_scale, stream),
           "moe_requantize_weights_nvfp4")


def moe_set_activation_scales(h, x_scale, h_scale, stream) -> None:
    _check(lib().moe_set_activation_scales(h, x_scale, h_scale, stream),
           "moe_set_activation_scales")


def moe_bind_weights(h, d_w1, d_w1s, d_w2, d_w2s, stream) -> None:
    _check(lib().moe_bind_weights(h, d_w1, d_w1s, d_w2, d_w2s, stream), "moe_bind_weights")


def moe_stage_inputs(h, d_out) -> None:
    _check(lib().moe_stage_inputs(h, d_out), "moe_stage_inputs")


def moe_forward(h, d_x, d_idx, d_w, num_tokens, stream) -> None:
    _check(lib().moe_forward(h, d_x, d_idx, d_w, num_tokens, stream), "moe_forward")


def moe_forward_status(h, d_x, d_idx, d_w, num_tokens, stream) -> int:
    """moe_forward returning the host status instead of raising."""
    return lib().moe_forward(h, d_x, d_idx, d_w, num_tokens, stream)


def moe_read_status(h, stream):
    """(status code, device status bits)"""
    bits = ctypes.c_uint32()
    s = lib().moe_read_status(h, ctypes.byref(bits), stream)
    return s, bits.value


def moe_debug_views(h) -> moe_debug_view:
    v = moe_debug_view()
    _check(lib().moe_debug_views(h, ctypes.byref(v)), "moe_debug_views")
    return v


def moe_set_profile_events(h, event_handles) -> None:
    n = len(event_handles)
    arr = (ctypes.c_void_p * max(n, 1))(*event_handles)
    _check(lib().moe_set_profile_events(h, arr, n), "moe_set_profile_events")


def moe_set_sm_budget(h, max_sms) -> None:
    _check(lib().moe_set_sm_budget(h, max_sms), "moe_set_sm_budget")


def moe_forward_plan(h, num_tokens) -> moe_plan:
    p = moe_plan()
    _check(lib().moe_forward_plan(h, num_tokens, ctypes.byref(p)), "moe_forward_plan")
    return p


def moe_route_noalloc(d_idx, d_w, num_tokens, top_k, num_experts, check_routes, d_counts,
                      d_offsets, d_perm, d_inv, d_status, stream) -> int:
    """Routing without any allocation (fixed device scratch); returns the host status."""
    return lib().moe_route_noalloc(d_idx, d_w, num_tokens, top_k, num_experts, check_routes,
                                   d_counts, d_offsets, d_perm, d_inv, d_status, stream)


def moe_destroy(h) -> None:
    if h:
        lib().moe_destroy(h)
