"""CPU oracle of the single-GPU MoE layer forward -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s cpu_baseline and
reference legs may import this package.  The product path (the C-ABI library
and its binding) never imports, links or runs anything here, and shares no code
with it.

The arithmetic lives in ``oracle.c`` (plain C, float64; see its header for
the definition followed, step by step, with citations).  This module only
marshals numpy arrays through ctypes.

Formats: ``fmt=0`` is the DeepSeek layout (1x128 activation, 128x128 weight
scales); ``fmt=1`` is MXFP8 (one scale per 32 elements along K, for
activations and for every weight row); the per-tensor format (one scale per
expert weight matrix, static calibrated activation scales) has its own
functions, ``quant_weights_pt`` and ``forward_pt``.

Parity status per function (pins live in ``tests/test_oracle_*.py``):
  e4m3 encode/decode, bf16 rounding, pow2 scale rule, 1x128 / 128x128 and
  MXFP8 1x32 quantisation, routing, FC1/FC2 block-scaled products in both
  formats, combine, the per-tensor quantisers and products: pinned.
  SwiGLU's exp: parity unpinned at the ulp level (host ``exp`` versus the
  GPU's ``expf``); covered by tolerance only.
  Combine summation order: parity unpinned at the ulp level (float64 here,
  float32 fused multiply-adds on the GPU); covered by tolerance only.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_lib = None

ERR_ROUTE_RANGE = 0x1
ERR_ROUTE_DUP = 0x2
ERR_ROUTE_NONFINITE = 0x4


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        L.or_e4m3_decode.argtypes = [ctypes.c_uint8]
        L.or_e4m3_decode.restype = ctypes.c_double
        L.or_e4m3_encode.argtypes = [ctypes.c_double]
        L.or_e4m3_encode.restype = ctypes.c_uint8
        L.or_bf16_round.argtypes = [ctypes.c_double]
        L.or_bf16_round.restype = ctypes.c_uint16
        L.or_bf16_decode.argtypes = [ctypes.c_uint16]
        L.or_bf16_decode.restype = ctypes.c_double
        L.or_pow2_scale_exp.argtypes = [ctypes.c_double]
        L.or_pow2_scale_exp.restype = ctypes.c_int
        L.or_swiglu.argtypes = [ctypes.c_uint16, ctypes.c_uint16]
        L.or_swiglu.restype = ctypes.c_float
        L.or_quant_rows.argtypes = [vp, i64, i64, vp, vp]
        L.or_quant_rows_bw.argtypes = [vp, i64, i64, i32, vp, vp]
        L.or_quant_rows_bf16.argtypes = [vp, i64, i64, vp, vp]
        L.or_quant_rows_bf16_bw.argtypes = [vp, i64, i64, i32, vp, vp]
        L.or_quant_weights.argtypes = [vp, i64, i64, i64, vp, vp]
        L.or_quant_weights_mx.argtypes = [vp, i64, i64, i64, vp, vp]
        L.or_e2m1_decode.argtypes = [ctypes.c_uint8]
        L.or_e2m1_decode.restype = ctypes.c_double
        L.or_dequant_nvfp4.argtypes = [vp, vp, vp, i64, i64, i64, vp]
        L.or_route.argtypes = [i64, i32, i32, vp, vp, i32, vp, vp, vp, vp]
        L.or_route.restype = ctypes.c_uint32
        L.or_expert_ffn.argtypes = [i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        L.or_expert_ffn_fmt.argtypes = [i32] + L.or_expert_ffn.argtypes
        L.or_combine.argtypes = [i64, i32, i32, vp, vp, vp, vp, vp]
        L.or_forward.argtypes = [i64, i32, i32, i32, i32, i32] + [vp] * 7 + [vp] * 13
        L.or_forward.restype = ctypes.c_uint32
        L.or_forward_fmt.argtypes = [i32] + L.or_forward.argtypes
        L.or_forward_fmt.restype = ctypes.c_uint32
        f32 = ctypes.c_float
        L.or_pt_weight_scale.argtypes = [vp, i64]
        L.or_pt_weight_scale.restype = f32
        L.or_quant_weights_pt.argtypes = [vp, i64, i64, i64, vp, vp]
        L.or_quant_values_pt.argtypes = [vp, i64, f32, vp]
        L.or_forward_pt.argtypes = ([i64, i32, i32, i32, i32, i32] + [vp] * 7 + [f32, f32]
                                    + [vp] * 11)
        L.or_forward_pt.restype = ctypes.c_uint32
        _lib = L
    return _lib


# --------------------------------------------------------------------------
# number formats
# --------------------------------------------------------------------------
def e4m3_decode(code: int) -> float:
    return lib().or_e4m3_decode(code)


def e4m3_encode(v: float) -> int:
    return lib().or_e4m3_encode(v)


def e4m3_table() -> np.ndarray:
    return np.array([e4m3_decode(c) for c in range(256)], dtype=np.float64)


def bf16_round(v: float) -> int:
    return lib().or_bf16_round(v)


def bf16_decode(b: int) -> float:
    return lib().or_bf16_decode(b)


def pow2_scale_exp(amax: float) -> int:
    return lib().or_pow2_scale_exp(amax)


def swiglu(g_bits: int, u_bits: int) -> float:
    return lib().or_swiglu(g_bits, u_bits)


# --------------------------------------------------------------------------
# quantisation
# --------------------------------------------------------------------------
def quant_rows(v: np.ndarray, block: int = 128):
    """1 x block quantisation of float64 rows (block 128, or 32 for MXFP8)
    -> (q uint8, s float32 [rows, cols/block])."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    rows, cols = v.shape
    q = np.empty((rows, cols), np.uint8)
    s = np.empty((rows, cols // block), np.float32)
    lib().or_quant_rows_bw(_p(v), rows, cols, block, _p(q), _p(s))
    return q, s


def quant_rows_bf16(x_bits: np.ndarray, block: int = 128):
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    rows, cols = x.shape
    q = np.empty((rows, cols), np.uint8)
    s = np.empty((rows, cols // block), np.float32)
    lib().or_quant_rows_bf16_bw(_p(x), rows, cols, block, _p(q), _p(s))
    return q, s


def quant_weights(w: np.ndarray):
    """128x128 block quantisation of float32 [nmat, rows, cols]."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    nmat, rows, cols = w.shape
    q = np.empty(w.shape, np.uint8)
    s = np.empty((nmat, rows // 128, cols // 128), np.float32)
    lib().or_quant_weights(_p(w), nmat, rows, cols, _p(q), _p(s))
    return q, s


def quant_weights_mx(w: np.ndarray):
    """MXFP8 quantisation of float32 [nmat, rows, cols]: every row 1x32 along
    the columns -> (q uint8, s float32 [nmat, rows, cols/32])."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    nmat, rows, cols = w.shape
    q = np.empty(w.shape, np.uint8)
    s = np.empty((nmat, rows, cols // 32), np.float32)
    lib().or_quant_weights_mx(_p(w), nmat, rows, cols, _p(q), _p(s))
    return q, s


def e2m1_decode(nibble: int) -> float:
    return lib().or_e2m1_decode(nibble)


def dequant_nvfp4(codes: np.ndarray, sblk: np.ndarray, g: np.ndarray) -> np.ndarray:
    """NVFP4 matrices -> float32 values: codes uint8 [nmat, rows, cols/2] (two
    E2M1 codes per byte, the even column in the low nibble), sblk uint8
    [nmat, rows, cols/16] (E4M3 scale per 16 columns), g float32 [nmat]."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    sblk = np.ascontiguousarray(sblk, dtype=np.uint8)
    g = np.ascontiguousarray(g, dtype=np.float32)
    nmat, rows, half = codes.shape
    cols = 2 * half
    assert sblk.shape == (nmat, rows, cols // 16) and g.shape == (nmat,)
    out = np.empty((nmat, rows, cols), np.float32)
    lib().or_dequant_nvfp4(_p(codes), _p(sblk), _p(g), nmat, rows, cols, _p(out))
    return out


def requant_nvfp4(codes: np.ndarray, sblk: np.ndarray, g: np.ndarray):
    """NVFP4 matrices -> the 128x128 FP8 weight format (q, s): the weight
    quantiser applied to the dequantised float values."""
    return quant_weights(dequant_nvfp4(codes, sblk, g))


# --------------------------------------------------------------------------
# routing, expert FFN, combine, forward
# --------------------------------------------------------------------------
def route(idx: np.ndarray, w: np.ndarray, E: int, check: bool = True):
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    w = np.ascontiguousarray(w, dtype=np.float32)
    T, K = idx.shape
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    perm = np.full(max(T * K, 1), -1, np.int32)
    inv = np.empty(max(T * K, 1), np.int32)
    err = lib().or_route(T, K, E, _p(idx), _p(w), int(check), _p(counts), _p(offsets), _p(perm),
                         _p(inv))
    R = int(offsets[E])
    return dict(err=int(err), counts=counts, offsets=offsets, perm=perm[:R], inv=inv[:T * K])


def expert_ffn(H, I, E, offsets, A, As, W1, W1s, W2, W2s, sel=None, fmt=0):
    R = int(offsets[E])
    n = max(R, 1)
    bw = 32 if fmt == 1 else 128
    gu = np.zeros((n, 2 * I), np.uint16)
    hq = np.zeros((n, I), np.uint8)
    hs = np.zeros((n, I // bw), np.float32)
    y = np.zeros((n, H), np.uint16)
    args = [np.ascontiguousarray(a) for a in (offsets, A, As, W1, W1s, W2, W2s)]
    sel_a = None if sel is None else np.ascontiguousarray(sel, dtype=np.uint8)
    lib().or_expert_ffn_fmt(fmt, H, I, E, *[_p(a) for a in args], _p(sel_a), _p(gu), _p(hq), _p(hs),
                            _p(y))
    return gu[:R], hq[:R], hs[:R], y[:R]


def combine(inv, w, y, T, K, H, tok_sel=None):
    out = np.zeros((T, H), np.uint16)
    inv = np.ascontiguousarray(inv, dtype=np.int32)
    w = np.ascontiguousarray(w, dtype=np.float32)
    y = np.ascontiguousarray(y, dtype=np.uint16)
    ts = None if tok_sel is None else np.ascontiguousarray(tok_sel, dtype=np.uint8)
    lib().or_combine(T, K, H, _p(inv), _p(w), _p(y), _p(ts), _p(out))
    return out


def forward(x_bits, idx, w, W1, W1s, W2, W2s, check=True, tok_sel=None, fmt=0):
    """Whole layer.  Returns a dict with every intermediate (sorted-position
    arrays cover the R active routes) and ``out`` (bf16 bits [T, H]).
    fmt=1: MXFP8 (W1s [E, 2I, H/32], W2s [E, H, I/32]; 1x32 activations)."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    w = np.ascontiguousarray(w, dtype=np.float32)
    T, H = x.shape
    K = idx.shape[1]
    E, twoI, _ = W1.shape
    I = twoI // 2
    RK = max(T * K, 1)
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    perm = np.full(RK, -1, np.int32)
    inv = np.empty(RK, np.int32)
    bw = 32 if fmt == 1 else 128
    xq = np.empty((T, H), np.uint8)
    xs = np.empty((T, H // bw), np.float32)
    A = np.zeros((RK, H), np.uint8)
    As = np.zeros((RK, H // bw), np.float32)
    gu = np.zeros((RK, 2 * I), np.uint16)
    hq = np.zeros((RK, I), np.uint8)
    hs = np.zeros((RK, I // bw), np.float32)
    y = np.zeros((RK, H), np.uint16)
    out = np.zeros((T, H), np.uint16)
    ins = [np.ascontiguousarray(a) for a in (W1, W1s, W2, W2s)]
    ts = None if tok_sel is None else np.ascontiguousarray(tok_sel, dtype=np.uint8)
    err = lib().or_forward_fmt(fmt, T, H, I, E, K, int(check), _p(x), _p(idx), _p(w),
                               *[_p(a) for a in ins],
                           _p(ts), _p(counts), _p(offsets), _p(perm), _p(inv), _p(xq), _p(xs),
                           _p(A), _p(As), _p(gu), _p(hq), _p(hs), _p(y), _p(out))
    R = int(offsets[E]) if err == 0 else 0
    return dict(err=int(err), counts=counts, offsets=offsets, perm=perm[:R], inv=inv[:T * K],
                xq=xq, xs=xs, A=A[:R], As=As[:R], gu=gu[:R], hq=hq[:R], hs=hs[:R], y=y[:R],
                out=out)


# --------------------------------------------------------------------------
# per-tensor format
# --------------------------------------------------------------------------
def pt_weight_scale(w: np.ndarray) -> float:
    w = np.ascontiguousarray(w, dtype=np.float32)
    return float(lib().or_pt_weight_scale(_p(w), w.size))


def quant_weights_pt(w: np.ndarray):
    """Per-tensor quantisation of float32 [nmat, rows, cols]: one scale per
    matrix, s = float(amax / 448) -> (q uint8, s float32 [nmat])."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    nmat, rows, cols = w.shape
    q = np.empty(w.shape, np.uint8)
    s = np.empty(nmat, np.float32)
    lib().or_quant_weights_pt(_p(w), nmat, rows, cols, _p(q), _p(s))
    return q, s


def quant_values_pt(v: np.ndarray, scale: float) -> np.ndarray:
    """E4M3 codes of float values (each exactly a float32) with a static scale."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    q = np.empty(v.shape, np.uint8)
    lib().or_quant_values_pt(_p(v), v.size, float(np.float32(scale)), _p(q))
    return q


def forward_pt(x_bits, idx, w, W1, W1s, W2, W2s, x_scale, h_scale, check=True, tok_sel=None):
    """Whole layer in the per-tensor format: W1s, W2s float32 [E]; x_scale and
    h_scale the static activation scales.  Returns a dict like ``forward``
    (no per-row scale arrays: the block scales are all 1)."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    w = np.ascontiguousarray(w, dtype=np.float32)
    T, H = x.shape
    K = idx.shape[1]
    E, twoI, _ = W1.shape
    I = twoI // 2
    RK = max(T * K, 1)
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    perm = np.full(RK, -1, np.int32)
    inv = np.empty(RK, np.int32)
    xq = np.empty((T, H), np.uint8)
    A = np.zeros((RK, H), np.uint8)
    gu = np.zeros((RK, 2 * I), np.uint16)
    hq = np.zeros((RK, I), np.uint8)
    y = np.zeros((RK, H), np.uint16)
    out = np.zeros((T, H), np.uint16)
    ins = [np.ascontiguousarray(a) for a in (W1, np.asarray(W1s, np.float32), W2,
                                             np.asarray(W2s, np.float32))]
    ts = None if tok_sel is None else np.ascontiguousarray(tok_sel, dtype=np.uint8)
    err = lib().or_forward_pt(T, H, I, E, K, int(check), _p(x), _p(idx), _p(w),
                              *[_p(a) for a in ins], float(np.float32(x_scale)),
                              float(np.float32(h_scale)), _p(ts), _p(counts), _p(offsets),
                              _p(perm), _p(inv), _p(xq), _p(A), _p(gu), _p(hq), _p(y), _p(out))
    R = int(offsets[E]) if err == 0 else 0
    return dict(err=int(err), counts=counts, offsets=offsets, perm=perm[:R], inv=inv[:T * K],
                xq=xq, A=A[:R], gu=gu[:R], hq=hq[:R], y=y[:R], out=out)
