"""Seeded synthetic inputs shared by the oracle and the GPU path.

Holds no arithmetic of the MoE layer: only the counter-based generator of
``moegen.h`` restated in numpy, thin loaders for its C (host) and CUDA
(device) builds, and the routing recipes of the five workloads.

Generator definition (identical in all three implementations):
  * SplitMix64 in counter form: ``u64(key, i) = mix64(key + (i+1)*GAMMA)``,
    ``key = mix64(seed*GAMMA + tag)`` (Steele, Lea, Flood, OOPSLA 2014).
  * normal variate j: Irwin-Hall sum of the twelve 16-bit lanes of outputs
    3j, 3j+1, 3j+2, ``z = (2*S - 12*65535) / 2**17`` (exact in float32).
  * bf16 activations: the upper 16 bits of z's float32 pattern.
  * weights: ``float32(z) * float32(sigma)`` rounded to nearest.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
M1 = np.uint64(0xBF58476D1CE4E5B9)
M2 = np.uint64(0x94D049BB133111EB)

STREAM_X = 1
STREAM_W1 = 2
STREAM_W2 = 3
STREAM_LOGITS = 4
STREAM_BLOCKPERM = 5
STREAM_EXPERTPERM = 6
STREAM_GUMBEL = 7
STREAM_WLOGITS = 8

_HERE = os.path.dirname(os.path.abspath(__file__))


def mix64(z):
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * M1
        z = (z ^ (z >> np.uint64(27))) * M2
    return z ^ (z >> np.uint64(31))


def key(seed: int, tag: int) -> np.uint64:
    with np.errstate(over="ignore"):
        k = np.array([seed], dtype=np.uint64) * GAMMA + np.uint64(tag)
    return mix64(k)[0]


def u64(seed: int, tag: int, idx) -> np.ndarray:
    """64-bit outputs number ``idx`` (array) of stream ``tag``."""
    k = key(seed, tag)
    idx = np.asarray(idx, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return mix64(k + (idx + np.uint64(1)) * GAMMA)


def _lanesum(v: np.ndarray) -> np.ndarray:
    m = np.uint64(0xFFFF)
    return ((v & m) + ((v >> np.uint64(16)) & m) + ((v >> np.uint64(32)) & m)
            + (v >> np.uint64(48))).astype(np.int64)


def normal(seed: int, tag: int, idx) -> np.ndarray:
    """float32 normal variates number ``idx`` (array) of stream ``tag``."""
    idx = np.asarray(idx, dtype=np.uint64)
    three = np.uint64(3)
    s = (_lanesum(u64(seed, tag, three * idx)) + _lanesum(u64(seed, tag, three * idx + np.uint64(1)))
         + _lanesum(u64(seed, tag, three * idx + np.uint64(2))))
    c = 2 * s - 12 * 65535
    return (c.astype(np.float32) * np.float32(1.0 / 131072.0)).astype(np.float32)


def normal_bf16_bits(seed: int, tag: int, idx) -> np.ndarray:
    return (normal(seed, tag, idx).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def uniform01(seed: int, tag: int, idx) -> np.ndarray:
    """float32 uniforms in [0, 1): the top 24 bits of each output times 2^-24."""
    return ((u64(seed, tag, idx) >> np.uint64(40)).astype(np.float32) * np.float32(2.0 ** -24))


def uniform_open(seed: int, tag: int, idx) -> np.ndarray:
    """float64 uniforms in (0, 1): (top 32 bits + 0.5) * 2^-32."""
    return ((u64(seed, tag, idx) >> np.uint64(32)).astype(np.float64) + 0.5) * 2.0 ** -32


def uniform_int(seed: int, tag: int, idx, n) -> np.ndarray:
    """integers in [0, n): (top 32 bits * n) >> 32."""
    hi = u64(seed, tag, idx) >> np.uint64(32)
    return ((hi * np.asarray(n, dtype=np.uint64)) >> np.uint64(32)).astype(np.int64)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def weight_sigma(fan_in: int) -> np.float32:
    """std of the synthetic weights: 1/sqrt(fan_in) rounded to float32."""
    return np.float32(1.0 / np.sqrt(float(fan_in)))


# ----------------------------------------------------------------------------
# native builds of the same generator
# ----------------------------------------------------------------------------
_host_lib = None
_dev_lib = None


def host_lib():
    global _host_lib
    if _host_lib is None:
        path = os.path.join(_HERE, "libmoegen_host.so")
        if not os.path.exists(path):
            from . import build as _b
            _b.build_host()
        lib = ctypes.CDLL(path)
        lib.moegen_fill_normal_f32.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint64,
                                               ctypes.c_int64, ctypes.c_float, ctypes.c_void_p]
        lib.moegen_fill_normal_bf16.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint64,
                                                ctypes.c_int64, ctypes.c_void_p]
        lib.moegen_fill_u64.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint64,
                                        ctypes.c_int64, ctypes.c_void_p]
        _host_lib = lib
    return _host_lib


def dev_lib():
    global _dev_lib
    if _dev_lib is None:
        path = os.path.join(_HERE, "libmoegen_dev.so")
        if not os.path.exists(path):
            from . import build as _b
            _b.build_dev()
        lib = ctypes.CDLL(path)
        lib.moegen_dev_fill_normal_f32.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint64,
                                                   ctypes.c_int64, ctypes.c_float, ctypes.c_void_p,
                                                   ctypes.c_void_p]
        lib.moegen_dev_fill_normal_f32.restype = ctypes.c_int
        lib.moegen_dev_fill_normal_bf16.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint64,
                                                    ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]
        lib.moegen_dev_fill_normal_bf16.restype = ctypes.c_int
        _dev_lib = lib
    return _dev_lib


def host_normal_f32(seed: int, tag: int, offset: int, n: int, sigma) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    host_lib().moegen_fill_normal_f32(seed, tag, offset, n, float(np.float32(sigma)),
                                      out.ctypes.data)
    return out


def host_normal_bf16(seed: int, tag: int, offset: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint16)
    host_lib().moegen_fill_normal_bf16(seed, tag, offset, n, out.ctypes.data)
    return out


def host_u64(seed: int, tag: int, offset: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    host_lib().moegen_fill_u64(seed, tag, offset, n, out.ctypes.data)
    return out


def dev_normal_f32(seed: int, tag: int, offset: int, n: int, sigma, d_ptr: int, stream: int) -> None:
    rc = dev_lib().moegen_dev_fill_normal_f32(seed, tag, offset, n, float(np.float32(sigma)),
                                              ctypes.c_void_p(d_ptr), ctypes.c_void_p(stream))
    if rc != 0:
        raise RuntimeError(f"moegen_dev_fill_normal_f32 failed: cuda error {rc}")


def dev_normal_bf16(seed: int, tag: int, offset: int, n: int, d_ptr: int, stream: int) -> None:
    rc = dev_lib().moegen_dev_fill_normal_bf16(seed, tag, offset, n, ctypes.c_void_p(d_ptr),
                                               ctypes.c_void_p(stream))
    if rc != 0:
        raise RuntimeError(f"moegen_dev_fill_normal_bf16 failed: cuda error {rc}")
