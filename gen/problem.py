"""Raw synthetic inputs of a workload on the host (numpy): bf16 x bits, routes,
float32 weights.  Quantisation of the weights is left to each side (the
oracle's own encoder on the CPU, the library's quantiser on the GPU)."""
from __future__ import annotations

import numpy as np

from . import inputs as g
from .configs import Workload


def x_bits(wl: Workload, tokens=None) -> np.ndarray:
    """bf16 bit patterns [T, H] (or the listed token rows)."""
    H = wl.H
    if tokens is None:
        return g.host_normal_bf16(wl.seed, g.STREAM_X, 0, wl.T * H).reshape(wl.T, H)
    rows = [g.host_normal_bf16(wl.seed, g.STREAM_X, int(t) * H, H) for t in tokens]
    return np.stack(rows) if rows else np.zeros((0, H), np.uint16)


def w1_f32(wl: Workload, experts=None) -> np.ndarray:
    """float32 W1 [E, 2I, H] (or the listed experts), gate rows first."""
    n = 2 * wl.I * wl.H
    ex = range(wl.E) if experts is None else experts
    sig = g.weight_sigma(wl.H)
    return np.stack([g.host_normal_f32(wl.seed, g.STREAM_W1, int(e) * n, n, sig)
                     .reshape(2 * wl.I, wl.H) for e in ex])


def w2_f32(wl: Workload, experts=None) -> np.ndarray:
    """float32 W2 [E, H, I] (or the listed experts)."""
    n = wl.H * wl.I
    ex = range(wl.E) if experts is None else experts
    sig = g.weight_sigma(wl.I)
    return np.stack([g.host_normal_f32(wl.seed, g.STREAM_W2, int(e) * n, n, sig)
                     .reshape(wl.H, wl.I) for e in ex])
