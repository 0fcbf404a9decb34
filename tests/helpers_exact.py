"""Independent exact-arithmetic helpers for the oracle pins (no oracle code)."""
from __future__ import annotations

from fractions import Fraction

import numpy as np
import torch


def e4m3_values() -> np.ndarray:
    """float64 value of every E4M3FN code, decoded by torch (a library routine)."""
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def bf16_values_all() -> np.ndarray:
    """float32 value of every bf16 bit pattern."""
    return (np.arange(65536, dtype=np.uint32) << np.uint32(16)).view(np.float32)


def f64_to_bf16_bits(d: np.ndarray) -> np.ndarray:
    """Round float64 to bf16 (nearest, ties to even) by integer bit manipulation
    of the float64 pattern; normal range only (asserted)."""
    d = np.asarray(d, dtype=np.float64)
    bits = d.view(np.uint64)
    sign = (bits >> np.uint64(63)).astype(np.uint64)
    exp = ((bits >> np.uint64(52)) & np.uint64(0x7FF)).astype(np.int64)
    man = bits & np.uint64((1 << 52) - 1)
    nz = d != 0
    assert np.all((exp[nz] - 1023 >= -126) & (exp[nz] - 1023 <= 127)), "outside bf16 normal range"
    keep = man >> np.uint64(45)
    low = man & np.uint64((1 << 45) - 1)
    half = np.uint64(1 << 44)
    up = (low > half) | ((low == half) & ((keep & np.uint64(1)) == np.uint64(1)))
    keep = keep + up.astype(np.uint64)
    carry = keep >> np.uint64(7)
    keep = keep & np.uint64(0x7F)
    e = exp - 1023 + carry.astype(np.int64) + 127
    out = (sign << np.uint64(15)) | (e.astype(np.uint64) << np.uint64(7)) | keep
    out = np.where(nz, out, sign << np.uint64(15))
    return out.astype(np.uint16)


def bf16_bits_to_f64(b) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def exact_round_bf16(x: Fraction) -> int:
    """bf16 bits nearest to the exact rational x (ties to even), by comparing x
    with the neighbours of a float64 first guess in exact arithmetic."""
    if x == 0:
        return 0
    guess = int(f64_to_bf16_bits(np.array([float(x)]))[0])
    cands = [guess - 1, guess, guess + 1]
    best, bestd = None, None
    for c in cands:
        v = Fraction(float(bf16_bits_to_f64(np.array([c], np.uint16))[0]))
        d = abs(v - x)
        if best is None or d < bestd or (d == bestd and c % 2 == 0):
            best, bestd = c, d
    return best
