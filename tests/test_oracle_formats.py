"""Pins of the oracle's number formats and quantisation rules (CPU only).

Each check ties the oracle to something other than itself: torch's FP8/BF16
conversions (library routines), a nearest-code search over all 256 codes,
integer bit manipulation, and exact rational arithmetic.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

from tests import helpers_exact as hx


def test_e4m3_decode_matches_library(orc):
    ref = hx.e4m3_values()
    mine = orc.e4m3_table()
    nan_ref = np.isnan(ref)
    assert np.array_equal(nan_ref, np.isnan(mine))
    assert nan_ref.sum() == 2  # 0x7F and 0xFF only: E4M3FN has no infinity
    assert np.array_equal(np.signbit(ref[~nan_ref]), np.signbit(mine[~nan_ref]))
    assert np.array_equal(ref[~nan_ref], mine[~nan_ref])
    assert mine[0x7E] == 448.0 and mine[0x01] == 2.0 ** -9


@pytest.mark.parametrize("scale_exp", [0, -6, 3, -12])
def test_e4m3_encode_matches_library_on_every_bf16(orc, scale_exp):
    """Every bf16 value divided by a power of two, where |v| <= 448: the oracle's
    encoder equals torch's round-to-nearest-even float8_e4m3fn cast."""
    with np.errstate(invalid="ignore"):
        v = hx.bf16_values_all().astype(np.float64) * 2.0 ** (-scale_exp)
    ok = np.isfinite(v) & (np.abs(v) <= 448.0)
    v = v[ok]
    ref = torch.from_numpy(v.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    enc = np.frompyfunc(orc.e4m3_encode, 1, 1)
    mine = enc(v).astype(np.uint8)
    assert np.array_equal(mine, ref)


def test_e4m3_encode_is_nearest_code(orc):
    """Brute force: the code minimising |v - dec(code)|, ties to the even code."""
    table = hx.e4m3_values()
    finite = np.where(np.isfinite(table))[0]
    rng = np.random.default_rng(1)
    vals = np.concatenate([rng.uniform(-448, 448, 3000), rng.uniform(-0.02, 0.02, 3000),
                           (table[finite] + np.roll(table[finite], 1)) / 2])  # midpoints
    vals = vals[np.abs(vals) <= 448]
    for v in vals:
        d = np.abs(table[finite] - v)
        best = finite[d == d.min()]
        if len(best) > 1:
            best = [c for c in best if c % 2 == 0 and (np.signbit(table[c]) == np.signbit(v) or table[c] == 0)] or best
        code = orc.e4m3_encode(float(v))
        assert table[code] == table[best[0]], (v, code, best)


def test_e4m3_negative_zero_and_saturation(orc):
    assert orc.e4m3_encode(-0.0) == 0x80
    assert orc.e4m3_encode(-1e-6) == 0x80
    assert orc.e4m3_encode(1e-6) == 0x00
    assert orc.e4m3_encode(1000.0) == 0x7E  # saturating (the satfinite reading)
    assert orc.e4m3_encode(-1000.0) == 0xFE


def test_bf16_round_matches_library_on_float32(orc):
    rng = np.random.default_rng(2)
    f = np.concatenate([rng.standard_normal(20000).astype(np.float32),
                        (rng.standard_normal(5000) * 1e-30).astype(np.float32),
                        (rng.standard_normal(5000) * 1e30).astype(np.float32),
                        np.float32([0.0, -0.0, 1e-40, -1e-41])])
    # exact bf16 midpoints: low 16 bits 0x8000 (ties) on both even and odd patterns
    mids = ((rng.integers(0x3000, 0x4F00, 4000).astype(np.uint32) << 16) | 0x8000).view(np.float32)
    f = np.concatenate([f, mids])
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    rnd = np.frompyfunc(orc.bf16_round, 1, 1)
    mine = rnd(f.astype(np.float64)).astype(np.uint16)
    assert np.array_equal(mine, ref)


def test_bf16_round_single_rounding_from_double(orc):
    """float64 inputs that a float32 intermediate would double-round: compare
    with integer bit rounding and with exact rational nearest search."""
    rng = np.random.default_rng(3)
    base = (rng.integers(0x3000, 0x4F00, 3000).astype(np.uint32) << 16 | 0x8000).view(np.float32)
    d = base.astype(np.float64) * (1.0 + np.where(rng.random(3000) < 0.5, -1, 1) * 2.0 ** -40)
    d = np.concatenate([d, rng.standard_normal(3000) * 100])
    rnd = np.frompyfunc(orc.bf16_round, 1, 1)
    mine = rnd(d).astype(np.uint16)
    assert np.array_equal(mine, hx.f64_to_bf16_bits(d))
    for v in d[:200]:
        assert orc.bf16_round(float(v)) == hx.exact_round_bf16(Fraction(float(v)))


def test_pow2_scale_rule_brute_force(orc):
    rng = np.random.default_rng(4)
    vals = np.concatenate([np.abs(rng.standard_normal(2000)) * 10.0 ** rng.integers(-20, 20, 2000),
                           448.0 * 2.0 ** np.arange(-30, 30), 448.0 * 2.0 ** np.arange(-30, 30) * (1 + 2 ** -20),
                           hx.bf16_values_all()[1:0x7F80:97].astype(np.float64)])
    for a in vals:
        e = orc.pow2_scale_exp(float(a))
        # brute force: the smallest e in [-127, 127] with a <= 448 * 2^e
        want = next(k for k in range(-127, 128) if Fraction(float(a)) <= 448 * Fraction(2) ** k)
        assert e == want, (a, e, want)
    assert orc.pow2_scale_exp(0.0) == 0
    assert orc.pow2_scale_exp(1e-45) == -127


def test_quant_rows_roundtrip_half_ulp(orc):
    """|x - dec(q)*s| <= half an E4M3 ulp of x/s (times s), and every code is the
    library cast of x/s."""
    rng = np.random.default_rng(5)
    x = rng.standard_normal((64, 512)) * 10.0 ** rng.integers(-3, 3, (64, 1))
    x[3, :128] = 0.0
    q, s = orc.quant_rows(x)
    table = hx.e4m3_values()
    sfull = np.repeat(s.astype(np.float64), 128, axis=1)
    v = x / sfull
    assert np.all(np.abs(v) <= 448.0)
    assert s[3, 0] == 1.0 and np.all(q[3, :128] == 0)
    ulp = np.where(np.abs(v) < 2.0 ** -6, 2.0 ** -9, 2.0 ** (np.floor(np.log2(np.maximum(np.abs(v), 2.0 ** -6))) - 3))
    assert np.all(np.abs(v - table[q]) <= 0.5 * ulp)
    ref = torch.from_numpy(v.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(q, ref)
    # the scale is minimal: halving it would overflow 448 for some element
    amax = np.abs(x).reshape(64, 4, 128).max(axis=2)
    assert np.all(amax <= 448.0 * s) and np.all((amax > 448.0 * s / 2) | (amax == 0))


def test_quant_weights_blocks(orc):
    rng = np.random.default_rng(6)
    w = (rng.standard_normal((2, 256, 384)) * 0.02).astype(np.float32)
    w[1, 128:, 256:] *= 1000.0
    q, s = orc.quant_weights(w)
    assert s.shape == (2, 2, 3)
    table = hx.e4m3_values()
    for m in range(2):
        for bi in range(2):
            for bj in range(3):
                blk = w[m, bi * 128:(bi + 1) * 128, bj * 128:(bj + 1) * 128].astype(np.float64)
                sc = float(s[m, bi, bj])
                assert sc == 2.0 ** round(np.log2(sc))
                amax = np.abs(blk).max()
                assert amax <= 448 * sc < 2 * amax
                ref = torch.from_numpy((blk / sc).astype(np.float32)).to(torch.float8_e4m3fn)
                assert np.array_equal(q[m, bi * 128:(bi + 1) * 128, bj * 128:(bj + 1) * 128],
                                      ref.view(torch.uint8).numpy())
    assert table[q].dtype == np.float64
