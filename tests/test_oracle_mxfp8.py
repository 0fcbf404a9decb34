"""Pins of the oracle's MXFP8 format (fmt=1; CPU only).

MXFP8 ("32e4m3xe8m0" on flashinfer PR #4688; the SM100 MXFP8 megakernels of
PR #4069's kernel drops): E4M3 values with one power-of-two scale per 32
consecutive elements along K -- 1x32 for the activations, and 1x32 along K
for every weight row -- under the same scale rule as the 1x128 blocks.

* The quantisers against the library float8 cast, the minimal-scale property
  and the half-ulp round trip.
* Reduction: on inputs whose every 32-chunk holds its 128-block's amax, MXFP8
  codes equal the (already pinned) 1x128 / 128x128 codes and the scales repeat.
* E = 1, K = 1: the layer is one dense SwiGLU FFN, recomputed with torch
  library routines on 1x32 blocks, bit for bit.
* FC1 / FC2 against exact rational arithmetic on 32-wide blocks.
"""
from fractions import Fraction

import numpy as np
import torch

from tests import helpers_exact as hx
from tests.test_oracle_layer import dequant, rand_problem, torch_quant


def _half_ulp_ok(v, dec):
    ulp = np.where(np.abs(v) < 2.0 ** -6, 2.0 ** -9,
                   2.0 ** (np.floor(np.log2(np.maximum(np.abs(v), 2.0 ** -6))) - 3))
    return np.all(np.abs(v - dec) <= 0.5 * ulp)


def test_mx_quant_rows_library_cast_minimal_scale_roundtrip(orc):
    rng = np.random.default_rng(51)
    x = rng.standard_normal((32, 256))
    x *= 10.0 ** rng.integers(-4, 4, (32, 8)).repeat(32, axis=1)   # magnitudes vary per 32-chunk
    x[5, 64:96] = 0.0                                              # an all-zero chunk
    q, s = orc.quant_rows(x, block=32)
    assert s.shape == (32, 8)
    v = x / np.repeat(s.astype(np.float64), 32, axis=1)
    assert np.all(np.abs(v) <= 448.0)
    assert s[5, 2] == 1.0 and np.all(q[5, 64:96] == 0)
    assert _half_ulp_ok(v, hx.e4m3_values()[q])
    ref = torch.from_numpy(v.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(q, ref)
    amax = np.abs(x).reshape(32, 8, 32).max(axis=2)
    assert np.all(amax <= 448.0 * s) and np.all((amax > 448.0 * s / 2) | (amax == 0))


def test_mx_reduces_to_1x128_when_chunks_share_the_block_amax(orc):
    rng = np.random.default_rng(52)
    x = rng.standard_normal((16, 512)) * 0.3
    blk = np.abs(x).reshape(16, 4, 128).max(axis=2) * 1.5          # each 128-block's amax
    for c in range(16):                                            # every 32-chunk holds it
        x[:, 32 * c] = blk[:, c // 4] * np.where(c % 2, -1.0, 1.0)
    q32, s32 = orc.quant_rows(x, block=32)
    q128, s128 = orc.quant_rows(x)
    assert np.array_equal(q32, q128)
    assert np.array_equal(s32, np.repeat(s128, 4, axis=1))


def test_mx_weights_library_cast_and_reduction(orc):
    rng = np.random.default_rng(53)
    w = (rng.standard_normal((2, 256, 384)) * 0.02).astype(np.float32)
    w[1, :, 64:96] *= 1000.0
    q, s = orc.quant_weights_mx(w)
    assert s.shape == (2, 256, 12)
    for m in range(2):
        rq, rs = torch_quant(torch.from_numpy(w[m]).to(torch.float64), 1, 32)
        assert np.array_equal(q[m], rq.view(torch.uint8).numpy())
        assert np.array_equal(s[m], rs.numpy().astype(np.float32))
    # reduction to 128x128: every row's 32-chunks inside a 128x128 block hold
    # that block's amax
    w2 = (rng.standard_normal((1, 256, 256)) * 0.05).astype(np.float32)
    amax = np.abs(w2[0]).reshape(2, 128, 2, 128).max(axis=(1, 3)) * 1.25
    for r in range(256):
        for c in range(8):
            w2[0, r, 32 * c + (r % 32)] = amax[r // 128, c // 4]
    qm, sm = orc.quant_weights_mx(w2)
    qb, sb = orc.quant_weights(w2)
    assert np.array_equal(qm, qb)
    assert np.array_equal(sm[0], np.repeat(np.repeat(sb[0], 128, axis=0), 4, axis=1))


def test_mx_dense_ffn_e1_k1_bit_exact(orc):
    T, H, I = 48, 256, 384
    x, _, _, w1, w2 = rand_problem(T, H, I, 1, 1, seed=54)
    idx = np.zeros((T, 1), np.int32)
    w = np.ones((T, 1), np.float32)
    W1q, W1s = torch_quant(torch.from_numpy(w1[0]).to(torch.float64), 1, 32)
    W2q, W2s = torch_quant(torch.from_numpy(w2[0]).to(torch.float64), 1, 32)
    r = orc.forward(x, idx, w, W1q.view(torch.uint8).numpy()[None], W1s.numpy().astype(np.float32)[None],
                    W2q.view(torch.uint8).numpy()[None], W2s.numpy().astype(np.float32)[None], fmt=1)
    assert r["err"] == 0
    xd = torch.from_numpy(hx.bf16_bits_to_f64(x))
    xq, xs = torch_quant(xd, 1, 32)
    gu_bits = hx.f64_to_bf16_bits((dequant(xq, xs, 1, 32) @ dequant(W1q, W1s, 1, 32).T).numpy())
    gu = torch.from_numpy(hx.bf16_bits_to_f64(gu_bits))
    gate, up = gu[:, :I], gu[:, I:]
    h = (gate / (1.0 + torch.exp(-gate)) * up).to(torch.float32).to(torch.float64)
    hq, hs = torch_quant(h, 1, 32)
    y_bits = hx.f64_to_bf16_bits((dequant(hq, hs, 1, 32) @ dequant(W2q, W2s, 1, 32).T).numpy())
    assert np.array_equal(r["xq"], xq.view(torch.uint8).numpy())
    assert np.array_equal(r["xs"], xs.numpy().astype(np.float32))
    assert np.array_equal(r["gu"], gu_bits)
    assert np.array_equal(r["hq"], hq.view(torch.uint8).numpy())
    assert np.array_equal(r["hs"], hs.numpy().astype(np.float32))
    assert np.array_equal(r["y"], y_bits)
    assert np.array_equal(r["out"], y_bits)


def test_mx_fc1_fc2_exact_rational(orc):
    T, H, I, E, K = 5, 128, 128, 3, 2
    x, idx, w, w1, w2 = rand_problem(T, H, I, E, K, seed=55)
    W1q, W1s = orc.quant_weights_mx(w1)
    W2q, W2s = orc.quant_weights_mx(w2)
    r = orc.forward(x, idx, w, W1q, W1s, W2q, W2s, fmt=1)
    dec = [Fraction(float(v)) if np.isfinite(v) else None for v in hx.e4m3_values()]
    off = r["offsets"]
    for pos in (0, int(off[E]) - 1):
        e = int(np.searchsorted(off, pos, side="right") - 1)
        a = [dec[c] for c in r["A"][pos]]
        for n in range(0, 2 * I, 23):
            tot = Fraction(0)
            for b in range(H // 32):
                bs = sum(a[j] * dec[W1q[e, n, j]] for j in range(32 * b, 32 * b + 32))
                tot += bs * Fraction(float(r["As"][pos, b])) * Fraction(float(W1s[e, n, b]))
            assert r["gu"][pos, n] == hx.exact_round_bf16(tot), (pos, n)
        hqd = [dec[c] for c in r["hq"][pos]]
        for c in range(0, H, 19):
            tot = Fraction(0)
            for b in range(I // 32):
                bs = sum(hqd[j] * dec[W2q[e, c, j]] for j in range(32 * b, 32 * b + 32))
                tot += bs * Fraction(float(r["hs"][pos, b])) * Fraction(float(W2s[e, c, b]))
            assert r["y"][pos, c] == hx.exact_round_bf16(tot), (pos, c)


def test_mx_token_permutation_permutes_output(orc):
    T, H, I, E, K = 24, 256, 128, 6, 2
    x, idx, w, w1, w2 = rand_problem(T, H, I, E, K, seed=56)
    wq = orc.quant_weights_mx(w1) + orc.quant_weights_mx(w2)
    base = orc.forward(x, idx, w, *wq, fmt=1)
    p = np.random.default_rng(57).permutation(T)
    perm = orc.forward(x[p], idx[p], w[p], *wq, fmt=1)
    assert np.array_equal(perm["out"], base["out"][p])
