"""Pins of the oracle's layer arithmetic (CPU only).

* E = 1, K = 1: the layer reduces to one dense SwiGLU FFN with the same
  quantisation chain; recomputed here with torch library routines (float8 and
  float64 casts, float64 matmul) and integer bf16 rounding -- bit for bit.
* FC1/FC2/combine against exact rational arithmetic on tiny inputs.
* Invariants: token permutation, poisoned empty experts, power-of-two
  scaling, masked routes.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

from gen import inputs as g
from tests import helpers_exact as hx


def torch_quant(v: torch.Tensor, rb: int, cb: int):
    """Block quantisation with torch ops: blocks of rb x cb, scale = the smallest
    power of two >= amax/448 (1 when amax = 0), codes = float8_e4m3fn cast."""
    R, C = v.shape
    blk = v.reshape(R // rb, rb, C // cb, cb)
    amax = blk.abs().amax(dim=(1, 3))
    e = torch.ceil(torch.log2(amax / 448.0)).clamp(-127, 127)
    e[amax == 0] = 0
    s = torch.pow(2.0, e)
    q = (blk / s[:, None, :, None]).to(torch.float32).to(torch.float8_e4m3fn).reshape(R, C)
    return q, s


def dequant(q: torch.Tensor, s: torch.Tensor, rb: int, cb: int) -> torch.Tensor:
    R, C = q.shape
    return (q.to(torch.float64).reshape(R // rb, rb, C // cb, cb) * s[:, None, :, None]).reshape(R, C)


def rand_problem(T, H, I, E, K, seed, mask=0.0):
    rng = np.random.default_rng(seed)
    x = g.normal_bf16_bits(seed, g.STREAM_X, np.arange(T * H, dtype=np.uint64)).reshape(T, H)
    idx = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    if mask:
        idx[rng.random(idx.shape) < mask] = -1
    w = rng.random((T, K)).astype(np.float32) + 0.1
    w1 = (rng.standard_normal((E, 2 * I, H)) / np.sqrt(H)).astype(np.float32)
    w2 = (rng.standard_normal((E, H, I)) / np.sqrt(I)).astype(np.float32)
    return x, idx, w, w1, w2


def test_dense_ffn_e1_k1_bit_exact(orc):
    T, H, I = 64, 512, 256
    x, _, _, w1, w2 = rand_problem(T, H, I, 1, 1, seed=21)
    idx = np.zeros((T, 1), np.int32)
    w = np.ones((T, 1), np.float32)
    W1q, W1s = torch_quant(torch.from_numpy(w1[0]).to(torch.float64), 128, 128)
    W2q, W2s = torch_quant(torch.from_numpy(w2[0]).to(torch.float64), 128, 128)
    r = orc.forward(x, idx, w, W1q.view(torch.uint8).numpy()[None], W1s.numpy().astype(np.float32)[None],
                    W2q.view(torch.uint8).numpy()[None], W2s.numpy().astype(np.float32)[None])
    assert r["err"] == 0
    # brute force dense FFN, torch library ops
    xd = torch.from_numpy(hx.bf16_bits_to_f64(x))
    xq, xs = torch_quant(xd, 1, 128)
    gu_d = dequant(xq, xs, 1, 128) @ dequant(W1q, W1s, 128, 128).T
    gu_bits = hx.f64_to_bf16_bits(gu_d.numpy())
    gu = torch.from_numpy(hx.bf16_bits_to_f64(gu_bits))
    gate, up = gu[:, :I], gu[:, I:]
    h = (gate / (1.0 + torch.exp(-gate)) * up).to(torch.float32).to(torch.float64)
    hq, hs = torch_quant(h, 1, 128)
    y_d = dequant(hq, hs, 1, 128) @ dequant(W2q, W2s, 128, 128).T
    y_bits = hx.f64_to_bf16_bits(y_d.numpy())
    assert np.array_equal(r["xq"], xq.view(torch.uint8).numpy())
    assert np.array_equal(r["xs"], xs.numpy().astype(np.float32))
    assert np.array_equal(r["gu"], gu_bits)        # perm is the identity for E = 1, K = 1
    assert np.array_equal(r["hq"], hq.view(torch.uint8).numpy())
    assert np.array_equal(r["hs"], hs.numpy().astype(np.float32))
    assert np.array_equal(r["y"], y_bits)
    assert np.array_equal(r["out"], y_bits)        # w = 1: combine is the identity


def test_fc1_fc2_combine_exact_rational(orc):
    T, H, I, E, K = 6, 256, 128, 3, 2
    x, idx, w, w1, w2 = rand_problem(T, H, I, E, K, seed=22)
    W1q, W1s = orc.quant_weights(w1)
    W2q, W2s = orc.quant_weights(w2)
    r = orc.forward(x, idx, w, W1q, W1s, W2q, W2s)
    dec = [Fraction(float(v)) if np.isfinite(v) else None for v in hx.e4m3_values()]
    off = r["offsets"]
    for pos in (0, int(off[1]), int(off[E]) - 1):
        e = int(np.searchsorted(off, pos, side="right") - 1)
        a = [dec[c] for c in r["A"][pos]]
        for n in range(0, 2 * I, 37):
            tot = Fraction(0)
            for kb in range(H // 128):
                bs = sum(a[j] * dec[W1q[e, n, j]] for j in range(kb * 128, kb * 128 + 128))
                tot += bs * Fraction(float(r["As"][pos, kb])) * Fraction(float(W1s[e, n // 128, kb]))
            assert r["gu"][pos, n] == hx.exact_round_bf16(tot), (pos, n)
        hqd = [dec[c] for c in r["hq"][pos]]
        for c in range(0, H, 41):
            tot = Fraction(0)
            for kb in range(I // 128):
                bs = sum(hqd[j] * dec[W2q[e, c, j]] for j in range(kb * 128, kb * 128 + 128))
                tot += bs * Fraction(float(r["hs"][pos, kb])) * Fraction(float(W2s[e, c // 128, kb]))
            assert r["y"][pos, c] == hx.exact_round_bf16(tot), (pos, c)
    ydec = hx.bf16_bits_to_f64(r["y"])
    for t in range(T):
        for c in range(0, H, 29):
            tot = sum(Fraction(float(w[t, k])) * Fraction(float(ydec[r["inv"][t * K + k], c]))
                      for k in range(K) if idx[t, k] >= 0)
            assert r["out"][t, c] == hx.exact_round_bf16(Fraction(tot)) if tot != 0 else r["out"][t, c] == 0


@pytest.fixture(scope="module")
def small_layer(orc):
    T, H, I, E, K = 40, 256, 256, 8, 2
    x, idx, w, w1, w2 = rand_problem(T, H, I, E, K, seed=23)
    W1q, W1s = orc.quant_weights(w1)
    W2q, W2s = orc.quant_weights(w2)
    return x, idx, w, W1q, W1s, W2q, W2s


def test_token_permutation_permutes_output(orc, small_layer):
    x, idx, w, *W = small_layer
    base = orc.forward(x, idx, w, *W)["out"]
    p = np.random.default_rng(24).permutation(x.shape[0])
    perm_out = orc.forward(x[p], idx[p], w[p], *W)["out"]
    assert np.array_equal(perm_out, base[p])


def test_empty_experts_contribute_nothing(orc, small_layer):
    x, idx, w, W1q, W1s, W2q, W2s = small_layer
    idx2 = np.where(idx >= 6, idx - 6, idx).astype(np.int32)   # experts 6, 7 now empty
    ok = np.all(idx2[:, :1] != idx2[:, 1:], axis=1)
    x2, idx2, w2_ = x[ok], idx2[ok], w[ok]
    base = orc.forward(x2, idx2, w2_, W1q, W1s, W2q, W2s)
    P1, P2 = W1q.copy(), W2q.copy()
    P1[6:], P2[6:] = 0x7F, 0x7F     # NaN codes in the unused experts
    S1, S2 = W1s.copy(), W2s.copy()
    S1[6:], S2[6:] = np.nan, np.nan
    pois = orc.forward(x2, idx2, w2_, P1, S1, P2, S2)
    assert np.all(base["counts"][6:] == 0)
    assert np.array_equal(pois["out"], base["out"])
    assert np.all(np.isfinite(hx.bf16_bits_to_f64(pois["out"])))


def test_pow2_scaling_invariance(orc, small_layer):
    x, idx, w, *W = small_layer
    base = orc.forward(x, idx, w, *W)
    x4 = (x.astype(np.uint32) + np.uint32(2 << 7)).astype(np.uint16)  # exponent + 2: x * 4
    x4 = np.where((x & 0x7FFF) == 0, x, x4)
    r4 = orc.forward(x4, idx, w, *W)
    assert np.array_equal(r4["xq"], base["xq"])
    assert np.array_equal(r4["xs"], base["xs"] * 4)
    r2 = orc.forward(x, idx, (w * 2).astype(np.float32), *W)
    assert np.array_equal(hx.bf16_bits_to_f64(r2["out"]), 2 * hx.bf16_bits_to_f64(base["out"]))


def test_masked_routes(orc, small_layer):
    x, idx, w, *W = small_layer
    allm = orc.forward(x, np.full_like(idx, -1), w, *W)
    assert allm["err"] == 0 and np.all(allm["out"] == 0)
    idxm = idx.copy()
    idxm[::3, 1] = -1
    a = orc.forward(x, idxm, w, *W)
    wn = w.copy()
    wn[::3, 1] = np.nan
    b = orc.forward(x, idxm, wn, *W)
    assert b["err"] == 0 and np.array_equal(a["out"], b["out"])
    # a token whose every route is masked gets +0
    idxm[5] = -1
    c = orc.forward(x, idxm, w, *W)
    assert np.all(c["out"][5] == 0)


def test_token_subset_matches_full(orc, small_layer):
    x, idx, w, *W = small_layer
    full = orc.forward(x, idx, w, *W)["out"]
    sel = np.zeros(x.shape[0], np.uint8)
    sel[[0, 7, 39]] = 1
    part = orc.forward(x, idx, w, *W, tok_sel=sel)["out"]
    assert np.array_equal(part[sel == 1], full[sel == 1])
