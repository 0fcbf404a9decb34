"""Pins of the oracle's per-tensor format (CPU only).

The "per_tensor" FP8 scale mode of flashinfer PR #4688 (Description, the
scale-mode-equalized comparison: per_tensor needs offline-calibrated
activation scales identical on every rank, blockwise needs none): one FP32
scale per expert weight matrix and one static, calibrated FP32 scale per
activation tensor (x, and the SwiGLU output h), no block scales.  Values
quantise as E4M3_RNE_sat(float(v) * float(1/s)); a weight matrix's scale is
float(amax / 448).

* The quantisers against the library float8 cast of the same float32 product,
  including saturation under a calibrated scale that is too small.
* E = 1, K = 1: the layer is one dense SwiGLU FFN, recomputed with torch
  library routines, bit for bit.
* FC1 / FC2 against exact rational arithmetic.
* Reduction: with unit scales and inputs whose 1x128 / 128x128 block scales
  are all 1, the per-tensor FC1 equals the (already pinned) blockwise FC1 bit
  for bit.
* x * 2 with the x scale * 2 keeps every code and doubles gate||up exactly.
"""
from fractions import Fraction

import numpy as np
import torch

from tests import helpers_exact as hx
from tests.test_oracle_layer import rand_problem

F32 = np.float32


def torch_pt_codes(v32: np.ndarray, r: np.float32) -> np.ndarray:
    """library float8 cast of the float32 product v * r, clamped to the finite
    E4M3 range first (saturation)"""
    p = torch.from_numpy(np.ascontiguousarray(v32, dtype=np.float32)) * torch.tensor(r, dtype=torch.float32)
    return p.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def pt_scale(w32: np.ndarray) -> np.float32:
    amax = F32(np.max(np.abs(w32)))
    return F32(amax / F32(448.0)) if amax > 0 else F32(1.0)


def test_pt_weight_quant_library_cast(orc):
    rng = np.random.default_rng(61)
    w = (rng.standard_normal((3, 256, 384)) * 0.03).astype(np.float32)
    w[1] *= 2.0 ** 30                       # a large matrix
    w[2] = 0.0                              # an all-zero matrix: scale 1, codes 0
    q, s = orc.quant_weights_pt(w)
    assert s.shape == (3,) and s[2] == 1.0 and np.all(q[2] == 0)
    for m in range(3):
        sm = pt_scale(w[m])
        assert s[m] == sm and orc.pt_weight_scale(w[m]) == sm
        assert np.array_equal(q[m], torch_pt_codes(w[m], F32(F32(1.0) / sm)))
    # the largest element maps to +-448 exactly (or rounds down by less than an ulp)
    dec = hx.e4m3_values()
    assert np.max(np.abs(dec[q[0]])) == 448.0


def test_pt_activation_quant_saturates_under_a_small_scale(orc):
    rng = np.random.default_rng(62)
    v = rng.standard_normal(4096).astype(np.float32) * 3.0
    v[:4] = [0.0, -0.0, 1e-30, -1e-30]
    for scale in (F32(6.0 / 448.0), F32(0.001), F32(2.0 ** -3)):
        q = orc.quant_values_pt(v.astype(np.float64), scale)
        ref = torch_pt_codes(v, F32(F32(1.0) / scale))
        assert np.array_equal(q, ref), scale
    q = orc.quant_values_pt(v.astype(np.float64), F32(0.001))
    assert np.sum((q & 0x7F) == 0x7E) > 100            # saturated codes, never NaN
    assert not np.any((q & 0x7F) == 0x7F)
    assert q[1] == 0x80                                 # -0 keeps its sign


def test_pt_dense_ffn_e1_k1_bit_exact(orc):
    T, H, I = 40, 256, 384
    x, _, _, w1, w2 = rand_problem(T, H, I, 1, 1, seed=63)
    idx = np.zeros((T, 1), np.int32)
    w = np.ones((T, 1), np.float32)
    sx, sh = F32(6.0 / 448.0), F32(20.0 / 448.0)
    W1q, W1s = orc.quant_weights_pt(w1)
    W2q, W2s = orc.quant_weights_pt(w2)
    r = orc.forward_pt(x, idx, w, W1q, W1s, W2q, W2s, sx, sh)
    assert r["err"] == 0
    dec = torch.from_numpy(hx.e4m3_values())
    xf = hx.bf16_bits_to_f64(x).astype(np.float32)
    xq = torch_pt_codes(xf, F32(F32(1.0) / sx))
    acc1 = dec[torch.from_numpy(xq).long()] @ dec[torch.from_numpy(W1q[0]).long()].T
    gu_bits = hx.f64_to_bf16_bits((acc1 * (float(sx) * float(W1s[0]))).numpy())
    gu = torch.from_numpy(hx.bf16_bits_to_f64(gu_bits))
    gate, up = gu[:, :I], gu[:, I:]
    h = (gate / (1.0 + torch.exp(-gate)) * up).to(torch.float32)
    hq = torch_pt_codes(h.numpy(), F32(F32(1.0) / sh))
    acc2 = dec[torch.from_numpy(hq).long()] @ dec[torch.from_numpy(W2q[0]).long()].T
    y_bits = hx.f64_to_bf16_bits((acc2 * (float(sh) * float(W2s[0]))).numpy())
    assert np.array_equal(r["xq"], xq)
    assert np.array_equal(r["gu"], gu_bits)
    assert np.array_equal(r["hq"], hq)
    assert np.array_equal(r["y"], y_bits)
    assert np.array_equal(r["out"], y_bits)


def test_pt_fc1_fc2_exact_rational(orc):
    T, H, I, E, K = 5, 128, 256, 3, 2
    x, idx, w, w1, w2 = rand_problem(T, H, I, E, K, seed=64)
    W1q, W1s = orc.quant_weights_pt(w1)
    W2q, W2s = orc.quant_weights_pt(w2)
    sx, sh = F32(5.5 / 448.0), F32(3.0 / 448.0)
    r = orc.forward_pt(x, idx, w, W1q, W1s, W2q, W2s, sx, sh)
    dec = [Fraction(float(v)) if np.isfinite(v) else None for v in hx.e4m3_values()]
    off = r["offsets"]
    for pos in (0, int(off[E]) - 1):
        e = int(np.searchsorted(off, pos, side="right") - 1)
        a = [dec[c] for c in r["A"][pos]]
        f1 = Fraction(float(sx)) * Fraction(float(W1s[e]))
        for n in range(0, 2 * I, 29):
            tot = sum(a[j] * dec[W1q[e, n, j]] for j in range(H)) * f1
            assert r["gu"][pos, n] == hx.exact_round_bf16(tot), (pos, n)
        hqd = [dec[c] for c in r["hq"][pos]]
        f2 = Fraction(float(sh)) * Fraction(float(W2s[e]))
        for c in range(0, H, 13):
            tot = sum(hqd[j] * dec[W2q[e, c, j]] for j in range(I)) * f2
            assert r["y"][pos, c] == hx.exact_round_bf16(tot), (pos, c)


def test_pt_fc1_equals_blockwise_fc1_on_unit_scales(orc):
    """Codes given directly, every weight scale 1 (128x128 blocks of 1, or one
    per-tensor 1); x with every 1x128 block's amax in (224, 448], so its
    blockwise scale is 1 too, and x scale 1: both formats quantise x to the
    same codes and compute the same gate||up."""
    rng = np.random.default_rng(65)
    T, H, I, E, K = 6, 256, 128, 2, 2
    codes = np.arange(256, dtype=np.uint8)
    finite = codes[(codes & 0x7F) != 0x7F]
    W1q = rng.choice(finite, size=(E, 2 * I, H)).astype(np.uint8)
    W2q = rng.choice(finite, size=(E, H, I)).astype(np.uint8)
    xv = rng.standard_normal((T, H)) * 30.0
    xv[:, ::128] = 300.0                                   # each 1x128 block's amax: 300
    x = hx.f64_to_bf16_bits(xv)
    assert np.all(np.abs(hx.bf16_bits_to_f64(x)).reshape(T, 2, 128).max(axis=2) == 300.0)
    idx = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    w = np.full((T, K), 0.5, np.float32)
    blk = orc.forward(x, idx, w, W1q, np.ones((E, 2 * I // 128, H // 128), np.float32),
                      W2q, np.ones((E, H // 128, I // 128), np.float32))
    pt = orc.forward_pt(x, idx, w, W1q, np.ones(E, np.float32), W2q, np.ones(E, np.float32),
                        1.0, 1.0)
    assert np.all(blk["xs"] == 1.0)
    assert np.array_equal(blk["xq"], pt["xq"])
    assert np.array_equal(blk["gu"], pt["gu"])


def test_pt_double_x_and_its_scale(orc):
    T, H, I, E, K = 12, 256, 128, 3, 2
    x, idx, w, w1, w2 = rand_problem(T, H, I, E, K, seed=66)
    wq = orc.quant_weights_pt(w1) + orc.quant_weights_pt(w2)
    sx, sh = F32(6.0 / 448.0), F32(4.0 / 448.0)
    a = orc.forward_pt(x, idx, w, *wq, sx, sh)
    x2 = hx.f64_to_bf16_bits(hx.bf16_bits_to_f64(x) * 2.0)
    b = orc.forward_pt(x2, idx, w, *wq, F32(2.0) * sx, sh)
    assert np.array_equal(a["xq"], b["xq"])
    assert np.array_equal(hx.bf16_bits_to_f64(a["gu"]) * 2.0, hx.bf16_bits_to_f64(b["gu"]))


def test_pt_token_permutation_permutes_output(orc):
    T, H, I, E, K = 20, 256, 128, 5, 2
    x, idx, w, w1, w2 = rand_problem(T, H, I, E, K, seed=67)
    wq = orc.quant_weights_pt(w1) + orc.quant_weights_pt(w2)
    base = orc.forward_pt(x, idx, w, *wq, F32(6.0 / 448.0), F32(8.0 / 448.0))
    p = np.random.default_rng(68).permutation(T)
    perm = orc.forward_pt(x[p], idx[p], w[p], *wq, F32(6.0 / 448.0), F32(8.0 / 448.0))
    assert np.array_equal(perm["out"], base["out"][p])
