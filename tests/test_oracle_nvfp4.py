"""Pins of the oracle's NVFP4 checkpoint path (CPU only).

flashinfer PR #4069 (Reviewer notes) runs NVFP4 checkpoints on its FP8
backend through a one-time requantization.  Here an NVFP4 matrix [rows, cols]
is E2M1 codes packed two per byte along the columns (even column in the low
nibble), one E4M3 scale per 16 columns of a row and one float scale per
matrix; value = e2m1 * e4m3(block scale) * global, rounded to float once; the
requantization is the 128x128 weight quantiser applied to those values.

* E2M1 decode against the format's published value table (0, 0.5, 1, 1.5, 2,
  3, 4, 6 and their negatives, -0 for code 8).
* The packing order on a hand-built row.
* Dequantisation against numpy float32 products of the decoded factors
  (IEEE round-to-nearest), bit for bit, including float subnormals.
* With power-of-two block scales and global scale (a ratio of at most 2^4
  inside each 128x128 block) every NVFP4 value is an E4M3 value times the
  block's power-of-two scale, so the requantization must be lossless.
"""
import numpy as np

from tests import helpers_exact as hx

F32 = np.float32
E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]   # codes 0..7; 8..15 are their negatives


def e2m1_np(nib: np.ndarray) -> np.ndarray:
    mag = np.asarray(E2M1_TABLE, dtype=np.float32)[nib & 7]
    return np.where(nib & 8, -mag, mag).astype(np.float32)


def pack(nibs: np.ndarray) -> np.ndarray:
    """[..., cols] nibbles -> [..., cols/2] bytes, the even column low"""
    return (nibs[..., 0::2] | (nibs[..., 1::2] << 4)).astype(np.uint8)


def test_e2m1_table(orc):
    for c in range(16):
        v = orc.e2m1_decode(c)
        want = E2M1_TABLE[c & 7] * (-1.0 if c & 8 else 1.0)
        assert v == want, (c, v)
        assert np.signbit(v) == bool(c & 8), c          # code 8 is -0


def test_packing_order(orc):
    one = 0x38                                          # E4M3 1.0
    assert hx.e4m3_values()[one] == 1.0
    row = np.array([0x21, 0x43, 0xF8, 0x0C] + [0] * 4, np.uint8).reshape(1, 1, 8)
    sblk = np.full((1, 1, 1), one, np.uint8)
    out = orc.dequant_nvfp4(row, sblk, np.ones(1, np.float32))[0, 0]
    want = np.array([0.5, 1, 1.5, 2, -0.0, -6, -2, 0] + [0] * 8, np.float32)
    assert np.array_equal(out, want) and np.signbit(out[4])


def test_dequant_equals_float32_products(orc):
    rng = np.random.default_rng(71)
    nmat, rows, cols = 3, 128, 256
    nibs = rng.integers(0, 16, size=(nmat, rows, cols)).astype(np.uint8)
    codes = pack(nibs)
    sblk = rng.integers(0, 0x7F, size=(nmat, rows, cols // 16)).astype(np.uint8)  # finite, >= 0
    g = np.array([0.00731, 3.1e-41 / 6.0, 1.7], np.float32)   # the second makes float subnormals
    out = orc.dequant_nvfp4(codes, sblk, g)
    dec = hx.e4m3_values().astype(np.float32)
    s = np.repeat(dec[sblk], 16, axis=2)
    want = (e2m1_np(nibs) * s) * g[:, None, None]               # float32 products, round to nearest
    assert np.array_equal(out.view(np.uint32), want.view(np.uint32))
    assert np.any((np.abs(out[1]) < np.finfo(np.float32).tiny) & (out[1] != 0))


def test_requant_lossless_on_power_of_two_scales(orc):
    rng = np.random.default_rng(72)
    nmat, rows, cols = 2, 256, 384
    nibs = rng.integers(0, 16, size=(nmat, rows, cols)).astype(np.uint8)
    # E4M3 codes of 2^k: exponent field k + 7, mantissa 0; k in a window of 4
    # per 128x128 block, varying from one 16-column group to the next
    k0 = rng.integers(-6, 4, size=(nmat, rows // 128, cols // 128))
    k = np.repeat(np.repeat(k0, 128, axis=1), 8, axis=2) + rng.integers(0, 5, size=(nmat, rows, cols // 16))
    sblk = ((k + 7) << 3).astype(np.uint8)
    g = np.array([2.0 ** -5, 2.0 ** 3], np.float32)
    v = orc.dequant_nvfp4(pack(nibs), sblk, g)
    q, s = orc.requant_nvfp4(pack(nibs), sblk, g)
    back = hx.e4m3_values()[q].astype(np.float64) * np.repeat(np.repeat(s, 128, axis=1), 128, axis=2)
    assert np.array_equal(back, v.astype(np.float64))
