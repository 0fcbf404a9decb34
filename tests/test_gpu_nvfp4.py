"""GPU: NVFP4 checkpoint weights through the one-time requantization into the
128x128 FP8 format (flashinfer PR #4069, Reviewer notes), then the layer.

* moe_requantize_weights_nvfp4 against the oracle's requant_nvfp4, bit for
  bit: E4M3 codes and power-of-two scales, with float-subnormal values, an
  all-zero block and negative zeros among the inputs.
* A whole layer whose W1 and W2 come from NVFP4 matrices: the requantized
  weights bind as any 128x128 weights, and the forward meets the oracle's
  bars on the oracle's requantized weights (output rel-L2 <= 1e-2 and
  max-abs <= 5e-2 * rms, gate||up rel-L2 <= 1e-3).
"""
import numpy as np
import pytest
import torch

from tests import gpu_harness as gh
from tests.test_gpu_parity import gate_out, small_problem

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as ge
    ge.build()
    import serving_route_gb300 as S
    return S


def random_nvfp4(rng, nmat, rows, cols, g):
    """codes [nmat, rows, cols/2] (even column low), E4M3 block scales of
    magnitude 0.5 .. 1.9, the given global scales"""
    nibs = rng.integers(0, 16, size=(nmat, rows, cols)).astype(np.uint8)
    codes = (nibs[..., 0::2] | (nibs[..., 1::2] << 4)).astype(np.uint8)
    sblk = rng.integers(0x30, 0x40, size=(nmat, rows, cols // 16)).astype(np.uint8)
    return codes, sblk, np.asarray(g, np.float32)


def gpu_requant(S, codes, sblk, g):
    t = [torch.from_numpy(a).cuda() for a in (codes, sblk, g)]
    q, s = S.MegaMoELayer.requantize_weights_nvfp4(*t)
    torch.cuda.synchronize()
    return q.cpu().numpy(), s.cpu().numpy()


def test_requant_bit_exact(lib, orc):
    rng = np.random.default_rng(81)
    codes, sblk, g = random_nvfp4(rng, 3, 256, 384, [0.0173, 2.0e-40, 3.5])
    codes[1, :128, :64] = 0                               # an all-zero 128x128 block: scale 1
    codes[2, 5, :8] = 0x88                                # negative zeros
    sblk[2, 7, 3] = 0x00                                  # a zero block scale
    sblk[0, 9, 1] = 0x05                                  # a subnormal block scale
    q, s = gpu_requant(lib, codes, sblk, g)
    q_ref, s_ref = orc.requant_nvfp4(codes, sblk, g)
    assert np.array_equal(s, s_ref)
    assert np.array_equal(q, q_ref)
    assert s[1, 0, 0] == 1.0 and not np.any(q[1, :128, :128])
    assert np.all(q[2, 5, :16] == 0x80)


@pytest.mark.parametrize("T,H,I,E,K", [(200, 256, 256, 4, 2), (300, 512, 384, 8, 4)])
def test_layer_from_nvfp4_weights(lib, orc, T, H, I, E, K):
    rng = np.random.default_rng(82 + T)
    x, idx, w, _, _ = small_problem(orc, T, H, I, E, K, seed=83 + T)
    c1, s1, g1 = random_nvfp4(rng, E, 2 * I, H, 0.5 / np.sqrt(H) * (1 + rng.random(E)))
    c2, s2, g2 = random_nvfp4(rng, E, H, I, 0.5 / np.sqrt(I) * (1 + rng.random(E)))
    wo = orc.requant_nvfp4(c1, s1, g1) + orc.requant_nvfp4(c2, s2, g2)
    t = [torch.from_numpy(a).cuda() for a in (c1, s1, g1, c2, s2, g2)]
    q1, sc1 = lib.MegaMoELayer.requantize_weights_nvfp4(*t[:3])
    q2, sc2 = lib.MegaMoELayer.requantize_weights_nvfp4(*t[3:])
    for a, b in zip((q1, sc1, q2, sc2), wo):
        assert np.array_equal(a.cpu().numpy(), b)
    layer = lib.MegaMoELayer(H, I, E, K, max_rows=T, fuse_fc1=False, emit_fc1=True)
    layer.bind_weights(q1, sc1, q2, sc2)
    out = layer.forward(*gh.to_device(x, idx, w))
    assert layer.read_status() == (0, 0)
    ref = orc.forward(x, idx, w, *wo)
    gate_out(gh.bf16_np(out), gh.bits_to_f64(ref["out"]))
    d = layer.debug()
    rows = gh.padded_rows(ref["offsets"], d["pad_offsets"].cpu().numpy(), len(ref["perm"]))
    gu = gh.bf16_np(d["gu"][torch.from_numpy(rows).cuda()])
    assert gh.rel_l2(gu, gh.bits_to_f64(ref["gu"])) <= 1e-3
