"""GPU parity of the token-as-N ("swap-AB") GEMMs of small forwards.

A forward of at most 64 tokens on the single-CTA tactic runs its GEMMs with
the weights as the M = 128 operand and the first 16, 32 or 64 rows of each
expert segment as the N operand (the small-M swap-AB variant flashinfer PR
#4069 lists under Limitations, with the token tiles PR #4688 picks per token
bucket).  Bars as in test_gpu_parity: bit-exact routing and activation
bytes; gate||up rel-L2 <= 1e-3 against the oracle; output rel-L2 <= 1e-2 and
max-abs <= 5e-2 * rms; the fused epilogue bit-equal to the unfused path and
one launch bit-equal to two, within the token-as-N kernels; the combine
folded into the token-as-N FC2 (opt-in) bit-equal to the combine kernel; the
plan reports the tile and the fold; NaN-poisoned padding rows change nothing.
"""
import numpy as np
import pytest
import torch

from gen import configs
from tests import gpu_harness as gh
from tests.test_gpu_parity import (check_quant, check_routing, compare_outputs, gate_out,
                                   small_problem)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as ge
    ge.build()
    import serving_route_gb300 as S
    return S


def make(S, orc, T, H, I, E, K, w1, w2, fmt="deepseek", **kw):
    q1, s1 = S.MegaMoELayer.quantize_weights(torch.from_numpy(w1).cuda(), fmt=fmt)
    q2, s2 = S.MegaMoELayer.quantize_weights(torch.from_numpy(w2).cuda(), fmt=fmt)
    quant = {"mxfp8": orc.quant_weights_mx, "per_tensor": orc.quant_weights_pt}.get(fmt, orc.quant_weights)
    wo = quant(w1) + quant(w2)
    layer = S.MegaMoELayer(H, I, E, K, max_rows=T, gemm="single", fmt=fmt, **kw)
    layer.bind_weights(q1, s1, q2, s2)
    if fmt == "per_tensor":
        layer.set_activation_scales(float(configs.PT_X_SCALE), float(configs.PT_H_SCALE))
    return layer, wo


def oracle(orc, fmt, x, idx, w, wo):
    if fmt == "per_tensor":
        return orc.forward_pt(x, idx, w, *wo, configs.PT_X_SCALE, configs.PT_H_SCALE)
    return orc.forward(x, idx, w, *wo, fmt=1 if fmt == "mxfp8" else 0)


@pytest.mark.parametrize("T,H,I,E,K,empty", [
    (1, 256, 128, 4, 1, ()),            # one token: tile 16, one live column
    (8, 512, 256, 64, 8, ()),           # decode-like: one row per touched expert
    (16, 384, 256, 6, 2, (2,)),         # tile 16 full; H % 256 == 128: FC2's last unit is half
    (17, 256, 384, 4, 2, ()),           # tile 32, ragged; three FC1 units per m-tile
    (40, 512, 256, 8, 4, (1, 5)),       # tile 64, empty experts
    (64, 768, 512, 3, 1, ()),           # tile 64 full in every expert
])
@pytest.mark.parametrize("fuse", [False, True])
def test_swap_layer_parity(lib, orc, T, H, I, E, K, empty, fuse):
    x, idx, w, w1, w2 = small_problem(orc, T, H, I, E, K, seed=80 + T, empty=empty)
    layer, wo = make(lib, orc, T, H, I, E, K, w1, w2, fuse_fc1=fuse, emit_fc1=True)
    tile = layer.plan(T)["swap_ab_tokens"]
    assert tile == (16 if T <= 16 else 32 if T <= 32 else 64)
    ref = oracle(orc, "deepseek", x, idx, w, wo)
    xt, it, wt = gh.to_device(x, idx, w)
    out = layer.forward(xt, it, wt)
    assert layer.read_status() == (0, 0)
    dbg = layer.debug()
    rows = check_routing(dbg, ref, T, K)
    check_quant(lib, dbg, ref["xq"], ref["xs"], ref["perm"], rows, K)
    stats = compare_outputs(dbg, out, ref, rows, check_gu=True)
    print("swap", T, H, I, E, K, tile, "fused" if fuse else "unfused", stats)


@pytest.mark.parametrize("fmt", ["mxfp8", "per_tensor"])
@pytest.mark.parametrize("T", [8, 33])
def test_swap_formats(lib, orc, fmt, T):
    H, I, E, K = 512, 384, 8, 4
    x, idx, w, w1, w2 = small_problem(orc, T, H, I, E, K, seed=90 + T)
    layer, wo = make(lib, orc, T, H, I, E, K, w1, w2, fmt=fmt, fuse_fc1=True, emit_fc1=True)
    assert layer.plan(T)["swap_ab_tokens"] > 0
    ref = oracle(orc, fmt, x, idx, w, wo)
    xt, it, wt = gh.to_device(x, idx, w)
    out = layer.forward(xt, it, wt)
    assert layer.read_status() == (0, 0)
    dbg = layer.debug()
    rows = check_routing(dbg, ref, T, K)
    stats = compare_outputs(dbg, out, ref, rows, check_gu=True)
    print("swap", fmt, T, stats)


@pytest.mark.parametrize("T", [12, 48])
def test_swap_fused_bit_equal_unfused_and_one_launch_equal_split(lib, orc, T):
    H, I, E, K = 768, 512, 16, 8
    x, idx, w, w1, w2 = small_problem(orc, T, H, I, E, K, seed=100 + T, mask=0.1)
    xt, it, wt = gh.to_device(x, idx, w)
    res = {}
    for name, kw in (("unfused", dict(fuse_fc1=False)),
                     ("split", dict(fuse_fc1=True, gemms="split")),
                     ("one_launch", dict(fuse_fc1=True, gemms="one_launch"))):
        layer, wo = make(lib, orc, T, H, I, E, K, w1, w2, **kw)
        assert layer.plan(T)["swap_ab_tokens"] > 0
        out = layer.forward(xt, it, wt).clone()
        assert layer.read_status() == (0, 0)
        d = layer.debug()
        off = d["offsets"].cpu().numpy()
        rows = torch.from_numpy(gh.padded_rows(off, d["pad_offsets"].cpu().numpy(), int(off[-1]))).cuda()
        sf = lib.sf_atom_rows(d["h_sf"], d["rows_alloc"], I // 128)[rows]
        res[name] = (out.view(torch.int16), d["hq"][rows].clone(), sf.clone(),
                     d["y"][rows].view(torch.int16).clone())
        del layer
    for a, b in zip(res["unfused"], res["split"]):
        assert torch.equal(a, b)
    for a, b in zip(res["split"], res["one_launch"]):
        assert torch.equal(a, b)
    ref = orc.forward(x, idx, w, *wo)
    gate_out(gh.bf16_np(res["split"][0].view(torch.bfloat16)), gh.bits_to_f64(ref["out"]))


def test_swap_agrees_with_the_m128_kernel(lib, orc):
    """Same forward through the token-as-N kernels and the M128 x N256 kernel
    (MOE_FLAG_NO_SWAP_AB): both within the oracle's bars, and close to each
    other (their FP32 accumulation orders need not be the same)."""
    T, H, I, E, K = 24, 1024, 512, 32, 8
    x, idx, w, w1, w2 = small_problem(orc, T, H, I, E, K, seed=111)
    xt, it, wt = gh.to_device(x, idx, w)
    outs = []
    for swap in (True, False):
        layer, wo = make(lib, orc, T, H, I, E, K, w1, w2, fuse_fc1=True, swap_ab=swap)
        assert (layer.plan(T)["swap_ab_tokens"] > 0) == swap
        outs.append(gh.bf16_np(layer.forward(xt, it, wt)))
        assert layer.read_status() == (0, 0)
        del layer
    ref = gh.bits_to_f64(orc.forward(x, idx, w, *wo)["out"])
    for o in outs:
        gate_out(o, ref)
    assert gh.rel_l2(outs[0], outs[1]) <= 2e-3
    print("swap vs m128 bit-identical:", np.array_equal(outs[0], outs[1]))


def test_swap_plan(lib, orc):
    H, I, E, K = 256, 128, 8, 2
    for T, want in ((1, 16), (16, 16), (17, 32), (32, 32), (33, 64), (64, 64), (65, 0), (300, 0)):
        layer = lib.MegaMoELayer(H, I, E, K, max_rows=max(T, 1), gemm="single")
        assert layer.plan(T)["swap_ab_tokens"] == want, T
    assert lib.MegaMoELayer(H, I, E, K, max_rows=8, gemm="pair").plan(8)["swap_ab_tokens"] == 0
    assert lib.MegaMoELayer(H, I, E, K, max_rows=8, swap_ab=False).plan(8)["swap_ab_tokens"] == 0


@pytest.mark.parametrize("fuse", [False, True])
def test_swap_poisoned_padding_rows_change_nothing(lib, orc, fuse):
    """Rows of an expert segment past its routed rows (inside the token tile)
    hold NaN codes, NaN scales and NaN BF16 between two forwards: the output
    is bit-identical (every token column is computed on its own)."""
    T, H, I, E, K = 20, 512, 256, 8, 2
    x, idx, w, w1, w2 = small_problem(orc, T, H, I, E, K, seed=120)
    layer, wo = make(lib, orc, T, H, I, E, K, w1, w2, fuse_fc1=fuse, emit_fc1=not fuse)
    xt, it, wt = gh.to_device(x, idx, w)
    first = layer.forward(xt, it, wt).clone()
    assert layer.read_status() == (0, 0)
    assert gh.poison_padding(layer) > 0
    second = layer.forward(xt, it, wt)
    assert layer.read_status() == (0, 0)
    assert torch.equal(first.view(torch.int16), second.view(torch.int16))


@pytest.mark.parametrize("T,H,I,E,K,mask,fmt,gemms", [
    (1, 256, 128, 4, 1, 0.0, "deepseek", "auto"),         # one token
    (8, 512, 256, 64, 8, 0.0, "deepseek", "one_launch"),  # decode-like, FC1 -> FC2 in one launch
    (20, 384, 256, 6, 2, 0.3, "deepseek", "split"),       # masked slots (some all-masked tokens); H % 256 == 128
    (40, 768, 256, 16, 6, 0.1, "mxfp8", "auto"),
    (64, 512, 384, 8, 8, 0.05, "per_tensor", "auto"),     # tile 64, every expert's rows up to the tile
])
def test_swap_folded_combine_bit_equal_combine_kernel(lib, orc, T, H, I, E, K, mask, fmt, gemms):
    """The token-as-N FC2 with the combine folded in (per token and n-tile
    completion counts; the completing warp combines) against the same
    forward with the separate combine kernel: the output bit for bit, and
    against the oracle."""
    x, idx, w, w1, w2 = small_problem(orc, T, H, I, E, K, seed=130 + T, mask=mask)
    if mask:
        idx[T // 2] = -1                 # a token with no route: +0 either way
    xt, it, wt = gh.to_device(x, idx, w)
    outs = []
    for fold in (True, False):
        layer, wo = make(lib, orc, T, H, I, E, K, w1, w2, fmt=fmt, fuse_fc1=True, gemms=gemms,
                         combine_in_fc2=fold)
        p = layer.plan(T)
        assert p["swap_ab_tokens"] > 0 and p["combine_in_fc2"] == (1 if fold else 0)
        assert p["kernels"] == p["route_kernels"] + 1 + p["gemm_launches"] + (0 if fold else 1)
        for _ in range(2):               # twice: the counters restart from zero
            out = layer.forward(xt, it, wt).clone()
            assert layer.read_status() == (0, 0)
        outs.append(out.view(torch.int16))
        del layer
    assert torch.equal(outs[0], outs[1])
    ref = oracle(orc, fmt, x, idx, w, wo)
    gate_out(gh.bf16_np(outs[0].view(torch.bfloat16)), gh.bits_to_f64(ref["out"]))
    if mask:
        assert not torch.any(outs[0][T // 2])
