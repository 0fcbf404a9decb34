"""GPU: the combine folded into the M128 x N256 FC2 (MOE_FLAG_COMBINE_IN_FC2 on
single-CTA forwards that do not run the token-as-N GEMMs).

FC2's epilogue warps count every routed row of a stored warp tile into its
token's per-n-tile count and queue the (token, n-tile) pairs they complete;
two warps of the launch (and the epilogue warps after their last tile)
combine those 256 columns (flashinfer PR #4069, Description: the grouped
combine after FC2).  The arithmetic is the combine
kernel's, so the bar is bit-identity with the same forward run with the
combine kernel, on:

* tiny and edge shapes: H % 256 == 128 (the last n-tile's second column half
  stores nothing and is still counted), masked slots and a token with no
  route (+0 rows), empty experts, few tokens (mostly padding rows);
* both GEMM launch forms (FC1 -> FC2 in one launch, two launches), the
  unfused FC1 path, the unit-counter schedule of decode-shaped forwards,
  and the three scale formats;
* the dsv2lite workload at full size (T=4096, H=2048, I=1408, E=64, K=6);
* two forwards in a row (the counters restart from zero) and a CUDA-graph
  replay.

Each small case is also compared with the oracle (output rel-L2 <= 1e-2 and
max-abs <= 5e-2 * rms), and the plan reports the fold only without CTA pairs.
"""
import numpy as np
import pytest
import torch

from gen import configs
from tests import gpu_harness as gh
from tests.test_gpu_parity import gate_out, small_problem

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
    layer = S.MegaMoELayer(H, I, E, K, max_rows=T, gemm="single", fmt=fmt, swap_ab=False, **kw)
    layer.bind_weights(q1, s1, q2, s2)
    if fmt == "per_tensor":
        layer.set_activation_scales(float(configs.PT_X_SCALE), float(configs.PT_H_SCALE))
    return layer, wo


def oracle(orc, fmt, x, idx, w, wo):
    if fmt == "per_tensor":
        return orc.forward_pt(x, idx, w, *wo, configs.PT_X_SCALE, configs.PT_H_SCALE)
    return orc.forward(x, idx, w, *wo, fmt=1 if fmt == "mxfp8" else 0)


@pytest.mark.parametrize("T,H,I,E,K,mask,empty,fmt,gemms,fuse", [
    (128, 256, 128, 4, 2, 0.0, (), "deepseek", "one_launch", True),     # tiny
    (300, 384, 256, 6, 2, 0.3, (2,), "deepseek", "split", True),        # H % 256 == 128, masks, empty expert
    (300, 384, 256, 6, 2, 0.3, (2,), "deepseek", "one_launch", True),
    (200, 512, 384, 8, 4, 0.1, (), "deepseek", "split", False),         # unfused FC1 (gate||up + swiglu_quant)
    (9, 512, 256, 16, 4, 0.0, (), "deepseek", "auto", True),            # few tokens: mostly padding rows
    (100, 512, 256, 64, 8, 0.05, (), "deepseek", "auto", True),         # unit-counter schedule (T*K < 128*E)
    (257, 768, 256, 16, 6, 0.1, (), "mxfp8", "auto", True),
    (190, 512, 384, 8, 8, 0.05, (), "per_tensor", "split", True),
])
def test_fold_bit_equal_combine_kernel(lib, orc, T, H, I, E, K, mask, empty, fmt, gemms, fuse):
    x, idx, w, w1, w2 = small_problem(orc, T, H, I, E, K, seed=500 + T + H, mask=mask, empty=empty)
    if mask:
        idx[T // 2] = -1                     # a token with no route: +0 either way
    xt, it, wt = gh.to_device(x, idx, w)
    outs = []
    for fold in (True, False):
        layer, wo = make(lib, orc, T, H, I, E, K, w1, w2, fmt=fmt, fuse_fc1=fuse, gemms=gemms,
                         combine_in_fc2=fold)
        p = layer.plan(T)
        assert p["swap_ab_tokens"] == 0 and p["combine_in_fc2"] == (1 if fold else 0)
        assert p["kernels"] == (p["route_kernels"] + 1 + p["gemm_launches"] + p["swiglu_kernels"]
                                + (0 if fold else 1))
        for _ in range(2):                   # twice: the counters restart from zero
            out = layer.forward(xt, it, wt).clone()
            assert layer.read_status() == (0, 0)
        outs.append(out.view(torch.int16))
        del layer
    assert torch.equal(outs[0], outs[1])
    ref = oracle(orc, fmt, x, idx, w, wo)
    gate_out(gh.bf16_np(outs[0].view(torch.bfloat16)), gh.bits_to_f64(ref["out"]))
    if mask:
        assert not torch.any(outs[0][T // 2])


def test_fold_ignored_under_cta_pairs(lib, orc):
    T, H, I, E, K = 256, 256, 128, 4, 2
    x, idx, w, w1, w2 = small_problem(orc, T, H, I, E, K, seed=531)
    q1, s1 = lib.MegaMoELayer.quantize_weights(torch.from_numpy(w1).cuda())
    q2, s2 = lib.MegaMoELayer.quantize_weights(torch.from_numpy(w2).cuda())
    outs = []
    for fold in (True, False):
        layer = lib.MegaMoELayer(H, I, E, K, max_rows=T, gemm="pair", fuse_fc1=True, combine_in_fc2=fold)
        layer.bind_weights(q1, s1, q2, s2)
        assert layer.plan(T)["combine_in_fc2"] == 0
        outs.append(layer.forward(*gh.to_device(x, idx, w)).clone().view(torch.int16))
        assert layer.read_status() == (0, 0)
        del layer
    assert torch.equal(outs[0], outs[1])


def test_fold_graph_replay(lib, orc):
    """A captured forward with the fold, replayed on new routes and masks:
    equal to the eager forward with the combine kernel every time."""
    T, H, I, E, K = 160, 512, 256, 8, 4
    x, idx, w, w1, w2 = small_problem(orc, T, H, I, E, K, seed=532)
    fold, _ = make(lib, orc, T, H, I, E, K, w1, w2, fuse_fc1=True, combine_in_fc2=True)
    plain, _ = make(lib, orc, T, H, I, E, K, w1, w2, fuse_fc1=True)
    xt, it, wt = gh.to_device(x, idx, w)
    fold.forward(xt, it, wt)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, capture_error_mode="global"):
        out_g = fold.forward(xt, it, wt)
    rng = np.random.default_rng(533)
    for live in (T, 97, 1):
        idx2 = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
        idx2[live:] = -1
        it.copy_(torch.from_numpy(idx2))
        graph.replay()
        torch.cuda.synchronize()
        assert fold.read_status() == (0, 0)
        ref = plain.forward(xt, it, wt)
        assert plain.read_status() == (0, 0)
        assert torch.equal(out_g.view(torch.int16), ref.view(torch.int16)), live
        assert not torch.any(out_g[live:].view(torch.int16))


def test_fold_v2lite_full_size(lib):
    """The dsv2lite workload at full size with the fold, against the same
    forward with the combine kernel (whose output test_gpu_workloads checks
    against the oracle element by element), bit for bit, in both launch
    forms."""
    wl = configs.V2LITE
    wd = gh.device_weights(wl, lib.MegaMoELayer)
    x, idx, w = gh.host_inputs(wl)
    xt, it, wt = gh.to_device(x, idx, w)
    outs = {}
    for fold in (False, True):
        for gemms in ("auto", "split"):
            layer = lib.MegaMoELayer(wl.H, wl.I, wl.E, wl.K, max_rows=wl.T, fuse_fc1=True, gemms=gemms,
                                     combine_in_fc2=fold)
            layer.bind_weights(*wd)
            p = layer.plan(wl.T)
            assert p["combine_in_fc2"] == (1 if fold and not layer.tactic()["gemm_pair"] else 0)
            outs[(fold, gemms)] = layer.forward(xt, it, wt).clone().view(torch.int16)
            assert layer.read_status() == (0, 0)
            del layer
    base = outs[(False, "auto")]
    for k, v in outs.items():
        assert torch.equal(v, base), k
