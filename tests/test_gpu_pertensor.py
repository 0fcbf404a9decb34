"""GPU parity of the per-tensor format (MOE_FLAG_PER_TENSOR) against the oracle.

The per_tensor scale mode of flashinfer PR #4688: one FP32 scale per expert
weight matrix, one static calibrated FP32 scale per activation tensor (x and
the SwiGLU output h).  Bars as in test_gpu_parity: bit-exact routing, weight
codes and scales, every gathered activation byte (block scales all 1);
gate||up rel-L2 <= 1e-3; y and output rel-L2 <= 1e-2 and max-abs <= 5e-2 *
rms; the fused epilogue bit-equal to the unfused path; one GEMM launch
bit-equal to two; the host-side contract (scales required, validated).
"""
import numpy as np
import pytest
import torch

from gen import configs
from tests import gpu_harness as gh
from tests.test_gpu_parity import check_routing, compare_outputs, gate_out, small_problem

pytestmark = pytest.mark.gpu

SX, SH = configs.PT_X_SCALE, configs.PT_H_SCALE


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as ge
    ge.build()
    import serving_route_gb300 as S
    return S


def pt_layer(S, orc, T, H, I, E, K, w1, w2, sx=SX, sh=SH, **kw):
    q1, s1 = S.MegaMoELayer.quantize_weights(torch.from_numpy(w1).cuda(), fmt="per_tensor")
    q2, s2 = S.MegaMoELayer.quantize_weights(torch.from_numpy(w2).cuda(), fmt="per_tensor")
    wo = orc.quant_weights_pt(w1) + orc.quant_weights_pt(w2)
    for a, b in zip((q1, s1, q2, s2), wo):
        assert np.array_equal(a.cpu().numpy(), b)
    layer = S.MegaMoELayer(H, I, E, K, max_rows=max(T, 1), fmt="per_tensor", **kw)
    layer.bind_weights(q1, s1, q2, s2)
    layer.set_activation_scales(float(sx), float(sh))
    return layer, wo


def check_quant_pt(S, dbg, xq, perm, rows, K, H):
    """every routed row of A equals the oracle's per-tensor codes of its token
    row; every block scale the tensor core applies is 1 (E8M0 127)"""
    if len(perm) == 0:
        return
    a = dbg["a"][torch.from_numpy(rows).cuda()].cpu().numpy()
    assert np.array_equal(a, xq[perm // K])
    sf = S.sf_atom_rows(dbg["a_sf"], dbg["rows_alloc"], H // 128).cpu().numpy()[rows]
    assert np.all(sf == 127)


def test_pt_weight_quantiser_bit_exact(lib, orc):
    rng = np.random.default_rng(71)
    w = (rng.standard_normal((4, 256, 384)) * 0.03).astype(np.float32)
    w[1] *= 2.0 ** 40                     # a large matrix
    w[2] = 0.0                            # all zero: scale 1
    w[3, :, :128] *= 2.0 ** -60           # mixed magnitudes: tiny values flush to subnormal / 0
    q, s = lib.MegaMoELayer.quantize_weights(torch.from_numpy(w).cuda(), fmt="per_tensor")
    rq, rs = orc.quant_weights_pt(w)
    assert np.array_equal(s.cpu().numpy(), rs)
    assert np.array_equal(q.cpu().numpy(), rq)


@pytest.mark.parametrize("gemm", ["single", "pair"])
@pytest.mark.parametrize("fuse", [False, True])
@pytest.mark.parametrize("T,H,I,E,K", [
    (77, 256, 384, 6, 2),       # ragged T, 3 FC1 n-tiles, an empty expert
    (300, 512, 256, 16, 4),
])
def test_pt_layer_parity(lib, orc, T, H, I, E, K, fuse, gemm):
    x, idx, w, w1, w2 = small_problem(orc, T, H, I, E, K, seed=72, empty=(1,))
    layer, wo = pt_layer(lib, orc, T, H, I, E, K, w1, w2, fuse_fc1=fuse, emit_fc1=True, gemm=gemm)
    ref = orc.forward_pt(x, idx, w, *wo, SX, SH)
    assert ref["err"] == 0
    xt, it, wt = gh.to_device(x, idx, w)
    out = layer.forward(xt, it, wt)
    assert layer.read_status() == (0, 0)
    dbg = layer.debug()
    rows = check_routing(dbg, ref, T, K)
    check_quant_pt(lib, dbg, ref["xq"], ref["perm"], rows, K, H)
    stats = compare_outputs(dbg, out, ref, rows, check_gu=True)
    sf = lib.sf_atom_rows(dbg["h_sf"], dbg["rows_alloc"], I // 128).cpu().numpy()[rows]
    assert np.all(sf == 127)
    print("per-tensor", T, H, I, E, K, "fused" if fuse else "unfused", gemm, stats)


@pytest.mark.parametrize("gemm", ["single", "pair"])
def test_pt_fused_bit_equal_unfused_and_one_launch_equal_split(lib, orc, gemm):
    T, H, I, E, K = 520, 768, 384, 12, 6
    x, idx, w, w1, w2 = small_problem(orc, T, H, I, E, K, seed=73, mask=0.05)
    xt, it, wt = gh.to_device(x, idx, w)
    res = {}
    for name, kw in (("unfused", dict(fuse_fc1=False)),
                     ("split", dict(fuse_fc1=True, gemms="split")),
                     ("one_launch", dict(fuse_fc1=True, gemms="one_launch"))):
        layer, wo = pt_layer(lib, orc, T, H, I, E, K, w1, w2, gemm=gemm, **kw)
        out = layer.forward(xt, it, wt).clone()
        assert layer.read_status() == (0, 0)
        d = layer.debug()
        off = d["offsets"].cpu().numpy()
        rows = torch.from_numpy(gh.padded_rows(off, d["pad_offsets"].cpu().numpy(), int(off[-1]))).cuda()
        res[name] = (out.view(torch.int16), d["hq"][rows].clone(), d["y"][rows].view(torch.int16).clone())
        del layer
    for a, b in zip(res["unfused"], res["split"]):
        assert torch.equal(a, b)
    for a, b in zip(res["split"], res["one_launch"]):
        assert torch.equal(a, b)
    ref = orc.forward_pt(x, idx, w, *wo, SX, SH)
    gate_out(gh.bf16_np(res["split"][0].view(torch.bfloat16)), gh.bits_to_f64(ref["out"]))


def test_pt_saturating_activation_scale(lib, orc):
    """A calibrated x scale that is too small saturates codes at +-448 on both
    sides identically (bytes bit-exact); the layer still matches the oracle
    that saturates the same way."""
    T, H, I, E, K = 64, 256, 256, 4, 2
    x, idx, w, w1, w2 = small_problem(orc, T, H, I, E, K, seed=74)
    sx = np.float32(1.0 / 448.0)          # |x| > 1 saturates
    layer, wo = pt_layer(lib, orc, T, H, I, E, K, w1, w2, sx=sx, fuse_fc1=True, emit_fc1=True)
    ref = orc.forward_pt(x, idx, w, *wo, sx, SH)
    assert np.sum((ref["xq"] & 0x7F) == 0x7E) > 1000
    xt, it, wt = gh.to_device(x, idx, w)
    out = layer.forward(xt, it, wt)
    assert layer.read_status() == (0, 0)
    dbg = layer.debug()
    rows = check_routing(dbg, ref, T, K)
    check_quant_pt(lib, dbg, ref["xq"], ref["perm"], rows, K, H)
    compare_outputs(dbg, out, ref, rows, check_gu=True)


def test_pt_scales_change_between_graph_replays(lib, orc):
    """The kernels read the activation scales from the weight store, so a new
    moe_set_activation_scales takes effect in the next replay of a captured
    forward."""
    T, H, I, E, K = 96, 256, 256, 4, 2
    x, idx, w, w1, w2 = small_problem(orc, T, H, I, E, K, seed=75)
    layer, wo = pt_layer(lib, orc, T, H, I, E, K, w1, w2, fuse_fc1=True)
    xt, it, wt = gh.to_device(x, idx, w)
    layer.forward(xt, it, wt)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            layer.forward(xt, it, wt, stream=s)
    for sx, sh in ((SX, SH), (np.float32(4.0 / 448.0), np.float32(12.0 / 448.0))):
        layer.set_activation_scales(float(sx), float(sh))
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        ref = orc.forward_pt(x, idx, w, *wo, sx, sh)
        gate_out(gh.bf16_np(layer.out[:T]), gh.bits_to_f64(ref["out"]))


def test_pt_host_contract(lib, orc):
    import serving_route_gb300.binding as B
    T, H, I, E, K = 32, 256, 256, 4, 2
    x, idx, w, w1, w2 = small_problem(orc, T, H, I, E, K, seed=76)
    q1, s1 = lib.MegaMoELayer.quantize_weights(torch.from_numpy(w1).cuda(), fmt="per_tensor")
    q2, s2 = lib.MegaMoELayer.quantize_weights(torch.from_numpy(w2).cuda(), fmt="per_tensor")
    layer = lib.MegaMoELayer(H, I, E, K, max_rows=T, fmt="per_tensor")
    layer.bind_weights(q1, s1, q2, s2)
    xt, it, wt = gh.to_device(x, idx, w)
    st = B.moe_forward_status(layer.handle, xt.data_ptr(), it.data_ptr(), wt.data_ptr(), T,
                              torch.cuda.current_stream().cuda_stream)
    assert st == B.MOE_ERR_NOT_BOUND                    # no activation scales yet
    for bad in ((0.0, 1.0), (1.0, -1.0), (float("nan"), 1.0), (1.0, float("inf"))):
        with pytest.raises(B.MoEError) as ei:
            layer.set_activation_scales(*bad)
        assert ei.value.status == B.MOE_ERR_INVALID_ARG
    layer.set_activation_scales(float(SX), float(SH))
    layer.forward(xt, it, wt)
    assert layer.read_status() == (0, 0)
    # a weight scale that is not positive and finite is refused at bind
    bad1 = s1.clone()
    bad1[2] = 0.0
    with pytest.raises(B.MoEError) as ei:
        layer.bind_weights(q1, bad1, q2, s2)
    assert ei.value.status == B.MOE_ERR_BAD_SCALE
    # block-scaled layers have no activation scales; MXFP8 and per-tensor do not combine
    ds = lib.MegaMoELayer(H, I, E, K, max_rows=T)
    with pytest.raises(B.MoEError) as ei:
        ds.set_activation_scales(1.0, 1.0)
    assert ei.value.status == B.MOE_ERR_UNSUPPORTED
    with pytest.raises(B.MoEError) as ei:
        B.moe_workspace_query(H, I, E, K, B.MOE_FLAG_MXFP8 | B.MOE_FLAG_PER_TENSOR, T, T)
    assert ei.value.status == B.MOE_ERR_INVALID_ARG


def test_pt_v2lite_full_layer(lib, orc):
    """The dsv2lite workload in the per-tensor format, every output element
    against the oracle; weight codes and scales bit-exact."""
    wl = configs.V2LITE
    wd = gh.device_weights(wl, lib.MegaMoELayer, fmt="per_tensor")
    wo = gh.oracle_weights(orc, wl, fmt="per_tensor")
    for a, b in zip(wd, wo):
        assert np.array_equal(a.cpu().numpy(), b)
    x, idx, w = gh.host_inputs(wl)
    ref = orc.forward_pt(x, idx, w, *wo, SX, SH)
    xt, it, wt = gh.to_device(x, idx, w)
    layer = lib.MegaMoELayer(wl.H, wl.I, wl.E, wl.K, max_rows=wl.T, fuse_fc1=True, fmt="per_tensor")
    layer.bind_weights(*wd)
    layer.set_activation_scales(float(SX), float(SH))
    out = layer.forward(xt, it, wt)
    assert layer.read_status() == (0, 0)
    dbg = layer.debug()
    rows = check_routing(dbg, ref, wl.T, wl.K)
    check_quant_pt(lib, dbg, ref["xq"], ref["perm"], rows, wl.K, wl.H)
    stats = compare_outputs(dbg, out, ref, rows, check_gu=False)
    print("v2lite per-tensor", stats)
