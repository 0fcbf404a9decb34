"""GPU parity of the MXFP8 format (MOE_FLAG_MXFP8) against the oracle (fmt=1).

MXFP8: E4M3 with one power-of-two scale per 32 elements along K, for the
activations (1x32) and for every weight row.  Bars as in test_gpu_parity:
bit-exact routing, weight codes and scales, every gathered activation byte
and per-chunk scale; gate||up rel-L2 <= 1e-3; output rel-L2 <= 1e-2 and
max-abs <= 5e-2 * rms; the fused epilogue bit-equal to the unfused path; one
GEMM launch bit-equal to two.
"""
import numpy as np
import pytest
import torch

from tests import gpu_harness as gh
from tests.test_gpu_parity import check_routing, compare_outputs, gate_out, small_problem

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as ge
    ge.build()
    import serving_route_gb300 as S
    return S


def mx_layer(S, orc, T, H, I, E, K, w1, w2, **kw):
    q1, s1 = S.MegaMoELayer.quantize_weights(torch.from_numpy(w1).cuda(), fmt="mxfp8")
    q2, s2 = S.MegaMoELayer.quantize_weights(torch.from_numpy(w2).cuda(), fmt="mxfp8")
    wo = orc.quant_weights_mx(w1) + orc.quant_weights_mx(w2)
    for a, b in zip((q1, s1, q2, s2), wo):
        assert np.array_equal(a.cpu().numpy(), b)
    layer = S.MegaMoELayer(H, I, E, K, max_rows=max(T, 1), fmt="mxfp8", **kw)
    layer.bind_weights(q1, s1, q2, s2)
    return layer, wo


def check_quant_mx(S, dbg, xq, xs, perm, rows, K):
    """every routed row of A equals the oracle's 1x32-quantised token row, byte
    for byte, with its per-chunk scales"""
    if len(perm) == 0:
        return
    tok = perm // K
    a = dbg["a"][torch.from_numpy(rows).cuda()].cpu().numpy()
    assert np.array_equal(a, xq[tok])
    units = xq.shape[1] // 32
    sf = S.sf_atom_rows(dbg["a_sf"], dbg["rows_alloc"], units).cpu().numpy()[rows].astype(np.int64) - 127
    assert np.array_equal(np.ldexp(1.0, sf).astype(np.float32), xs[tok])


def test_mx_weight_quantiser_bit_exact(lib, orc):
    rng = np.random.default_rng(61)
    w = (rng.standard_normal((3, 256, 384)) * 0.03).astype(np.float32)
    w[0, 5, 32:64] = 0.0                   # all-zero chunk: scale 1
    w[1, 128:, 256:288] *= 2.0 ** 40       # large chunks
    w[2, :3, :] *= 2.0 ** -100             # tiny rows
    q, s = lib.MegaMoELayer.quantize_weights(torch.from_numpy(w).cuda(), fmt="mxfp8")
    rq, rs = orc.quant_weights_mx(w)
    assert np.array_equal(q.cpu().numpy(), rq)
    assert np.array_equal(s.cpu().numpy(), rs)


@pytest.mark.parametrize("gemm", ["single", "pair"])
@pytest.mark.parametrize("fuse", [False, True])
@pytest.mark.parametrize("T,H,I,E,K", [
    (77, 256, 384, 6, 2),       # ragged T, 3 FC1 n-tiles
    (300, 512, 256, 16, 4),
])
def test_mx_layer_parity(lib, orc, T, H, I, E, K, fuse, gemm):
    x, idx, w, w1, w2 = small_problem(orc, T, H, I, E, K, seed=62, empty=(1,))
    layer, wo = mx_layer(lib, orc, T, H, I, E, K, w1, w2, fuse_fc1=fuse, emit_fc1=True, gemm=gemm)
    ref = orc.forward(x, idx, w, *wo, fmt=1)
    assert ref["err"] == 0
    xt, it, wt = gh.to_device(x, idx, w)
    out = layer.forward(xt, it, wt)
    assert layer.read_status() == (0, 0)
    dbg = layer.debug()
    rows = check_routing(dbg, ref, T, K)
    check_quant_mx(lib, dbg, ref["xq"], ref["xs"], ref["perm"], rows, K)
    stats = compare_outputs(dbg, out, ref, rows)
    print("mxfp8", gemm, "fused" if fuse else "unfused", stats)


def test_mx_fused_bit_equal_unfused_and_one_launch_equal_split(lib, orc):
    T, H, I, E, K = 513, 768, 640, 12, 6
    x, idx, w, w1, w2 = small_problem(orc, T, H, I, E, K, seed=63)
    xt, it, wt = gh.to_device(x, idx, w)
    res = []
    for fuse, gemms in ((False, "auto"), (True, "split"), (True, "one_launch")):
        layer, wo = mx_layer(lib, orc, T, H, I, E, K, w1, w2, fuse_fc1=fuse, emit_fc1=True,
                             gemms=gemms)
        out = layer.forward(xt, it, wt).clone()
        assert layer.read_status() == (0, 0)
        d = layer.debug()
        off = d["offsets"].cpu().numpy()
        rows = torch.from_numpy(gh.padded_rows(off, d["pad_offsets"].cpu().numpy(), int(off[-1]))).cuda()
        sf = lib.sf_atom_rows(d["h_sf"], d["rows_alloc"], I // 32)[rows]
        res.append((out.view(torch.int16), d["hq"][rows], sf, d["gu"][rows].view(torch.int16),
                    d["y"][rows].view(torch.int16)))
    for other in res[1:]:
        for a, b in zip(res[0], other):
            assert torch.equal(a, b)
    ref = orc.forward(x, idx, w, *wo, fmt=1)
    gate_out(gh.bf16_np(res[0][0].view(torch.bfloat16)), gh.bits_to_f64(ref["out"]))


def test_mx_bind_rejects_non_power_of_two_scale(lib, orc):
    import serving_route_gb300.binding as B
    T, H, I, E, K = 8, 256, 128, 2, 1
    x, idx, w, w1, w2 = small_problem(orc, T, H, I, E, K, seed=64)
    q1, s1 = lib.MegaMoELayer.quantize_weights(torch.from_numpy(w1).cuda(), fmt="mxfp8")
    q2, s2 = lib.MegaMoELayer.quantize_weights(torch.from_numpy(w2).cuda(), fmt="mxfp8")
    s1[1, 7, 3] = 0.75
    layer = lib.MegaMoELayer(H, I, E, K, max_rows=T, fmt="mxfp8")
    with pytest.raises(B.MoEError):
        layer.bind_weights(q1, s1, q2, s2)


@pytest.mark.parametrize("gemms", ["split", "one_launch"])
@pytest.mark.parametrize("gemm", ["single", "pair"])
def test_mx_sm_budget_bit_identical(lib, orc, gemm, gemms):
    """Under an SM budget each GEMM CTA runs many tiles in a row: full tiles
    and expert tails whose all-padding row quadrants skip their epilogue work
    mixed in any order.  The outputs stay bit-identical to the full grid's and
    within the oracle's bars."""
    T, H, I, E, K = 513, 512, 384, 8, 6
    x, idx, w, w1, w2 = small_problem(orc, T, H, I, E, K, seed=65)
    layer, wo = mx_layer(lib, orc, T, H, I, E, K, w1, w2, fuse_fc1=True, gemm=gemm, gemms=gemms)
    xt, it, wt = gh.to_device(x, idx, w)
    full = layer.forward(xt, it, wt).clone()
    assert layer.read_status() == (0, 0)
    for budget in (2, 6, 0):
        layer.set_sm_budget(budget)
        out = layer.forward(xt, it, wt).clone()
        assert layer.read_status() == (0, 0), budget
        assert torch.equal(out.view(torch.int16), full.view(torch.int16)), budget
    ref = orc.forward(x, idx, w, *wo, fmt=1)
    dbg = layer.debug()
    compare_outputs(dbg, full, ref, check_routing(dbg, ref, T, K), check_gu=False)


@pytest.mark.parametrize("gemm", ["single", "pair"])
def test_mx_poisoned_padding_rows_change_nothing(lib, orc, gemm):
    """MXFP8: NaN codes, NaN per-chunk scales and NaN BF16 in every padding
    row between two forwards leave the output bit-identical."""
    T, H, I, E, K = 300, 512, 384, 8, 4
    x, idx, w, w1, w2 = small_problem(orc, T, H, I, E, K, seed=72)
    layer, wo = mx_layer(lib, orc, T, H, I, E, K, w1, w2, fuse_fc1=True, gemm=gemm, gemms="one_launch")
    xt, it, wt = gh.to_device(x, idx, w)
    first = layer.forward(xt, it, wt).clone()
    assert layer.read_status() == (0, 0)
    assert gh.poison_padding(layer) > 0
    again = layer.forward(xt, it, wt)
    assert layer.read_status() == (0, 0)
    assert torch.equal(again.view(torch.int16), first.view(torch.int16))
    ref = orc.forward(x, idx, w, *wo, fmt=1)
    dbg = layer.debug()
    compare_outputs(dbg, again, ref, check_routing(dbg, ref, T, K), check_gu=False)
