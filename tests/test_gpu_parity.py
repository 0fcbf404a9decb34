"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Bars (written here, derived from the layer definition):
  * bit-exact: expert counts, offsets, perm, inv, the padded row map, every
    quantised FP8 byte and E8M0 scale of the gathered activations, and the
    library's FP8 weight quantiser;
  * gate||up (FC1 pre-activation, BF16 vs the oracle's BF16): rel-L2 <= 1e-3;
  * output (BF16): rel-L2 <= 1e-2 and max-abs <= 5e-2 * rms(reference);
  * fused FC1 epilogue vs the unfused path: bit-equal (hq, scales, out).
Where FP32 accumulation flips a BF16 rounding of gate||up, the re-quantised
hq may differ by one E4M3 code: the flip count is reported, not gated; the
per-route FC2 output y is gated at rel-L2 <= 1e-2 and its max-abs reported
(a flipped hq code moves one route's y by an hq ulp times a W2 column).
"""
import numpy as np
import pytest
import torch

from gen import configs, problem
from gen import inputs as g
from tests import gpu_harness as gh

pytestmark = pytest.mark.gpu

GU_TOL = 1e-3
OUT_TOL = 1e-2
MAXABS_FRAC = 5e-2


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as ge
    ge.build()
    import serving_route_gb300 as S
    assert torch.cuda.is_available()
    return S


def make_layer(S, wl, weights, max_rows=None, fuse=False, emit=True, check=True, cf=1.0,
               gemm="auto"):
    layer = S.MegaMoELayer(wl.H, wl.I, wl.E, wl.K, max_rows=max_rows or wl.T, fuse_fc1=fuse,
                           emit_fc1=emit, check_routes=check, capacity_factor=cf, gemm=gemm)
    layer.bind_weights(*weights)
    return layer


def check_routing(dbg, ref, T, K):
    R = int(ref["offsets"][-1])
    assert np.array_equal(dbg["counts"].cpu().numpy(), ref["counts"])
    assert np.array_equal(dbg["offsets"].cpu().numpy(), ref["offsets"])
    assert np.array_equal(dbg["perm"][:R].cpu().numpy(), ref["perm"])
    assert np.array_equal(dbg["inv"][:T * K].cpu().numpy(), ref["inv"])
    pad = dbg["pad_offsets"].cpu().numpy()
    # GEMM segments are padded to 128 rows (single CTA) or 256 rows (CTA pairs)
    assert any(np.array_equal(np.diff(pad), (ref["counts"] + g - 1) // g * g) for g in (128, 256))
    rows = gh.padded_rows(ref["offsets"], pad, R)
    inv_pad = dbg["inv_pad"][:T * K].cpu().numpy()
    act = ref["inv"] >= 0
    assert np.array_equal(inv_pad[act], rows[ref["inv"][act]])
    assert np.all(inv_pad[~act] == -1)
    return rows


def check_quant(S, dbg, xq, xs, perm, rows, K):
    """every routed row of A equals the oracle's quantised token row, byte for byte"""
    R = len(perm)
    if R == 0:
        return
    tok = perm // K
    a = dbg["a"][torch.from_numpy(rows).cuda()].cpu().numpy()
    assert np.array_equal(a, xq[tok])
    sf = S.sf_atom_rows(dbg["a_sf"], dbg["rows_alloc"], xq.shape[1] // 128).cpu().numpy()[rows].astype(np.int64) - 127
    assert np.array_equal(np.ldexp(1.0, sf).astype(np.float32), xs[tok])


def run_full(S, orc, wl, fuse, emit=True, weights_dev=None, weights_orc=None, gemm="auto"):
    x, idx, w = gh.host_inputs(wl)
    ref = orc.forward(x, idx, w, *weights_orc)
    assert ref["err"] == 0
    layer = make_layer(S, wl, weights_dev, fuse=fuse, emit=emit, gemm=gemm)
    xt, it, wt = gh.to_device(x, idx, w)
    out = layer.forward(xt, it, wt)
    st, bits = layer.read_status()
    assert st == 0 and bits == 0, (st, bits)
    return layer, layer.debug(), out, ref, x, idx, w


def gate_out(o: np.ndarray, r: np.ndarray, what="out") -> dict:
    """The output bar: rel-L2 <= 1e-2 and max-abs <= 5e-2 * rms(reference)."""
    rel = gh.rel_l2(o, r)
    rms = float(np.sqrt(np.mean(r * r))) if r.size else 0.0
    mx = float(np.max(np.abs(o - r))) if r.size else 0.0
    assert rel <= OUT_TOL, (what, rel)
    assert mx <= MAXABS_FRAC * rms + 1e-30, (what, mx, rms)
    return {f"{what}_rel_l2": rel, f"{what}_maxabs": mx}


def compare_outputs(dbg, out, ref, rows, check_gu=True):
    R = len(rows)
    stats = {}
    if check_gu and "gu" in dbg and R:
        gu = gh.bf16_np(dbg["gu"][torch.from_numpy(rows).cuda()])
        stats["gu_rel_l2"] = gh.rel_l2(gu, gh.bits_to_f64(ref["gu"]))
        assert stats["gu_rel_l2"] <= GU_TOL, stats
    if R:
        hq = dbg["hq"][torch.from_numpy(rows).cuda()].cpu().numpy()
        stats["hq_code_flips"] = int(np.sum(hq != ref["hq"]))
        # y (FC2 output per route, BF16): the output's rel-L2 bar.  Its
        # max-abs is reported, not gated: one E4M3 code flip of hq (where the
        # FP32 accumulation flips a BF16 rounding of gate||up) moves a single
        # route's y by up to one hq ulp times its W2 column, which the
        # top-k combine then averages; the max-abs bar is the combined
        # output's, gated below
        y = gh.bf16_np(dbg["y"][torch.from_numpy(rows).cuda()])
        yr = gh.bits_to_f64(ref["y"])
        stats["y_rel_l2"] = gh.rel_l2(y, yr)
        stats["y_maxabs"] = float(np.max(np.abs(y - yr)))
        assert stats["y_rel_l2"] <= OUT_TOL, stats
    o = gh.bf16_np(out)
    r = gh.bits_to_f64(ref["out"])
    stats["out_rel_l2"] = gh.rel_l2(o, r)
    rms = float(np.sqrt(np.mean(r * r))) if r.size else 0.0
    stats["out_maxabs"] = float(np.max(np.abs(o - r))) if r.size else 0.0
    assert stats["out_rel_l2"] <= OUT_TOL, stats
    assert stats["out_maxabs"] <= MAXABS_FRAC * rms + 1e-30, (stats, rms)
    return stats


# ----------------------------------------------------------------------------
# generator and weight quantiser
# ----------------------------------------------------------------------------
def test_device_generator_matches_host(lib):
    n = 1 << 20
    d = torch.empty(n, dtype=torch.float32, device="cuda")
    g.dev_normal_f32(0, g.STREAM_W1, 12345, n, g.weight_sigma(7168), d.data_ptr(),
                     torch.cuda.current_stream().cuda_stream)
    h = g.host_normal_f32(0, g.STREAM_W1, 12345, n, g.weight_sigma(7168))
    assert np.array_equal(d.cpu().numpy().view(np.uint32), h.view(np.uint32))
    b = torch.empty(n, dtype=torch.int16, device="cuda")
    g.dev_normal_bf16(3, g.STREAM_X, 777, n, b.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert np.array_equal(b.cpu().numpy().view(np.uint16), g.host_normal_bf16(3, g.STREAM_X, 777, n))


def test_weight_quantiser_bit_exact(lib, orc):
    S = lib
    rng = np.random.default_rng(7)
    w = (rng.standard_normal((3, 256, 384)) * 0.03).astype(np.float32)
    w[1, :128, :128] = 0.0                     # all-zero block: scale 1
    w[2, 128:, 256:] *= 2.0 ** 40              # large block
    w[0, 128:, :128] *= 2.0 ** -100            # tiny block
    q, s = S.MegaMoELayer.quantize_weights(torch.from_numpy(w).cuda())
    rq, rs = orc.quant_weights(w)
    assert np.array_equal(q.cpu().numpy(), rq)
    assert np.array_equal(s.cpu().numpy(), rs)


# ----------------------------------------------------------------------------
# tiny workload: whole-layer oracle comparison, fused and unfused
# ----------------------------------------------------------------------------
@pytest.fixture(scope="module")
def tiny(lib, orc):
    wl = configs.TINY
    return wl, gh.device_weights(wl, lib.MegaMoELayer), gh.oracle_weights(orc, wl)


def test_tiny_weights_match_oracle_quantiser(lib, tiny):
    wl, wd, wo = tiny
    for a, b in zip(wd, wo):
        assert np.array_equal(a.cpu().numpy(), b)


@pytest.mark.parametrize("gemm", ["single", "pair"])
@pytest.mark.parametrize("fuse", [False, True])
def test_tiny_layer_parity(lib, orc, tiny, fuse, gemm):
    wl, wd, wo = tiny
    layer, dbg, out, ref, x, idx, w = run_full(lib, orc, wl, fuse, True, wd, wo, gemm=gemm)
    rows = check_routing(dbg, ref, wl.T, wl.K)
    check_quant(lib, dbg, ref["xq"], ref["xs"], ref["perm"], rows, wl.K)
    stats = compare_outputs(dbg, out, ref, rows)
    print("tiny", gemm, "fused" if fuse else "unfused", stats)


def test_fused_epilogue_bit_equal_unfused(lib, orc, tiny):
    """Routed rows only: padded GEMM rows hold whatever the workspace held."""
    wl, wd, _ = tiny
    x, idx, w = gh.host_inputs(wl)
    xt, it, wt = gh.to_device(x, idx, w)
    res = []
    for fuse in (False, True):
        layer = make_layer(lib, wl, wd, fuse=fuse, emit=True)
        out = layer.forward(xt, it, wt).clone()
        d = layer.debug()
        off = d["offsets"].cpu().numpy()
        rows = torch.from_numpy(gh.padded_rows(off, d["pad_offsets"].cpu().numpy(), int(off[-1]))).cuda()
        sf = lib.sf_atom_rows(d["h_sf"], d["rows_alloc"], wl.I // 128)[rows]
        res.append((out.view(torch.int16), d["hq"][rows], sf, d["gu"][rows].view(torch.int16),
                    d["y"][rows].view(torch.int16)))
    for a, b in zip(*res):
        assert torch.equal(a, b)


# ----------------------------------------------------------------------------
# edge cases on small shapes
# ----------------------------------------------------------------------------
def small_problem(orc, T, H, I, E, K, seed, mask=0.0, empty=()):
    rng = np.random.default_rng(seed)
    x = g.normal_bf16_bits(seed, g.STREAM_X, np.arange(T * H, dtype=np.uint64)).reshape(T, H)
    pool = np.array([e for e in range(E) if e not in empty])
    idx = np.stack([rng.permutation(pool)[:K] for _ in range(T)]).astype(np.int32) if T else \
        np.zeros((0, K), np.int32)
    if mask and T:
        idx[rng.random(idx.shape) < mask] = -1
    w = (rng.random((T, K)) + 0.05).astype(np.float32)
    w1 = (rng.standard_normal((E, 2 * I, H)) / np.sqrt(H)).astype(np.float32)
    w2 = (rng.standard_normal((E, H, I)) / np.sqrt(I)).astype(np.float32)
    return x, idx, w, w1, w2


def layer_from_float(S, orc, T, H, I, E, K, w1, w2, fuse=True, emit=True, max_rows=None, cf=1.0,
                     gemm="auto", gemms="auto"):
    q1, s1 = S.MegaMoELayer.quantize_weights(torch.from_numpy(w1).cuda())
    q2, s2 = S.MegaMoELayer.quantize_weights(torch.from_numpy(w2).cuda())
    wo = orc.quant_weights(w1) + orc.quant_weights(w2)
    layer = S.MegaMoELayer(H, I, E, K, max_rows=max_rows or max(T, 1), fuse_fc1=fuse,
                           emit_fc1=emit, capacity_factor=cf, gemm=gemm, gemms=gemms)
    layer.bind_weights(q1, s1, q2, s2)
    return layer, wo


@pytest.mark.parametrize("T,H,I,E,K,mask,empty,fuse", [
    (77, 256, 384, 6, 2, 0.0, (), True),        # ragged T, odd I/128, H/256 with a half tile
    (77, 384, 256, 6, 2, 0.0, (), False),       # H % 256 == 128: FC2's last N tile is half
    (300, 512, 256, 16, 4, 0.25, (3, 7, 11), True),   # masked slots and empty experts
    (1, 256, 128, 4, 1, 0.0, (), True),         # one token, top-1
    (130, 256, 256, 64, 8, 0.1, tuple(range(40)), False),  # many empty experts, top-8
    (513, 1024, 512, 8, 6, 0.05, (), True),     # several m-tiles per expert
])
@pytest.mark.parametrize("gemm", ["single", "pair"])
def test_edge_shapes(lib, orc, T, H, I, E, K, mask, empty, fuse, gemm):
    x, idx, w, w1, w2 = small_problem(orc, T, H, I, E, K, seed=T + H, mask=mask, empty=empty)
    layer, wo = layer_from_float(lib, orc, T, H, I, E, K, w1, w2, fuse=fuse, gemm=gemm)
    ref = orc.forward(x, idx, w, *wo)
    xt, it, wt = gh.to_device(x, idx, w)
    out = layer.forward(xt, it, wt)
    st, bits = layer.read_status()
    assert st == 0 and bits == 0
    dbg = layer.debug()
    rows = check_routing(dbg, ref, T, K)
    check_quant(lib, dbg, ref["xq"], ref["xs"], ref["perm"], rows, K)
    compare_outputs(dbg, out, ref, rows)
    for e in empty:
        assert int(dbg["counts"][e].item()) == 0


def test_all_masked_and_nan_masked_weights(lib, orc):
    T, H, I, E, K = 40, 256, 256, 8, 2
    x, idx, w, w1, w2 = small_problem(orc, T, H, I, E, K, seed=5)
    layer, wo = layer_from_float(lib, orc, T, H, I, E, K, w1, w2)
    xt, it, wt = gh.to_device(x, np.full_like(idx, -1), w)
    out = layer.forward(xt, it, wt)
    assert layer.read_status() == (0, 0)
    assert torch.count_nonzero(out.view(torch.int16)).item() == 0   # +0 everywhere
    idxm = idx.copy()
    idxm[::2, 1] = -1
    wn = w.copy()
    wn[::2, 1] = np.nan
    ref = orc.forward(x, idxm, wn, *wo)
    xt, it, wt = gh.to_device(x, idxm, wn)
    out = layer.forward(xt, it, wt)
    assert layer.read_status() == (0, 0)
    compare_outputs(layer.debug(), out, ref, np.zeros(0, np.int64), check_gu=False)


@pytest.mark.parametrize("gemm", ["single", "pair"])
@pytest.mark.parametrize("fuse,gemms", [(True, "split"), (True, "one_launch"), (False, "split")])
def test_poisoned_padding_rows_change_nothing(lib, orc, gemm, fuse, gemms):
    """The padding rows of the expert segments are computed over but never
    read into a routed row: filling them with NaN codes, NaN scales and NaN
    BF16 between two forwards leaves the output bit-identical (the tensor
    core keeps rows apart; the epilogues skip all-padding quadrants; combine
    reads y through inv)."""
    T, H, I, E, K = 300, 512, 384, 8, 4
    x, idx, w, w1, w2 = small_problem(orc, T, H, I, E, K, seed=71)
    layer, wo = layer_from_float(lib, orc, T, H, I, E, K, w1, w2, fuse=fuse, gemm=gemm, gemms=gemms)
    xt, it, wt = gh.to_device(x, idx, w)
    first = layer.forward(xt, it, wt).clone()
    assert layer.read_status() == (0, 0)
    assert gh.poison_padding(layer) > 0
    again = layer.forward(xt, it, wt)
    assert layer.read_status() == (0, 0)
    assert torch.equal(again.view(torch.int16), first.view(torch.int16))
    ref = orc.forward(x, idx, w, *wo)
    dbg = layer.debug()
    compare_outputs(dbg, again, ref, check_routing(dbg, ref, T, K))


@pytest.mark.parametrize("gemm", ["single", "pair"])
def test_poisoned_empty_experts_contribute_nothing(lib, orc, gemm):
    """An expert with no route contributes nothing: with its W1 / W2 codes all
    0x7F (E4M3 NaN) the output is bit-identical to the clean weights and finite."""
    T, H, I, E, K = 200, 384, 256, 8, 2
    empty = (2, 5)
    x, idx, w, w1, w2 = small_problem(orc, T, H, I, E, K, seed=71, empty=empty)
    q1, s1 = lib.MegaMoELayer.quantize_weights(torch.from_numpy(w1).cuda())
    q2, s2 = lib.MegaMoELayer.quantize_weights(torch.from_numpy(w2).cuda())
    xt, it, wt = gh.to_device(x, idx, w)
    outs = []
    for poison in (False, True):
        a1, a2 = q1.clone(), q2.clone()
        if poison:
            for e in empty:
                a1[e].fill_(0x7F)
                a2[e].fill_(0x7F)
        layer = lib.MegaMoELayer(H, I, E, K, max_rows=T, fuse_fc1=True, gemm=gemm)
        layer.bind_weights(a1, s1, a2, s2)
        outs.append(layer.forward(xt, it, wt).clone())
        assert layer.read_status() == (0, 0)
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    assert torch.isfinite(outs[1].float()).all()


def test_route_errors_set_status(lib, orc):
    import serving_route_gb300.binding as B
    T, H, I, E, K = 16, 256, 128, 4, 2
    x, idx, w, w1, w2 = small_problem(orc, T, H, I, E, K, seed=9)
    layer, _ = layer_from_float(lib, orc, T, H, I, E, K, w1, w2)
    cases = []
    bad = idx.copy(); bad[3, 0] = E; cases.append((bad, w, B.MOE_DEV_ROUTE_RANGE))
    bad = idx.copy(); bad[4, 0] = -7; cases.append((bad, w, B.MOE_DEV_ROUTE_RANGE))
    bad = idx.copy(); bad[5, 1] = bad[5, 0]; cases.append((bad, w, B.MOE_DEV_ROUTE_DUP))
    wb = w.copy(); wb[6, 1] = np.inf; cases.append((idx, wb, B.MOE_DEV_ROUTE_NONFINITE))
    # one routing kernel, then the three-kernel form (under an SM budget)
    for budget in (0, 4):
        layer.set_sm_budget(budget)
        assert layer.route_kernels(T) == (3 if budget else 1)
        for bi, bw, bit in cases:
            xt, it, wt = gh.to_device(x, bi, bw)
            layer.forward(xt, it, wt)
            st, bits = layer.read_status()
            assert st == B.MOE_ERR_BAD_ROUTE and bits == bit, (budget, st, bits, bit)
            assert orc.route(bi, bw, E)["err"] == bit
    layer.set_sm_budget(0)
    # a clean forward clears the word again
    xt, it, wt = gh.to_device(x, idx, w)
    layer.forward(xt, it, wt)
    assert layer.read_status() == (0, 0)


def test_host_errors_and_zero_tokens(lib, orc):
    import serving_route_gb300.binding as B
    T, H, I, E, K = 8, 256, 128, 4, 2
    x, idx, w, w1, w2 = small_problem(orc, T, H, I, E, K, seed=10)
    layer, _ = layer_from_float(lib, orc, T, H, I, E, K, w1, w2)
    xt, it, wt = gh.to_device(x, idx, w)
    sp = torch.cuda.current_stream().cuda_stream
    assert B.moe_forward_status(layer.handle, xt.data_ptr(), it.data_ptr(), wt.data_ptr(), T + 1,
                                sp) == B.MOE_ERR_CAPACITY
    assert B.moe_forward_status(layer.handle, xt.data_ptr(), it.data_ptr(), wt.data_ptr(), -1,
                                sp) == B.MOE_ERR_INVALID_ARG
    before = layer.out.clone()
    assert B.moe_forward_status(layer.handle, 0, 0, 0, 0, sp) == B.MOE_OK
    torch.cuda.synchronize()
    assert torch.equal(before.view(torch.int16), layer.out.view(torch.int16))
    # unbound weights
    fresh = lib.MegaMoELayer(H, I, E, K, max_rows=T)
    assert B.moe_forward_status(fresh.handle, xt.data_ptr(), it.data_ptr(), wt.data_ptr(), T,
                                sp) == B.MOE_ERR_NOT_BOUND
    # non power-of-two scale refused at bind time
    q = torch.zeros((E, 2 * I, H), dtype=torch.uint8, device="cuda")
    s1 = torch.ones((E, 2 * I // 128, H // 128), dtype=torch.float32, device="cuda")
    q2 = torch.zeros((E, H, I), dtype=torch.uint8, device="cuda")
    s2 = torch.ones((E, H // 128, I // 128), dtype=torch.float32, device="cuda")
    s2[1, 0, 0] = 3.0
    with pytest.raises(B.MoEError) as ei:
        fresh.bind_weights(q, s1, q2, s2)
    assert ei.value.status == B.MOE_ERR_BAD_SCALE


def test_capacity_overflow_is_reported(lib, orc):
    import serving_route_gb300.binding as B
    T, H, I, E, K = 1024, 256, 128, 2, 2
    x, idx, w, w1, w2 = small_problem(orc, T, H, I, E, K, seed=11)
    # capacity for 10% of the routes (plus segment padding): 2048 routed rows overflow it
    layer, _ = layer_from_float(lib, orc, T, H, I, E, K, w1, w2, cf=0.1)
    xt, it, wt = gh.to_device(x, idx, w)
    layer.forward(xt, it, wt)
    st, bits = layer.read_status()
    assert st == B.MOE_ERR_CAPACITY and bits == B.MOE_DEV_CAPACITY


def test_cuda_graph_replay_with_tail_masking(lib, orc):
    T, H, I, E, K = 96, 512, 256, 8, 2
    x, idx, w, w1, w2 = small_problem(orc, T, H, I, E, K, seed=12)
    layer, wo = layer_from_float(lib, orc, T, H, I, E, K, w1, w2, fuse=True, emit=False)
    xt, it, wt = gh.to_device(x, idx, w)
    layer.forward(xt, it, wt)        # warm-up outside capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s, capture_error_mode="global"):
            layer.forward(xt, it, wt, stream=s)
    for live in (T, 50, 1):
        idx2 = idx.copy()
        idx2[live:] = -1                                   # tail masking
        it.copy_(torch.from_numpy(idx2).cuda())
        graph.replay()
        torch.cuda.synchronize()
        ref = orc.forward(x, idx2, w, *wo)
        o = gh.bf16_np(layer.out[:T])
        r = gh.bits_to_f64(ref["out"])
        gate_out(o, r)
        assert np.all(o[live:] == 0)
    # a replay observes the routing checker on the rebound inputs
    idx3 = idx.copy()
    idx3[0, 0] = E + 3
    it.copy_(torch.from_numpy(idx3).cuda())
    graph.replay()
    st, bits = layer.read_status(stream=s)
    assert bits & 0x1


def test_token_permutation_and_pow2_weight_scaling(lib, orc):
    T, H, I, E, K = 64, 256, 256, 8, 2
    x, idx, w, w1, w2 = small_problem(orc, T, H, I, E, K, seed=13)
    layer, _ = layer_from_float(lib, orc, T, H, I, E, K, w1, w2)
    xt, it, wt = gh.to_device(x, idx, w)
    base = layer.forward(xt, it, wt).clone()
    p = np.random.default_rng(1).permutation(T)
    xt2, it2, wt2 = gh.to_device(x[p], idx[p], w[p])
    perm_out = layer.forward(xt2, it2, wt2).clone()
    assert torch.equal(perm_out.view(torch.int16), base[torch.from_numpy(p).cuda()].view(torch.int16))
    xt3, it3, wt3 = gh.to_device(x, idx, w * 2)
    dbl = layer.forward(xt3, it3, wt3).clone()
    assert torch.equal(dbl.float(), base.float() * 2)


@pytest.mark.parametrize("gemm", ["single", "pair"])
@pytest.mark.parametrize("T,H,I,E,K", [
    (64, 16384, 128, 2, 1),    # H at its limit: FC1 K = 16384 (128 K blocks), FC2 N = 16384
    (64, 128, 16384, 2, 1),    # I at its limit: FC1 N = 32768, FC2 K = 16384
    (40, 256, 128, 1024, 8),   # E at its limit: most experts empty
])
def test_dimension_limits(lib, orc, T, H, I, E, K, gemm):
    """The largest H, I and E the ABI accepts, through the whole layer."""
    x, idx, w, w1, w2 = small_problem(orc, T, H, I, E, K, seed=H + I + E)
    layer, wo = layer_from_float(lib, orc, T, H, I, E, K, w1, w2, fuse=True, emit=False, gemm=gemm)
    ref = orc.forward(x, idx, w, *wo)
    xt, it, wt = gh.to_device(x, idx, w)
    out = layer.forward(xt, it, wt)
    assert layer.read_status() == (0, 0)
    dbg = layer.debug()
    rows = check_routing(dbg, ref, T, K)
    check_quant(lib, dbg, ref["xq"], ref["xs"], ref["perm"], rows, K)
    compare_outputs(dbg, out, ref, rows, check_gu=False)


@pytest.mark.parametrize("gemm", ["single", "pair"])
def test_sm_budget_bit_identical(lib, orc, gemm):
    """moe_set_sm_budget changes only grid sizes: outputs are bit-identical for
    every budget (each GEMM tile and each element is computed the same way)."""
    import serving_route_gb300.binding as B
    T, H, I, E, K = 513, 1024, 512, 8, 6
    x, idx, w, w1, w2 = small_problem(orc, T, H, I, E, K, seed=5)
    layer, wo = layer_from_float(lib, orc, T, H, I, E, K, w1, w2, fuse=True, gemm=gemm)
    xt, it, wt = gh.to_device(x, idx, w)
    full = layer.forward(xt, it, wt).clone()
    assert layer.read_status() == (0, 0)
    for budget in (2, 3, 40, 151, 0):
        layer.set_sm_budget(budget)
        out = layer.forward(xt, it, wt).clone()
        assert layer.read_status() == (0, 0), budget
        assert torch.equal(out.view(torch.int16), full.view(torch.int16)), budget
        ctas = layer.debug()["gemm_ctas"]
        if budget:
            assert ctas <= budget and (ctas % 2 == 0 or gemm == "single")
    for bad in (-1, 1):
        with pytest.raises(B.MoEError):
            layer.set_sm_budget(bad)
    ref = orc.forward(x, idx, w, *wo)
    compare_outputs(layer.debug(), full, ref, check_routing(layer.debug(), ref, T, K))


@pytest.mark.parametrize("T,H,E,K,mask", [
    (1, 256, 4, 2, 0.0),         # one token: a grid of one block
    (700, 256, 64, 6, 0.1),      # two 512-token blocks, ragged tail, masked slots
    (4096, 256, 64, 6, 0.0),     # the dsv2lite routing: 8 blocks (32 in the three-kernel form)
    (80000, 128, 256, 8, 0.05),  # 157 blocks, more than the SMs
    (3000, 128, 1024, 8, 0.0),   # E at its limit: 72 KB of shared memory per block
])
def test_one_kernel_routing_matches_three_kernels(lib, orc, T, H, E, K, mask):
    """The cooperative one-kernel routing (the default) and the three-kernel
    routing (taken under an SM budget) give the same tables bit for bit, equal
    to the oracle's, and the same layer output."""
    I = 128
    x, idx, w, w1, w2 = small_problem(orc, T, H, I, E, K, seed=21, mask=mask)
    layer, _ = layer_from_float(lib, orc, T, H, I, E, K, w1, w2)
    assert layer.route_kernels(T) == 1
    xt, it, wt = gh.to_device(x, idx, w)
    keys = ("counts", "offsets", "pad_offsets", "perm", "inv", "inv_pad")
    one = layer.forward(xt, it, wt).clone()
    assert layer.read_status() == (0, 0)
    d1 = {k: layer.debug()[k].clone() for k in keys}
    layer.set_sm_budget(64)
    assert layer.route_kernels(T) == 3
    three = layer.forward(xt, it, wt).clone()
    assert layer.read_status() == (0, 0)
    d3 = layer.debug()
    R = int(d1["offsets"][-1])
    n = {"perm": R, "inv": T * K, "inv_pad": T * K}
    for k in keys:
        a, b = d1[k][:n.get(k, d1[k].numel())], d3[k][:n.get(k, d3[k].numel())]
        assert torch.equal(a, b), k
    assert torch.equal(one.view(torch.int16), three.view(torch.int16))
    ref = orc.route(idx, w, E)
    assert np.array_equal(d1["counts"].cpu().numpy(), ref["counts"])
    assert np.array_equal(d1["offsets"].cpu().numpy(), ref["offsets"])
    assert np.array_equal(d1["perm"][:R].cpu().numpy(), ref["perm"])
    assert np.array_equal(d1["inv"][:T * K].cpu().numpy(), ref["inv"])


def test_shared_workspace_between_layers(lib, orc):
    """Two layers of different dims share one workspace (workspace pooling) and
    run in turn on one stream: every output is bit-identical to the same layer
    with a workspace of its own, and matches the oracle."""
    S = lib
    dims = [(300, 512, 256, 8, 2), (517, 256, 384, 6, 4)]
    probs = [small_problem(orc, T, H, I, E, K, seed=31 + j) for j, (T, H, I, E, K) in enumerate(dims)]
    need = max(S.MegaMoELayer.workspace_bytes(H, I, E, K, max_rows=T, fuse_fc1=True)
               for T, H, I, E, K in dims)
    shared = torch.empty(need, dtype=torch.uint8, device="cuda")
    pooled, private, refs, inputs = [], [], [], []
    for (T, H, I, E, K), (x, idx, w, w1, w2) in zip(dims, probs):
        q1, s1 = S.MegaMoELayer.quantize_weights(torch.from_numpy(w1).cuda())
        q2, s2 = S.MegaMoELayer.quantize_weights(torch.from_numpy(w2).cuda())
        for lst, ws in ((pooled, shared), (private, None)):
            layer = S.MegaMoELayer(H, I, E, K, max_rows=T, fuse_fc1=True, workspace=ws)
            layer.bind_weights(q1, s1, q2, s2)
            lst.append(layer)
        refs.append(orc.forward(x, idx, w, *(orc.quant_weights(w1) + orc.quant_weights(w2))))
        inputs.append(gh.to_device(x, idx, w))
    assert pooled[0].workspace.data_ptr() == pooled[1].workspace.data_ptr()
    expect = []
    for layer, (xt, it, wt) in zip(private, inputs):
        expect.append(layer.forward(xt, it, wt).clone())
        assert layer.read_status() == (0, 0)
    for rnd in range(3):  # alternate: each forward overwrites what the other left
        for j, (layer, (xt, it, wt)) in enumerate(zip(pooled, inputs)):
            out = layer.forward(xt, it, wt)
            assert layer.read_status() == (0, 0)
            assert torch.equal(out.view(torch.int16), expect[j].view(torch.int16)), (rnd, j)
    for j, (T, H, I, E, K) in enumerate(dims):
        o = gh.bf16_np(expect[j])
        r = gh.bits_to_f64(refs[j]["out"])
        gate_out(o, r)


@pytest.mark.parametrize("T,H,I,E,K,gemm,emit,empty", [
    (77, 256, 384, 6, 2, "single", True, ()),      # ragged T, 3 FC1 n-tiles, gate||up kept
    (513, 1024, 512, 8, 6, "pair", False, ()),     # CTA pairs
    (300, 512, 256, 16, 4, "single", False, (3, 7, 11)),  # empty experts
    (8, 512, 256, 64, 8, "auto", False, ()),       # decode-like: one row per touched expert
    (2048, 768, 640, 32, 8, "pair", True, (0,)),   # pairs, odd FC2 n-tile count, an empty expert
])
def test_megakernel_matches_two_launches(lib, orc, T, H, I, E, K, gemm, emit, empty):
    """The one-launch FC1 -> FC2 kernel (per-m-tile fc1_done counts) and the two
    launches compute every tile the same way: output, hq, its scales and
    gate||up are bit-identical; the output also matches the oracle."""
    x, idx, w, w1, w2 = small_problem(orc, T, H, I, E, K, seed=41, empty=empty)
    xt, it, wt = gh.to_device(x, idx, w)
    res = []
    for split in (False, True):
        q1, s1 = lib.MegaMoELayer.quantize_weights(torch.from_numpy(w1).cuda())
        q2, s2 = lib.MegaMoELayer.quantize_weights(torch.from_numpy(w2).cuda())
        layer = lib.MegaMoELayer(H, I, E, K, max_rows=T, fuse_fc1=True, emit_fc1=emit, gemm=gemm,
                                 gemms="split" if split else "one_launch")
        layer.bind_weights(q1, s1, q2, s2)
        out = layer.forward(xt, it, wt).clone()
        assert layer.read_status() == (0, 0), split
        d = layer.debug()
        off = d["offsets"].cpu().numpy()
        rows = torch.from_numpy(gh.padded_rows(off, d["pad_offsets"].cpu().numpy(), int(off[-1]))).cuda()
        sf = lib.sf_atom_rows(d["h_sf"], d["rows_alloc"], I // 128)[rows]
        r = [out.view(torch.int16), d["hq"][rows], sf, d["y"][rows].view(torch.int16)]
        if emit:
            r.append(d["gu"][rows].view(torch.int16))
        res.append(r)
    for a, b in zip(*res):
        assert torch.equal(a, b)
    ref = orc.forward(x, idx, w, *(orc.quant_weights(w1) + orc.quant_weights(w2)))
    o = gh.bf16_np(res[0][0].view(torch.bfloat16))
    gate_out(o, gh.bits_to_f64(ref["out"]))


def test_forward_plan(lib):
    """moe_forward_plan: one GEMM launch for short fused forwards, two for long
    ones and for the unfused path; the flags force either; an SM budget keeps
    the routing in three kernels."""
    S = lib
    dv2 = (2048, 1408, 64, 6)
    short = S.MegaMoELayer(*dv2, max_rows=4096, fuse_fc1=True)
    assert short.plan(4096) == dict(route_kernels=1, gemm_launches=1, swiglu_kernels=0, kernels=4,
                                    swap_ab_tokens=0, combine_in_fc2=0)
    assert short.plan(0)["kernels"] == 0
    dv3 = (7168, 2048, 256, 8)
    long_ = S.MegaMoELayer(*dv3, max_rows=1024, fuse_fc1=True, gemm="single")
    assert long_.plan(8)["gemm_launches"] == 1          # decode, few tile rounds
    assert long_.plan(1024)["gemm_launches"] == 2       # every expert touched
    forced = S.MegaMoELayer(*dv3, max_rows=1024, fuse_fc1=True, gemm="single", gemms="one_launch")
    assert forced.plan(1024)["gemm_launches"] == 1
    split = S.MegaMoELayer(*dv2, max_rows=4096, fuse_fc1=True, gemms="split")
    assert split.plan(4096)["gemm_launches"] == 2
    unfused = S.MegaMoELayer(*dv2, max_rows=4096, fuse_fc1=False)
    assert unfused.plan(4096) == dict(route_kernels=1, gemm_launches=2, swiglu_kernels=1, kernels=6,
                                      swap_ab_tokens=0, combine_in_fc2=0)
    short.set_sm_budget(64)
    assert short.plan(4096)["route_kernels"] == 3


def test_programmatic_launch_matches_serialised(lib, orc):
    """Profiling events between the kernels turn the programmatic-dependent
    launches back into plain stream order; the outputs are bit-identical."""
    T, H, I, E, K = 300, 512, 256, 16, 4
    x, idx, w, w1, w2 = small_problem(orc, T, H, I, E, K, seed=9)
    layer, wo = layer_from_float(lib, orc, T, H, I, E, K, w1, w2, fuse=True)
    xt, it, wt = gh.to_device(x, idx, w)
    chained = layer.forward(xt, it, wt).clone()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(10)]
    layer.set_profile_events(ev)
    serial = layer.forward(xt, it, wt).clone()
    layer.set_profile_events([])
    assert layer.read_status() == (0, 0)
    assert torch.equal(chained.view(torch.int16), serial.view(torch.int16))


@pytest.mark.parametrize("expected_m,E,K,pair", [
    (8192, 256, 8, True),    # 256 rows per expert: no padding either way, pairs
    (4096, 64, 6, False),    # 384 rows: 512 with pairs against 384, one CTA per SM
    (16384, 128, 8, True),   # 1024 rows
    (8, 256, 8, False),      # decode: a fraction of a row
])
def test_automatic_tactic(lib, expected_m, E, K, pair):
    layer = lib.MegaMoELayer(256, 256, E, K, max_rows=64, expected_m=expected_m)
    t = layer.tactic()
    if t["gemm_ctas"] and pair:
        assert t["gemm_pair"] and t["pad_rows"] == 256 and t["gemm_ctas"] % 2 == 0
    if not pair:
        assert not t["gemm_pair"] and t["pad_rows"] == 128
