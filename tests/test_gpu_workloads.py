"""GPU parity on the five synthetic workloads at their full sizes.

* dsv2lite (T=4096, H=2048, I=1408, E=64, K=6): the whole layer against the
  oracle (every output element).
* dsv3 prefill / decode sweep / skew: routing tables, every quantised byte and
  scale of the gathered activations -- in full; the expert FFN and combine on
  sampled tokens chosen to reach every expert and every position of the GEMM
  tiles: the oracle runs on a problem made of those tokens with the routes
  they have (a token's output depends only on its own row, its routes and
  those experts' weights).  The prefill and decode samples share the dsv3
  weights, so one oracle call covers all of them.  The launch configuration
  is the one bench.py times (fused FC1 epilogue); a second run of the
  unfused reference path must give the same output bit for bit, and its
  gate||up is compared with the oracle's on every sampled route.
"""
import numpy as np
import pytest
import torch

from gen import configs, problem
from tests import gpu_harness as gh
from tests.test_gpu_parity import (GU_TOL, check_quant, check_routing, compare_outputs,
                                   gate_out, make_layer)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as ge
    ge.build()
    import serving_route_gb300 as S
    return S


_orc_full = {}


def oracle_all_experts(orc, wl, chunk=8):
    """The oracle's weights for every expert of a workload (host generator and
    the oracle's quantiser), built in expert chunks into preallocated arrays and
    kept for the module (the dsv3 prefill and decode workloads share them)."""
    key = (wl.H, wl.I, wl.E, wl.seed)
    if key not in _orc_full:
        _orc_full.clear()
        E, H, I = wl.E, wl.H, wl.I
        w1q = np.empty((E, 2 * I, H), np.uint8)
        w1s = np.empty((E, 2 * I // 128, H // 128), np.float32)
        w2q = np.empty((E, H, I), np.uint8)
        w2s = np.empty((E, H // 128, I // 128), np.float32)
        for e0 in range(0, E, chunk):
            ex = list(range(e0, min(E, e0 + chunk)))
            w1q[ex], w1s[ex] = orc.quant_weights(problem.w1_f32(wl, ex))
            w2q[ex], w2s[ex] = orc.quant_weights(problem.w2_f32(wl, ex))
        _orc_full[key] = (w1q, w1s, w2q, w2s)
    return _orc_full[key]


def test_v2lite_full_layer(lib, orc):
    wl = configs.V2LITE
    wd = gh.device_weights(wl, lib.MegaMoELayer)
    wo = gh.oracle_weights(orc, wl)
    for a, b in zip(wd, wo):
        assert np.array_equal(a.cpu().numpy(), b)
    x, idx, w = gh.host_inputs(wl)
    ref = orc.forward(x, idx, w, *wo)
    xt, it, wt = gh.to_device(x, idx, w)
    outs = {}
    for fuse, emit in ((False, True), (True, False)):
        layer = make_layer(lib, wl, wd, fuse=fuse, emit=emit)
        out = layer.forward(xt, it, wt)
        assert layer.read_status() == (0, 0)
        dbg = layer.debug()
        rows = check_routing(dbg, ref, wl.T, wl.K)
        check_quant(lib, dbg, ref["xq"], ref["xs"], ref["perm"], rows, wl.K)
        stats = compare_outputs(dbg, out, ref, rows, check_gu=not fuse)
        print("v2lite", "fused" if fuse else "unfused", stats)
        outs[fuse] = out.clone()
        del layer
    assert torch.equal(outs[False].view(torch.int16), outs[True].view(torch.int16))


def test_v2lite_full_layer_mxfp8(lib, orc):
    """The dsv2lite workload in the MXFP8 format, every output element against
    the oracle (fmt=1); weight codes and per-chunk scales bit-exact."""
    from tests.test_gpu_mxfp8 import check_quant_mx
    wl = configs.V2LITE
    wd = gh.device_weights(wl, lib.MegaMoELayer, fmt="mxfp8")
    wo = gh.oracle_weights(orc, wl, fmt="mxfp8")
    for a, b in zip(wd, wo):
        assert np.array_equal(a.cpu().numpy(), b)
    x, idx, w = gh.host_inputs(wl)
    ref = orc.forward(x, idx, w, *wo, fmt=1)
    xt, it, wt = gh.to_device(x, idx, w)
    layer = lib.MegaMoELayer(wl.H, wl.I, wl.E, wl.K, max_rows=wl.T, fuse_fc1=True, fmt="mxfp8")
    layer.bind_weights(*wd)
    out = layer.forward(xt, it, wt)
    assert layer.read_status() == (0, 0)
    dbg = layer.debug()
    rows = check_routing(dbg, ref, wl.T, wl.K)
    check_quant_mx(lib, dbg, ref["xq"], ref["xs"], ref["perm"], rows, wl.K)
    stats = compare_outputs(dbg, out, ref, rows, check_gu=False)
    print("v2lite mxfp8", stats)


@pytest.fixture(scope="module")
def v3_weights(lib):
    wd = gh.device_weights(configs.V3_PREFILL, lib.MegaMoELayer)
    yield wd
    del wd
    torch.cuda.empty_cache()


# --------------------------------------------------------------------------
# sampled tokens
# --------------------------------------------------------------------------
# dsv3 prefill: block-permutation routing gives every block of E/K = 32 tokens
# exactly one route to every expert, so expert e's routed row j (in token
# order) comes from block j.  CTA pairs pad segments to 256 rows: rows 0-127
# belong to the pair's first CTA, 128-255 to its second, 32 rows per TMEM lane
# quadrant.  These blocks put rows 0, 40, 72, 127 (first CTA: quadrants 0-3)
# and 128, 168, 200, 255 (second CTA) of EVERY expert into the sample.
PREFILL_BLOCKS = (0, 40, 72, 127, 128, 168, 200, 255)


def sample_tokens(name: str, wl, idx) -> np.ndarray:
    if name == "v3prefill":
        B = wl.E // wl.K
        return np.concatenate([np.arange(b * B, (b + 1) * B) for b in PREFILL_BLOCKS])
    if name.startswith("v3decode"):
        if wl.T <= 256:
            return np.arange(wl.T)                      # every token
        rng = np.random.default_rng(wl.T)
        rest = rng.choice(np.arange(1, wl.T - 1), size=254, replace=False)
        return np.unique(np.concatenate([[0, wl.T - 1], rest]))
    if name == "skew":
        # the hottest expert's first 256-row tile and its last two (the partial
        # tail and the full one before it; every token routed into them), the
        # token of every non-empty expert's last routed row (each expert's
        # tail tile), and 128 random tokens
        flat = idx.ravel()
        counts = np.bincount(flat[flat >= 0], minlength=wl.E)
        hot = int(np.argmax(counts))
        toks_hot = np.nonzero((idx == hot).any(axis=1))[0]   # token order = row order
        last0 = max(0, (len(toks_hot) - 1) // 256 * 256 - 256)
        tail = [int(np.nonzero((idx == e).any(axis=1))[0][-1]) for e in np.nonzero(counts)[0]]
        rng = np.random.default_rng(3)
        return np.unique(np.concatenate([toks_hot[:256], toks_hot[last0:], tail,
                                         rng.choice(wl.T, 128, replace=False)]))
    raise ValueError(name)


def oracle_on_tokens(orc, parts, W):
    """One oracle call over the union of several workloads' sampled tokens that
    share the weights W: rows stacked, each with its own routes.  Returns, per
    part, the oracle's output rows and a map (token i of the part, k) ->
    oracle row of gate||up."""
    X = np.concatenate([p["x"] for p in parts])
    IDX = np.concatenate([p["idx"] for p in parts]).astype(np.int32)
    WT = np.concatenate([p["w"] for p in parts]).astype(np.float32)
    ref = orc.forward(X, IDX, WT, *W)
    assert ref["err"] == 0
    K = IDX.shape[1]
    res, t0 = {}, 0
    for p in parts:
        n = len(p["x"])
        res[p["name"]] = dict(out=ref["out"][t0:t0 + n],
                              inv=ref["inv"][t0 * K:(t0 + n) * K].reshape(n, K), gu=ref["gu"])
        t0 += n
    return res


@pytest.fixture(scope="module")
def dsv3_reference(orc):
    """The oracle on the sampled tokens of the prefill and of every decode size,
    in one call (the expert weights are decoded once for all of them)."""
    parts = []
    for name in ["v3prefill"] + [f"v3decode{t}" for t in configs.DECODE_TOKENS]:
        wl = configs.WORKLOADS[name]
        x, idx, w = gh.host_inputs(wl)
        toks = sample_tokens(name, wl, idx)
        parts.append(dict(name=name, tokens=toks, x=x[toks], idx=idx[toks], w=w[toks]))
    res = oracle_on_tokens(orc, parts, oracle_all_experts(orc, configs.V3_PREFILL))
    for p in parts:
        res[p["name"]]["tokens"] = p["tokens"]
    return res


def gpu_run_and_compare(lib, orc, wl, wd, tokens, ref_part, check_cta_halves=False):
    """Full-size forwards of the workload on the GPU (the bench configuration,
    then the unfused path with gate||up kept): routing tables and every
    quantised activation byte in full against the oracle; fused = unfused bit
    for bit; the sampled tokens' outputs and every sampled route's gate||up
    against the oracle."""
    x, idx, w = gh.host_inputs(wl)
    ref_route = orc.route(idx, w, wl.E)
    assert ref_route["err"] == 0
    xq, xs = orc.quant_rows_bf16(x)
    xt, it, wt = gh.to_device(x, idx, w)
    layer = make_layer(lib, wl, wd, fuse=True, emit=False)
    out_f = layer.forward(xt, it, wt).clone()
    assert layer.read_status() == (0, 0)
    dbg = layer.debug()
    rows = check_routing(dbg, ref_route, wl.T, wl.K)
    check_quant(lib, dbg, xq, xs, ref_route["perm"], rows, wl.K)
    rows_t = torch.from_numpy(rows).cuda()
    hq_f = dbg["hq"][rows_t].clone()
    pair = dbg["gemm_pair"]
    del layer, dbg
    layer = make_layer(lib, wl, wd, fuse=False, emit=True)
    out_u = layer.forward(xt, it, wt).clone()
    assert layer.read_status() == (0, 0)
    dbg = layer.debug()
    assert torch.equal(out_f.view(torch.int16), out_u.view(torch.int16))
    assert torch.equal(hq_f, dbg["hq"][rows_t])
    # outputs of the sampled tokens
    tokens = np.asarray(tokens)
    o = gh.bf16_np(out_f[torch.from_numpy(tokens).cuda()])
    stats = gate_out(o, gh.bits_to_f64(ref_part["out"]))
    # gate||up of every sampled route: GPU padded row vs the oracle's row
    inv_pad = dbg["inv_pad"][:wl.T * wl.K].cpu().numpy().reshape(wl.T, wl.K)
    sub = idx[tokens]
    act = sub >= 0
    gpu_rows = inv_pad[tokens][act]
    orc_rows = ref_part["inv"][act]
    gu = gh.bf16_np(dbg["gu"][torch.from_numpy(gpu_rows).cuda()])
    stats["gu_rel_l2"] = gh.rel_l2(gu, gh.bits_to_f64(ref_part["gu"][orc_rows]))
    assert stats["gu_rel_l2"] <= GU_TOL, stats
    # where the sampled routes sit in their experts' GEMM tiles
    pad = dbg["pad_offsets"].cpu().numpy()
    in_seg = gpu_rows - pad[sub[act]]
    stats.update(tokens=len(tokens), routes=int(act.sum()),
                 experts=len(np.unique(sub[act])), gemm_pair=bool(pair))
    if check_cta_halves:
        # every sampled expert has sampled rows in both CTAs of its pair tile
        # and in all four lane quadrants of each
        assert pair
        for e in np.unique(sub[act]):
            r = in_seg[sub[act] == e]
            assert {int(v) // 32 for v in r} == set(range(8)), (e, sorted(r))
    print(wl.name, stats)
    del layer, dbg
    return stats


def test_v3_prefill_sampled(lib, orc, v3_weights, dsv3_reference):
    """Eight whole routing blocks: every one of the 256 experts, rows in both
    CTAs of its pair tile and in all four TMEM lane quadrants of each."""
    r = dsv3_reference["v3prefill"]
    st = gpu_run_and_compare(lib, orc, configs.V3_PREFILL, v3_weights, r["tokens"], r,
                             check_cta_halves=True)
    assert st["experts"] == 256 and st["tokens"] == 256


@pytest.mark.parametrize("T", configs.DECODE_TOKENS)
def test_v3_decode_sampled(lib, orc, v3_weights, dsv3_reference, T):
    """T = 8, 64, 256: every token; T = 1024: 256 tokens (the first and last
    among them)."""
    r = dsv3_reference[f"v3decode{T}"]
    st = gpu_run_and_compare(lib, orc, configs.V3_DECODE.with_tokens(T), v3_weights, r["tokens"], r)
    assert st["tokens"] == min(T, 256)


def test_skew_sampled(lib, orc):
    """Every token routed into the hottest expert's first and last two 256-row
    tiles, the last routed row of every non-empty expert, and 128 random
    tokens."""
    wl = configs.SKEW
    wd = gh.device_weights(wl, lib.MegaMoELayer)
    x, idx, w = gh.host_inputs(wl)
    counts = np.bincount(idx.ravel(), minlength=wl.E)
    assert (counts == 0).sum() == 38 and counts.max() > 8000   # ragged M, empty groups
    toks = sample_tokens("skew", wl, idx)
    assert len(toks) >= 512
    # the oracle on the non-empty experts only (relabelled; empty experts have no route)
    experts = np.nonzero(counts)[0]
    remap = np.full(wl.E, -1, np.int32)
    remap[experts] = np.arange(len(experts), dtype=np.int32)
    sub = idx[toks]
    mini = np.where(sub >= 0, remap[np.clip(sub, 0, wl.E - 1)], -1).astype(np.int32)
    W = gh.oracle_weights(orc, wl, [int(e) for e in experts])
    part = dict(name="skew", x=x[toks], idx=mini, w=w[toks])
    ref = oracle_on_tokens(orc, [part], W)["skew"]
    st = gpu_run_and_compare(lib, orc, wl, wd, toks, ref)
    assert st["experts"] == len(experts) == 90
    del wd
    torch.cuda.empty_cache()
