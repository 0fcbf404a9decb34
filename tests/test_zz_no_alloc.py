"""moe_route_noalloc: the routing step for callers that cannot allocate device
memory and cannot be handed a workspace (for example a plugin invoked from
another runtime's enqueue callback, where cudaMalloc is not allowed).  Its
scratch is a fixed device array inside the library.

Through the C ABI, this file checks the call against the oracle's routing
(counts, offsets, the stable permutation, its inverse, and the status bits)
and against the routing moe_forward computes, twice in a row with different
routes; at both limits of the fixed scratch (num_tokens * top_k = 131072 and
ceil(num_tokens / 128) * num_experts = 32768) and one step past each, which
must be refused; with every route error; and with no token.  Routing is
integer work, so every comparison is exact.

The file name makes pytest collect it last; it also passes on its own in a
fresh process (the first call there performs the per-context set-up).
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

LIMIT_ROUTES = 131072        # num_tokens * top_k
LIMIT_BLOCK_EXPERTS = 32768  # ceil(num_tokens / 128) * num_experts


@pytest.fixture(scope="module")
def B():
    import __graft_entry__ as ge
    ge.build()
    import serving_route_gb300.binding as binding
    return binding


def _routes(T, E, K, seed, mask):
    rng = np.random.default_rng(seed)
    idx = np.argsort(rng.random((T, E)), axis=1)[:, :K].astype(np.int32)   # K distinct experts
    idx[rng.random(idx.shape) < mask] = -1
    w = (rng.random((T, K)) + 0.05).astype(np.float32)
    return idx, w


class Bufs:
    def __init__(self, T, K, E):
        self.counts = torch.full((E,), -7, dtype=torch.int32, device="cuda")
        self.offsets = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
        self.perm = torch.full((max(T * K, 1),), -7, dtype=torch.int32, device="cuda")
        self.inv = torch.full((max(T * K, 1),), -7, dtype=torch.int32, device="cuda")
        self.status = torch.full((1,), 0x7F, dtype=torch.int32, device="cuda")


def _call(B, idx_t, w_t, T, K, E, bufs, check=1):
    stream = torch.cuda.current_stream().cuda_stream
    return B.moe_route_noalloc(idx_t.data_ptr() if idx_t is not None else 0,
                               w_t.data_ptr() if w_t is not None else 0, T, K, E, check,
                               bufs.counts.data_ptr(), bufs.offsets.data_ptr(), bufs.perm.data_ptr(),
                               bufs.inv.data_ptr(), bufs.status.data_ptr(), stream)


def _check_against_oracle(orc, bufs, idx, w, E, check=True):
    T, K = idx.shape
    ref = orc.route(idx, w, E, check=check)
    torch.cuda.synchronize()
    assert int(bufs.status.item()) == ref["err"]
    assert np.array_equal(bufs.counts.cpu().numpy(), ref["counts"])
    assert np.array_equal(bufs.offsets.cpu().numpy(), ref["offsets"])
    R = int(ref["offsets"][-1])
    assert np.array_equal(bufs.perm[:R].cpu().numpy(), ref["perm"])
    assert np.array_equal(bufs.inv[:T * K].cpu().numpy(), ref["inv"])
    return ref


def test_route_noalloc_matches_forward_routing_twice(B, orc):
    """Two calls in a row with different routes: each equals the routing that
    moe_forward (the entry point with a workspace) computes for the same
    routes, and the oracle's."""
    import serving_route_gb300 as S

    T, H, I, E, K = 300, 256, 128, 16, 4
    layer = S.MegaMoELayer(H, I, E, K, max_rows=T)
    w1 = torch.zeros((E, 2 * I, H), dtype=torch.uint8, device="cuda")
    s1 = torch.ones((E, 2 * I // 128, H // 128), dtype=torch.float32, device="cuda")
    w2 = torch.zeros((E, H, I), dtype=torch.uint8, device="cuda")
    s2 = torch.ones((E, H // 128, I // 128), dtype=torch.float32, device="cuda")
    layer.bind_weights(w1, s1, w2, s2)
    x = torch.zeros((T, H), dtype=torch.bfloat16, device="cuda")
    bufs = Bufs(T, K, E)

    for call, (seed, mask) in enumerate(((1, 0.0), (2, 0.3))):
        idx, w = _routes(T, E, K, seed, mask)
        it = torch.from_numpy(idx).cuda()
        wt = torch.from_numpy(w).cuda()
        # the existing entry point
        layer.forward(x, it, wt)
        assert layer.read_status() == (0, 0)
        d = layer.debug()
        ref_counts = d["counts"].clone()
        ref_offsets = d["offsets"].clone()
        R = int(ref_offsets[-1].item())
        ref_perm = d["perm"][:R].clone()
        ref_inv = d["inv"][:T * K].clone()
        # the allocation-free entry point
        rc = _call(B, it, wt, T, K, E, bufs)
        assert rc == B.MOE_OK, (call, B.status_str(rc))
        torch.cuda.synchronize()
        assert int(bufs.status.item()) == 0, call
        assert torch.equal(bufs.counts, ref_counts), call
        assert torch.equal(bufs.offsets, ref_offsets), call
        assert torch.equal(bufs.perm[:R], ref_perm), call
        assert torch.equal(bufs.inv[:T * K], ref_inv), call
        _check_against_oracle(orc, bufs, idx, w, E)


@pytest.mark.parametrize("T,K,E", [
    (16384, 8, 256),   # T*K = 131072 and ceil(T/128)*E = 32768: both limits exactly
    (4096, 8, 1024),   # ceil(T/128)*E = 32768 with the largest E
    (1, 1, 1),
    (129, 6, 64),      # a ragged 128-token block
])
def test_route_noalloc_at_the_scratch_limits(B, orc, T, K, E):
    assert T * K <= LIMIT_ROUTES and (T + 127) // 128 * E <= LIMIT_BLOCK_EXPERTS
    idx, w = _routes(T, E, K, seed=T + E, mask=0.1)
    bufs = Bufs(T, K, E)
    rc = _call(B, torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda(), T, K, E, bufs)
    assert rc == B.MOE_OK, B.status_str(rc)
    _check_against_oracle(orc, bufs, idx, w, E)


@pytest.mark.parametrize("T,K,E", [
    (16385, 8, 64),    # T*K = 131080 > 131072
    (4097, 8, 1024),   # ceil(T/128)*E = 33792 > 32768
    (1 << 40, 8, 8),   # far past every limit (no overflow in the size arithmetic)
])
def test_route_noalloc_refuses_past_the_limits(B, T, K, E):
    bufs = Bufs(1, K, E)
    idx_t = torch.zeros((1, K), dtype=torch.int32, device="cuda")
    w_t = torch.ones((1, K), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    assert _call(B, idx_t, w_t, T, K, E, bufs) == B.MOE_ERR_CAPACITY
    torch.cuda.synchronize()
    assert int(bufs.status.item()) == 0x7F   # refused before anything was enqueued


@pytest.mark.parametrize("bad", ["range_high", "range_negative", "duplicate", "nonfinite"])
def test_route_noalloc_route_errors(B, orc, bad):
    """Each route error sets its status bit, as the oracle's validation does;
    an out-of-range id is treated as masked (inv = -1), a duplicate or a
    non-finite weight is flagged and the route kept -- the tables equal the
    oracle's in every case."""
    T, K, E = 200, 4, 32
    idx, w = _routes(T, E, K, seed=9, mask=0.0)
    if bad == "range_high":
        idx[5, 1] = E + 3
    elif bad == "range_negative":
        idx[7, 2] = -2
    elif bad == "duplicate":
        idx[11, 3] = idx[11, 0]
    else:
        w[13, 1] = np.nan
    bufs = Bufs(T, K, E)
    rc = _call(B, torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda(), T, K, E, bufs)
    assert rc == B.MOE_OK
    ref = _check_against_oracle(orc, bufs, idx, w, E)
    bit = {"range_high": B.MOE_DEV_ROUTE_RANGE, "range_negative": B.MOE_DEV_ROUTE_RANGE,
           "duplicate": B.MOE_DEV_ROUTE_DUP, "nonfinite": B.MOE_DEV_ROUTE_NONFINITE}[bad]
    assert ref["err"] == bit and int(bufs.status.item()) == bit
    if bad.startswith("range"):
        r = 5 * K + 1 if bad == "range_high" else 7 * K + 2
        assert int(bufs.inv[r].item()) == -1


def test_route_noalloc_no_tokens(B):
    """num_tokens = 0: the status word is cleared, counts and offsets are zero,
    nothing else is written (the route arrays may be NULL)."""
    E, K = 16, 2
    bufs = Bufs(0, K, E)
    stream = torch.cuda.current_stream().cuda_stream
    rc = B.moe_route_noalloc(0, 0, 0, K, E, 1, bufs.counts.data_ptr(), bufs.offsets.data_ptr(), 0, 0,
                             bufs.status.data_ptr(), stream)
    assert rc == B.MOE_OK
    torch.cuda.synchronize()
    assert int(bufs.status.item()) == 0
    assert torch.count_nonzero(bufs.counts) == 0 and torch.count_nonzero(bufs.offsets) == 0
    assert int(bufs.perm[0].item()) == -7 and int(bufs.inv[0].item()) == -7
