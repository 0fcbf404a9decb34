"""moe_route_noalloc: the routing step for callers that cannot allocate device
memory and cannot be handed a workspace (for example a plugin invoked from
another runtime's enqueue callback, where cudaMalloc is not allowed).  Its
scratch is a fixed device array inside the library; this test calls it
through the C ABI twice in a row, with different routes, and checks each
result against the routing that moe_forward computes for the same routes.
Routing is integer work, so the comparison is exact.

The file name makes pytest collect it last; it also passes on its own in a
fresh process (the first call there performs the per-device set-up).
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _routes(T, E, K, seed, mask):
    rng = np.random.default_rng(seed)
    idx = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    idx[rng.random(idx.shape) < mask] = -1
    w = (rng.random((T, K)) + 0.05).astype(np.float32)
    return idx, w


def test_route_noalloc_matches_forward_routing_twice():
    import __graft_entry__ as ge
    ge.build()
    import serving_route_gb300 as S
    import serving_route_gb300.binding as B

    T, H, I, E, K = 300, 256, 128, 16, 4
    layer = S.MegaMoELayer(H, I, E, K, max_rows=T)
    w1 = torch.zeros((E, 2 * I, H), dtype=torch.uint8, device="cuda")
    s1 = torch.ones((E, 2 * I // 128, H // 128), dtype=torch.float32, device="cuda")
    w2 = torch.zeros((E, H, I), dtype=torch.uint8, device="cuda")
    s2 = torch.ones((E, H // 128, I // 128), dtype=torch.float32, device="cuda")
    layer.bind_weights(w1, s1, w2, s2)
    x = torch.zeros((T, H), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream

    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    perm = torch.empty(T * K, dtype=torch.int32, device="cuda")
    inv = torch.empty(T * K, dtype=torch.int32, device="cuda")
    status = torch.full((1,), 0x7F, dtype=torch.int32, device="cuda")

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
        rc = B.moe_route_noalloc(it.data_ptr(), wt.data_ptr(), T, K, E, 1, counts.data_ptr(),
                                 offsets.data_ptr(), perm.data_ptr(), inv.data_ptr(),
                                 status.data_ptr(), stream)
        assert rc == B.MOE_OK, (call, B.status_str(rc))
        torch.cuda.synchronize()
        assert int(status.item()) == 0, call
        assert torch.equal(counts, ref_counts), call
        assert torch.equal(offsets, ref_offsets), call
        assert torch.equal(perm[:R], ref_perm), call
        assert torch.equal(inv, ref_inv), call

    # sizes beyond the fixed scratch are refused before anything is enqueued
    big = B.moe_route_noalloc(it.data_ptr(), wt.data_ptr(), 40000, 8, 16, 1, counts.data_ptr(),
                              offsets.data_ptr(), perm.data_ptr(), inv.data_ptr(),
                              status.data_ptr(), stream)
    assert big == B.MOE_ERR_CAPACITY
