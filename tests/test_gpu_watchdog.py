"""Device watchdog (failure detection without a GPU fault).

Every wait inside the GEMM kernels and the routing kernel's grid barrier is
bounded.  With MOE_FLAG_WATCHDOG_TEST
the first GEMM CTA withholds one pipeline stage -- a barrier that nothing
completes; on CTA pairs the first pair's second CTA withholds its share, which
the leader's barrier still expects -- and the wait bound drops to 20 ms: the
kernel must record
MOE_DEV_TIMEOUT, wind down (drain its copies and MMAs, free tensor memory) and
return, and the context must stay usable for the next forward.  No trap, no
fault, no hang.
"""
import numpy as np
import pytest
import torch

from tests import gpu_harness as gh
from tests.test_gpu_parity import compare_outputs, small_problem

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("gemm,fold", [("single", False), ("pair", False), ("swap", False),
                                       ("single", True), ("swap", True)])
@pytest.mark.parametrize("split", [False, True])
def test_watchdog_expires_with_status_and_context_survives(orc, split, gemm, fold):
    """split=False: the one-launch FC1 -> FC2 kernel, where the FC2 tiles of
    the other CTAs also wait in vain for the m-tile counts that CTA 0 (or
    pair 0) never publishes, and expire on their own bound.  gemm="pair": the
    leader's MMA wait expires; the peer's waits on the leader's commits expire
    too, and both CTAs meet at the cluster barrier before freeing the pair's
    tensor memory.  gemm="swap": a 40-token forward on single CTAs, which runs
    the token-as-N kernels (double-buffered accumulators, counter schedule).
    fold: the combine folded into FC2 as well, whose queue and counters wait
    on the tiles the expired CTA never stores (their waits end on the abort
    flag or their own bound)."""
    import __graft_entry__ as ge
    ge.build()
    import serving_route_gb300 as S
    import serving_route_gb300.binding as B

    T, H, I, E, K = (40 if gemm == "swap" else 300), 512, 256, 8, 2
    swap = gemm == "swap"
    gemm = "single" if swap else gemm
    x, idx, w, w1, w2 = small_problem(orc, T, H, I, E, K, seed=31)
    q1, s1 = S.MegaMoELayer.quantize_weights(torch.from_numpy(w1).cuda())
    q2, s2 = S.MegaMoELayer.quantize_weights(torch.from_numpy(w2).cuda())
    xt, it, wt = gh.to_device(x, idx, w)

    bad = S.MegaMoELayer(H, I, E, K, max_rows=T, fuse_fc1=True, gemm=gemm, watchdog_test=True,
                         gemms="split" if split else "one_launch", combine_in_fc2=fold)
    assert (bad.plan(T)["swap_ab_tokens"] > 0) == swap
    assert bad.plan(T)["combine_in_fc2"] == (1 if fold else 0)
    bad.bind_weights(q1, s1, q2, s2)
    bad.forward(xt, it, wt)
    st, bits = bad.read_status()
    assert st == B.MOE_ERR_DEVICE_TIMEOUT and bits & B.MOE_DEV_TIMEOUT, (st, bits)

    # the context is intact: a normal forward right after is correct
    good = S.MegaMoELayer(H, I, E, K, max_rows=T, fuse_fc1=True, gemm=gemm)
    good.bind_weights(q1, s1, q2, s2)
    out = good.forward(xt, it, wt)
    assert good.read_status() == (0, 0)
    ref = orc.forward(x, idx, w, *orc.quant_weights(w1), *orc.quant_weights(w2))
    compare_outputs(good.debug(), out, ref, np.zeros(0, np.int64), check_gu=False)


def test_routing_barrier_expires_with_status_and_context_survives(orc):
    """MOE_FLAG_WATCHDOG_ROUTE_TEST: the one-kernel routing's last block never
    arrives at the grid barrier.  Every block gives up after 20 ms, records
    MOE_DEV_TIMEOUT and marks its routes unrouted, so no expert is computed
    and the output is zero; a normal forward on the same context right after
    is correct."""
    import __graft_entry__ as ge
    ge.build()
    import serving_route_gb300 as S
    import serving_route_gb300.binding as B

    T, H, I, E, K = 1100, 256, 256, 8, 2           # three routing blocks of 512 tokens
    x, idx, w, w1, w2 = small_problem(orc, T, H, I, E, K, seed=33)
    q1, s1 = S.MegaMoELayer.quantize_weights(torch.from_numpy(w1).cuda())
    q2, s2 = S.MegaMoELayer.quantize_weights(torch.from_numpy(w2).cuda())
    xt, it, wt = gh.to_device(x, idx, w)

    bad = S.MegaMoELayer(H, I, E, K, max_rows=T, fuse_fc1=True, watchdog_route_test=True)
    assert bad.route_kernels(T) == 1
    bad.bind_weights(q1, s1, q2, s2)
    out = bad.forward(xt, it, wt)
    st, bits = bad.read_status()
    assert st == B.MOE_ERR_DEVICE_TIMEOUT and bits & B.MOE_DEV_TIMEOUT, (st, bits)
    assert not torch.any(out[:T].view(torch.int16))

    good = S.MegaMoELayer(H, I, E, K, max_rows=T, fuse_fc1=True)
    good.bind_weights(q1, s1, q2, s2)
    out = good.forward(xt, it, wt)
    assert good.read_status() == (0, 0)
    ref = orc.forward(x, idx, w, *orc.quant_weights(w1), *orc.quant_weights(w2))
    compare_outputs(good.debug(), out, ref, np.zeros(0, np.int64), check_gu=False)
