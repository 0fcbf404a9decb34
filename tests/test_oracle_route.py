"""Pins of the oracle's routing step: brute force on tiny inputs, numpy's stable
argsort (a library routine), and the validation rules of flashinfer PR #6398
("fuse Rubin MegaMoE forward preparation": expert-id bounds, no duplicate
routes, finite scores on active routes; masked slots may hold NaN)."""
import numpy as np
import pytest


def brute_route(idx, E):
    T, K = idx.shape
    counts = [sum(1 for t in range(T) for k in range(K) if idx[t, k] == e) for e in range(E)]
    offsets = [0]
    for c in counts:
        offsets.append(offsets[-1] + c)
    perm = []
    for e in range(E):            # expert-major, then ascending flat route id
        for t in range(T):
            for k in range(K):
                if idx[t, k] == e:
                    perm.append(t * K + k)
    inv = [-1] * (T * K)
    for pos, r in enumerate(perm):
        inv[r] = pos
    return counts, offsets, perm, inv


@pytest.mark.parametrize("T,K,E,mask", [(7, 2, 5, 0.0), (16, 4, 9, 0.3), (33, 8, 16, 0.1), (1, 1, 1, 0.0),
                                        (5, 6, 40, 0.5), (0, 2, 4, 0.0)])
def test_route_brute_force(orc, T, K, E, mask):
    rng = np.random.default_rng(T * 100 + K)
    idx = np.stack([rng.permutation(E)[:K] if E >= K else rng.integers(0, E, K) for _ in range(T)]) \
        if T else np.zeros((0, K), np.int32)
    idx = idx.astype(np.int32)
    if T:
        idx[rng.random(idx.shape) < mask] = -1
    w = rng.random(idx.shape).astype(np.float32)
    r = orc.route(idx, w, E)
    counts, offsets, perm, inv = brute_route(idx, E)
    assert r["err"] == 0
    assert list(r["counts"]) == counts
    assert list(r["offsets"]) == offsets
    assert list(r["perm"]) == perm
    assert list(r["inv"]) == inv


def test_route_matches_stable_argsort(orc):
    rng = np.random.default_rng(11)
    T, K, E = 300, 6, 64
    idx = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    idx[rng.random(idx.shape) < 0.2] = -1
    w = rng.random(idx.shape).astype(np.float32)
    r = orc.route(idx, w, E)
    flat = idx.ravel()
    active = np.where(flat >= 0)[0]
    order = active[np.argsort(flat[active], kind="stable")]
    assert np.array_equal(r["perm"], order)
    assert np.array_equal(r["counts"], np.bincount(flat[active], minlength=E))
    # bijection onto the active routes; monotone offsets; sum of counts = R
    assert sorted(r["perm"].tolist()) == active.tolist()
    assert np.all(np.diff(r["offsets"]) >= 0) and r["offsets"][-1] == len(active)
    assert np.all(r["inv"][r["perm"]] == np.arange(len(active)))


def test_route_validation(orc):
    w = np.ones((2, 2), np.float32)
    ok = np.array([[0, 1], [1, -1]], np.int32)
    assert orc.route(ok, w, 2)["err"] == 0
    assert orc.route(np.array([[0, 2], [1, 0]], np.int32), w, 2)["err"] == orc.ERR_ROUTE_RANGE
    assert orc.route(np.array([[0, -2], [1, 0]], np.int32), w, 2)["err"] == orc.ERR_ROUTE_RANGE
    assert orc.route(np.array([[1, 1], [1, 0]], np.int32), w, 2)["err"] == orc.ERR_ROUTE_DUP
    # masked duplicates are not duplicates
    assert orc.route(np.array([[-1, -1], [1, 0]], np.int32), w, 2)["err"] == 0
    wn = w.copy()
    wn[0, 1] = np.nan
    assert orc.route(ok, wn, 2)["err"] == orc.ERR_ROUTE_NONFINITE
    wn2 = w.copy()
    wn2[1, 1] = np.inf   # masked slot: non-finite allowed
    assert orc.route(ok, wn2, 2)["err"] == 0
    # with checks off only the bounds rule remains
    assert orc.route(np.array([[1, 1], [1, 0]], np.int32), w, 2, check=False)["err"] == 0
    assert orc.route(np.array([[0, 5], [1, 0]], np.int32), w, 2, check=False)["err"] == orc.ERR_ROUTE_RANGE
