"""Routing recipes of the five synthetic workloads (router model code, not the layer).

Every recipe returns ``topk_idx`` int32 [T, K] and ``topk_w`` float32 [T, K].
The router is not part of the hot path: the layer takes the routes as input
(flashinfer PR #6398 "fuse Rubin MegaMoE forward preparation", description:
routes are staged as (expert id, score) with -1 marking an unused slot).
"""
from __future__ import annotations

import numpy as np

from . import inputs as g


def _softmax_rows(logits: np.ndarray) -> np.ndarray:
    l = logits.astype(np.float64)
    l = l - l.max(axis=1, keepdims=True)
    e = np.exp(l)
    return (e / e.sum(axis=1, keepdims=True)).astype(np.float32)


def _topk_desc(keys: np.ndarray, k: int) -> np.ndarray:
    """indices of the k largest keys per row, largest first; ties -> lower index."""
    return np.argsort(-keys, axis=1, kind="stable")[:, :k]


def softmax_topk(T: int, E: int, K: int, seed: int, dist: str):
    """Router logits ~N(0,1) ('normal') or U[0,1) ('uniform') over E experts;
    take the top-K and renormalise the softmax over the K chosen."""
    idx = np.arange(T * E, dtype=np.uint64)
    if dist == "normal":
        logits = g.normal(seed, g.STREAM_LOGITS, idx).reshape(T, E)
    elif dist == "uniform":
        logits = g.uniform01(seed, g.STREAM_LOGITS, idx).reshape(T, E)
    else:
        raise ValueError(dist)
    top = _topk_desc(logits, K)
    chosen = np.take_along_axis(logits, top, axis=1)
    return top.astype(np.int32), _softmax_rows(chosen)


def _chosen_weights(T: int, K: int, seed: int) -> np.ndarray:
    l = g.normal(seed, g.STREAM_WLOGITS, np.arange(T * K, dtype=np.uint64)).reshape(T, K)
    return _softmax_rows(l)


def _fisher_yates(n: int, draws_seed: int, tag: int, base: np.ndarray) -> np.ndarray:
    """one permutation of range(n) per entry of ``base`` (draw index base + i)."""
    nb = base.shape[0]
    p = np.tile(np.arange(n, dtype=np.int64), (nb, 1))
    rows = np.arange(nb)
    for i in range(n - 1, 0, -1):
        j = g.uniform_int(draws_seed, tag, base.astype(np.uint64) + np.uint64(i), i + 1)
        pi = p[rows, i].copy()
        p[rows, i] = p[rows, j]
        p[rows, j] = pi
    return p


def block_permutation(T: int, E: int, K: int, seed: int):
    """Balanced routing: each block of E/K tokens takes one random permutation of
    the E experts and token j of the block gets experts perm[K*j : K*j+K], so
    every expert receives exactly T*K/E rows (the 'block-permutation' routing of
    flashinfer PR #4688, benchmark description)."""
    if E % K != 0:
        raise ValueError("block permutation needs K | E")
    B = E // K
    nblocks = (T + B - 1) // B
    perms = _fisher_yates(E, seed, g.STREAM_BLOCKPERM, np.arange(nblocks, dtype=np.int64) * E)
    idx = perms.reshape(nblocks * B, K)[:T]
    return idx.astype(np.int32), _chosen_weights(T, K, seed)


def zipf_skew(T: int, E: int, K: int, seed: int, s: float = 1.2, empty_frac: float = 0.3):
    """Skewed routing: a seeded permutation pi of the experts; the last
    floor(empty_frac*E) entries of pi receive no token; the others get
    popularity p_r ~ r^-s by rank r in pi; every token draws K distinct experts
    without replacement by Gumbel-top-K on log p_r."""
    n_empty = int(np.floor(empty_frac * E))
    npop = E - n_empty
    if npop < K:
        raise ValueError("too few popular experts")
    pi = _fisher_yates(E, seed, g.STREAM_EXPERTPERM, np.zeros(1, dtype=np.int64))[0]
    logp = -s * np.log(np.arange(1, npop + 1, dtype=np.float64))
    u = g.uniform_open(seed, g.STREAM_GUMBEL, np.arange(T * npop, dtype=np.uint64)).reshape(T, npop)
    keys = logp[None, :] - np.log(-np.log(u))
    top = _topk_desc(keys, K)
    idx = pi[top]
    return idx.astype(np.int32), _chosen_weights(T, K, seed)
