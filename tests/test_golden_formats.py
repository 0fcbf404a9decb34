"""Pins the oracle's scale-block geometry to the formats the pages name
(tests/golden/scale_formats.txt, each line cited there).

A single outlier raises the scale of the block that holds it: exactly the
elements of that block get new E4M3 codes, every other code stays.  The set of
changed codes must be the fixture's block, for activations (through the whole
layer) and for weights.  Scales must be powers of two, within E8M0's exponent
range where the fixture says e8m0.
"""
import os

import numpy as np
import pytest

from tests import helpers_exact as hx

HERE = os.path.dirname(os.path.abspath(__file__))


def formats():
    rows = {}
    for line in open(os.path.join(HERE, "golden", "scale_formats.txt")):
        line = line.split("#")[0].split()
        if line:
            name, act, wt, elem, scale = line
            rows[name] = ([int(v) for v in act.split("x")], [int(v) for v in wt.split("x")], elem, scale)
    return rows


FMT = {"blockwise": 0, "mxfp8": 1}


def test_fixture_lists_both_formats():
    assert set(formats()) == set(FMT)


def _values(rng, shape):
    # magnitudes in [0.5, 1.5): every code moves when its block's scale grows
    return (rng.uniform(0.5, 1.5, shape) * rng.choice([-1.0, 1.0], shape))


def _pow2_ok(s, scale):
    e = np.log2(s.astype(np.float64))
    assert np.all(e == np.round(e))
    if scale == "e8m0":
        assert np.all((e >= -127) & (e <= 127))


@pytest.mark.parametrize("name", sorted(FMT))
def test_activation_block(orc, name):
    (ar, ac), _, elem, scale = formats()[name]
    assert ar == 1 and elem == "e4m3"
    fmt = FMT[name]
    T, H, I = 3, 512, 128
    rng = np.random.default_rng(81)
    x = hx.f64_to_bf16_bits(_values(rng, (T, H)))
    w1 = (rng.standard_normal((1, 2 * I, H)) * 0.05).astype(np.float32)
    w2 = (rng.standard_normal((1, H, I)) * 0.05).astype(np.float32)
    wq = (orc.quant_weights_mx(w1) + orc.quant_weights_mx(w2)) if fmt else \
        (orc.quant_weights(w1) + orc.quant_weights(w2))
    idx = np.zeros((T, 1), np.int32)
    wt = np.ones((T, 1), np.float32)
    base = orc.forward(x, idx, wt, *wq, fmt=fmt)
    _pow2_ok(base["xs"], scale)
    for j0 in (0, 37, 200, H - 1):
        x2 = x.copy()
        x2[1, j0] = hx.f64_to_bf16_bits(np.array([300.0]))[0]
        r = orc.forward(x2, idx, wt, *wq, fmt=fmt)
        changed = np.argwhere(r["xq"] != base["xq"])
        a = j0 // ac * ac
        assert set(map(tuple, changed)) == {(1, c) for c in range(a, a + ac)}, (name, j0)


@pytest.mark.parametrize("name", sorted(FMT))
def test_weight_block(orc, name):
    _, (br, bc), elem, scale = formats()[name]
    quant = orc.quant_weights_mx if FMT[name] else orc.quant_weights
    rng = np.random.default_rng(82)
    w = _values(rng, (2, 256, 384)).astype(np.float32)
    q0, s0 = quant(w)
    _pow2_ok(s0, scale)
    for (m, r0, c0) in ((0, 0, 0), (1, 130, 77), (1, 255, 383)):
        w2 = w.copy()
        w2[m, r0, c0] = 300.0
        q, _ = quant(w2)
        changed = set(map(tuple, np.argwhere(q != q0)))
        ra, ca = r0 // br * br, c0 // bc * bc
        want = {(m, r, c) for r in range(ra, ra + br) for c in range(ca, ca + bc)}
        assert changed == want, (name, m, r0, c0)
