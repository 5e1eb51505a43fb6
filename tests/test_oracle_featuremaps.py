"""Pins of the ReLU and exp feature maps (the other two maps the MALA page's
ablation names beside ELU+1) and of the zero-denominator rule (CPU only).

Facts outside the oracle's own code: hand values of max(x, 0) and e^x, central
differences of the maps and of the whole forward, the explicit N x N form,
the textbook global linear attention at M = 1, exact invariances (exp turns a
shift of the inputs into a positive scale of the features, ReLU is positively
homogeneous, and DIVISIVE cancels a positive scale of phi(q) or of all
phi(k)), and constructed queries whose denominator is exactly zero.
"""

import numpy as np
import pytest

from oracle import mhla_backward_oracle as orb
from oracle import mhla_oracle as orc

NORMS = ["divisive", "none", "mala"]
MAPS = [orc.RELU, orc.EXP]


def _inputs(seed, grid, block, d, scale=1.0):
    rng = np.random.default_rng(seed)
    N = int(np.prod(grid))
    M = int(np.prod([g // b for g, b in zip(grid, block)]))
    q, k, v = (rng.standard_normal((N, d)) * scale for _ in range(3))
    # keep every entry away from the kink of ReLU so differences stay smooth
    q = np.where(np.abs(q) < 2e-2, 0.5, q)
    k = np.where(np.abs(k) < 2e-2, 0.5, k)
    mc = rng.uniform(0.1, 1.0, (M, M))
    dout = rng.standard_normal((N, d))
    return q, k, v, mc, dout


def test_map_values_by_hand():
    x = np.array([-2.0, -0.5, 0.0, 0.25, 3.0])
    np.testing.assert_array_equal(orc.feature_map(x, orc.RELU), [0.0, 0.0, 0.0, 0.25, 3.0])
    np.testing.assert_allclose(orc.feature_map(x, orc.EXP),
                               [0.1353352832366127, 0.6065306597126334, 1.0, 1.2840254166877414,
                                20.085536923187668], rtol=1e-15)
    np.testing.assert_array_equal(orb.feature_map_grad(x, orc.RELU), [0.0, 0.0, 0.0, 1.0, 1.0])
    np.testing.assert_allclose(orb.feature_map_grad(x, orc.EXP), orc.feature_map(x, orc.EXP), rtol=0)


@pytest.mark.parametrize("fmap", MAPS)
def test_map_derivative_matches_differences(fmap):
    x = np.array([-1.7, -0.3, 0.2, 0.9, 2.4])
    h = 1e-6
    fd = (orc.feature_map(x + h, fmap) - orc.feature_map(x - h, fmap)) / (2 * h)
    np.testing.assert_allclose(orb.feature_map_grad(x, fmap), fd, rtol=1e-8, atol=1e-9)


@pytest.mark.parametrize("norm", NORMS)
@pytest.mark.parametrize("fmap", MAPS)
def test_factored_equals_explicit_matrix(fmap, norm):
    grid, block, d = (2, 6, 4), (1, 3, 2), 5
    q, k, v, mc, _ = _inputs(21, grid, block, d)
    a = orc.mhla_head64(q, k, v, mc, grid, block, fmap, norm)
    b = orc.mhla_bruteforce64(q, k, v, mc, grid, block, fmap, norm)
    assert orc.relative_max_error(a, b) < 1e-12


@pytest.mark.parametrize("fmap", MAPS)
def test_single_block_is_textbook_linear_attention(fmap):
    grid, block, d = (1, 1, 24), (1, 1, 24), 6
    q, k, v, _, _ = _inputs(22, grid, block, d)
    pq = orc.feature_map(q, fmap)
    pk = orc.feature_map(k, fmap)
    want = np.zeros_like(v)
    for t in range(q.shape[0]):
        w = np.array([pq[t] @ pk[j] for j in range(k.shape[0])])
        want[t] = (w @ v) / w.sum()
    got = orc.mhla_head64(q, k, v, np.array([[1.0]]), grid, block, fmap, "divisive")
    assert orc.relative_max_error(got, want) < 1e-12


def test_exp_shift_of_inputs_cancels_under_divisive():
    # phi(x + c) = e^c phi(x): a shift of one query, or of every key, is a
    # positive scale that the DIVISIVE normalisation removes
    grid, block, d = (1, 6, 6), (1, 3, 3), 4
    q, k, v, mc, _ = _inputs(23, grid, block, d)
    base = orc.mhla_head64(q, k, v, mc, grid, block, orc.EXP, "divisive")
    qs = q.copy()
    qs[5] += 1.3
    assert orc.relative_max_error(orc.mhla_head64(qs, k, v, mc, grid, block, orc.EXP, "divisive"), base) < 1e-12
    assert orc.relative_max_error(orc.mhla_head64(q, k - 0.7, v, mc, grid, block, orc.EXP, "divisive"),
                                  base) < 1e-12
    # NONE is not invariant: the output scales by e^c
    none = orc.mhla_head64(q, k, v, mc, grid, block, orc.EXP, "none")
    shifted = orc.mhla_head64(q, k + 0.5, v, mc, grid, block, orc.EXP, "none")
    assert orc.relative_max_error(shifted, np.exp(0.5) * none) < 1e-12


def test_relu_positive_homogeneity():
    grid, block, d = (1, 6, 6), (1, 3, 3), 4
    q, k, v, mc, _ = _inputs(24, grid, block, d)
    base = orc.mhla_head64(q, k, v, mc, grid, block, orc.RELU, "divisive")
    assert orc.relative_max_error(orc.mhla_head64(2.5 * q, k, v, mc, grid, block, orc.RELU, "divisive"),
                                  base) < 1e-12
    none = orc.mhla_head64(q, k, v, mc, grid, block, orc.RELU, "none")
    assert orc.relative_max_error(orc.mhla_head64(q, 3.0 * k, v, mc, grid, block, orc.RELU, "none"),
                                  3.0 * none) < 1e-12


@pytest.mark.parametrize("norm", NORMS)
def test_zero_denominator_gives_zero_output(norm):
    grid, block, d = (1, 4, 4), (1, 2, 2), 3
    q, k, v, mc, _ = _inputs(25, grid, block, d)
    q[0] = -np.abs(q[0]) - 0.1            # phi(q_0) = 0
    k[:, 0] = -np.abs(k[:, 0]) - 0.1      # no key has feature 0
    q[5] = np.array([0.8, -0.4, -1.1])    # phi(q_5) nonzero only in feature 0
    o = orc.mhla_head64(q, k, v, mc, grid, block, orc.RELU, norm)
    b = orc.mhla_bruteforce64(q, k, v, mc, grid, block, orc.RELU, norm)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(b))
    np.testing.assert_array_equal(o[[0, 5]], 0.0)
    np.testing.assert_array_equal(b[[0, 5]], 0.0)
    live = np.ones(q.shape[0], bool)
    live[[0, 5]] = False
    assert orc.relative_max_error(o[live], b[live]) < 1e-12
    # the numerator of those queries is zero too, so num / (s + eps) = 0 for any eps > 0
    num = orc.mhla_head64(q, k, v, mc, grid, block, orc.RELU, "none")
    np.testing.assert_array_equal(num[[0, 5]], 0.0)


def _loss(q, k, v, mc, grid, block, dout, fmap, norm):
    return float(np.sum(orc.mhla_head64(q, k, v, mc, grid, block, fmap, norm) * dout))


def _fd(fun, x, h=1e-6):
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        idx = it.multi_index
        xp, xm = x.copy(), x.copy()
        xp[idx] += h
        xm[idx] -= h
        g[idx] = (fun(xp) - fun(xm)) / (2 * h)
    return g


@pytest.mark.parametrize("norm", NORMS)
@pytest.mark.parametrize("fmap", MAPS)
def test_gradients_match_finite_differences(fmap, norm):
    grid, block, d = (1, 4, 4), (1, 2, 2), 3
    q, k, v, mc, dout = _inputs(26, grid, block, d)
    if fmap == orc.RELU:
        q[3] = -np.abs(q[3]) - 0.2        # a query with s = 0: constant output, no gradient
    got = orb.mhla_head_backward64(q, k, v, mc, grid, block, dout, fmap, norm)
    f = lambda **kw: _loss(kw.get("q", q), kw.get("k", k), kw.get("v", v), kw.get("mc", mc), grid, block, dout,
                           fmap, norm)
    for name, g, x in zip(("q", "k", "v", "mc"), got, (q, k, v, mc)):
        want = _fd(lambda y: f(**{name: y}), x)
        assert orc.relative_max_error(g, want) < 1e-6, name
    if fmap == orc.RELU:
        np.testing.assert_array_equal(got[0][3], 0.0)


@pytest.mark.parametrize("norm", NORMS)
@pytest.mark.parametrize("fmap", MAPS)
def test_factored_gradients_equal_explicit(fmap, norm):
    grid, block, d = (2, 4, 4), (1, 2, 4), 4
    q, k, v, mc, dout = _inputs(27, grid, block, d)
    q[1] = -np.abs(q[1]) - 0.1
    a = orb.mhla_head_backward64(q, k, v, mc, grid, block, dout, fmap, norm)
    b = orb.mhla_bruteforce_backward64(q, k, v, mc, grid, block, dout, fmap, norm)
    scale = max(np.max(np.abs(g)) for g in b[:3])
    for x, y in zip(a, b):
        assert np.max(np.abs(x - y)) <= 1e-10 * max(np.max(np.abs(y)), scale)
