"""Pins of the float64 backward oracle (CPU).

The gradients are tied to facts outside their own code: central finite
differences of the forward oracle, an independent differentiation of the
explicit N x N form, the invariances the forward has (Mc row scaling and
phi(q) scaling leave the DIVISIVE output unchanged, rows of the score matrix
sum to one for DIVISIVE and MALA so shifting every value row shifts every
output row), and a planted mistake that the finite-difference pin catches.
"""

import numpy as np
import pytest

from oracle import mhla_backward_oracle as orb
from oracle import mhla_oracle as orc

NORMS = ["divisive", "none", "mala"]


def _inputs(seed, grid, block, d, positive=False):
    rng = np.random.default_rng(seed)
    N = int(np.prod(grid))
    M = int(np.prod([g // b for g, b in zip(grid, block)]))
    q, k, v = (rng.standard_normal((N, d)) for _ in range(3))
    if positive:
        q, k = np.abs(q) + 0.2, np.abs(k) + 0.2
    else:
        # keep every entry away from the kink of ELU+1 so differences stay smooth
        q = np.where(np.abs(q) < 1e-2, 0.5, q)
        k = np.where(np.abs(k) < 1e-2, -0.5, k)
    mc = rng.uniform(0.1, 1.0, (M, M))
    dout = rng.standard_normal((N, d))
    return q, k, v, mc, dout


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


CASES = [((1, 4, 4), (1, 2, 2), 3), ((2, 2, 3), (1, 2, 3), 2), ((1, 1, 12), (1, 1, 4), 3)]


@pytest.mark.parametrize("norm", NORMS)
@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}-{c[1]}-d{c[2]}")
@pytest.mark.parametrize("fmap", ["elu1", "identity"])
def test_gradients_match_finite_differences(case, norm, fmap):
    grid, block, d = case
    q, k, v, mc, dout = _inputs(11, grid, block, d, positive=(fmap == "identity"))
    dq, dk, dv, dmc = orb.mhla_head_backward64(q, k, v, mc, grid, block, dout, fmap, norm)
    f = lambda **kw: _loss(kw.get("q", q), kw.get("k", k), kw.get("v", v), kw.get("mc", mc), grid, block, dout,
                           fmap, norm)
    for name, got, x in (("q", dq, q), ("k", dk, k), ("v", dv, v), ("mc", dmc, mc)):
        want = _fd(lambda y: f(**{name: y}), x)
        err = orc.relative_max_error(got, want)
        assert err < 1e-6, f"d{name}: {err:.2e}"


@pytest.mark.parametrize("norm", NORMS)
@pytest.mark.parametrize("case", [((1, 8, 8), (1, 4, 4), 8), ((2, 6, 4), (2, 3, 2), 5), ((1, 1, 30), (1, 1, 10), 4),
                                  ((1, 4, 4), (1, 4, 4), 6)],
                         ids=lambda c: f"{c[0]}-{c[1]}-d{c[2]}")
def test_factored_equals_explicit_matrix(case, norm):
    grid, block, d = case
    q, k, v, mc, dout = _inputs(5, grid, block, d)
    a = orb.mhla_head_backward64(q, k, v, mc, grid, block, dout, "elu1", norm)
    b = orb.mhla_bruteforce_backward64(q, k, v, mc, grid, block, dout, "elu1", norm)
    # (with a single block dMc vanishes under DIVISIVE: compare on the scale
    # of the other gradients)
    scale = max(np.max(np.abs(g)) for g in b[:3])
    for name, x, y in zip(("dq", "dk", "dv", "dmc"), a, b):
        assert np.max(np.abs(x - y)) <= 1e-10 * max(np.max(np.abs(y)), scale), name


def test_divisive_mc_row_scaling_gives_orthogonal_gradient():
    # o does not change when a row of Mc is scaled, so the derivative along
    # that row vanishes: sum_b Mc[i,b] dMc[i,b] = 0 for every i
    grid, block, d = (1, 8, 8), (1, 4, 2), 4
    q, k, v, mc, dout = _inputs(3, grid, block, d)
    _, _, _, dmc = orb.mhla_head_backward64(q, k, v, mc, grid, block, dout, "elu1", "divisive")
    proj = np.sum(mc * dmc, axis=1)
    assert np.max(np.abs(proj)) < 1e-10 * np.max(np.abs(mc * dmc))


def test_divisive_phi_q_scaling_gives_orthogonal_gradient():
    # with phi(x) = x, o_t does not change when q_t is scaled: q_t . dq_t = 0
    grid, block, d = (1, 4, 6), (1, 2, 3), 5
    q, k, v, mc, dout = _inputs(4, grid, block, d, positive=True)
    dq, _, _, _ = orb.mhla_head_backward64(q, k, v, mc, grid, block, dout, "identity", "divisive")
    assert np.max(np.abs(np.sum(q * dq, axis=1))) < 1e-10 * np.max(np.abs(q * dq))


@pytest.mark.parametrize("norm", ["divisive", "mala"])
def test_unit_row_sums_give_value_gradient_sum(norm):
    # rows of the score matrix sum to 1, so adding c to every value row adds c
    # to every output row: sum_j dv_j = sum_t dO_t
    grid, block, d = (2, 4, 4), (1, 2, 4), 3
    q, k, v, mc, dout = _inputs(7, grid, block, d)
    _, _, dv, _ = orb.mhla_head_backward64(q, k, v, mc, grid, block, dout, "elu1", norm)
    np.testing.assert_allclose(dv.sum(axis=0), dout.sum(axis=0), rtol=1e-10, atol=1e-10)


def test_none_norm_value_gradient_is_transposed_matrix():
    grid, block, d = (1, 6, 6), (1, 3, 3), 4
    q, k, v, mc, dout = _inputs(8, grid, block, d)
    _, _, dv, _ = orb.mhla_head_backward64(q, k, v, mc, grid, block, dout, "elu1", "none")
    A = orc.attention_matrix64(q, k, mc, grid, block)
    assert orc.relative_max_error(dv, A.T @ dout) < 1e-12


def test_batched_gradients_sum_mc_over_heads():
    rng = np.random.default_rng(9)
    grid, block, d = (1, 4, 4), (1, 2, 2), 3
    q, k, v, dout = (rng.standard_normal((2, 3, 16, d)) for _ in range(4))
    mc = rng.uniform(0.1, 1, (4, 4))
    dq, dk, dv, dmc = orb.mhla_backward64(q, k, v, mc, grid, block, dout)
    want = sum(orb.mhla_head_backward64(q[b, h], k[b, h], v[b, h], mc, grid, block, dout[b, h])[3]
               for b in range(2) for h in range(3))
    assert orc.relative_max_error(dmc, want) < 1e-14
    g = orb.mhla_head_backward64(q[1, 2], k[1, 2], v[1, 2], mc, grid, block, dout[1, 2])
    assert orc.relative_max_error(dq[1, 2], g[0]) == 0.0


def test_planted_mistake_in_feature_map_derivative_is_caught(monkeypatch):
    grid, block, d = (1, 4, 4), (1, 2, 2), 3
    q, k, v, mc, dout = _inputs(12, grid, block, d)
    monkeypatch.setattr(orb, "feature_map_grad", lambda x, kind="elu1": np.ones_like(np.asarray(x, float)))
    dq, _, _, _ = orb.mhla_head_backward64(q, k, v, mc, grid, block, dout)
    want = _fd(lambda y: _loss(y, k, v, mc, grid, block, dout, "elu1", "divisive"), q)
    assert orc.relative_max_error(dq, want) > 1e-3
