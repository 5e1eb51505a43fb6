"""Pins of the float64 causal backward oracle (CPU).

The causal gradients are tied to facts outside their own code: central
finite differences of the causal forward oracle (itself pinned to the masked
N x N form), an independent differentiation of the masked explicit form,
the structure causality forces on them (no gradient reaches Mc above its
diagonal; an output's gradient reaches only the tokens at or before it), and
planted mistakes that these pins catch.
"""

import numpy as np
import pytest

from oracle import mhla_causal_backward_oracle as ocb
from oracle import mhla_causal_oracle as oca
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
        # away from the kink of ELU+1 so that differences stay smooth
        q = np.where(np.abs(q) < 1e-2, 0.5, q)
        k = np.where(np.abs(k) < 1e-2, -0.5, k)
    mc = rng.uniform(0.1, 1.0, (M, M))
    dout = rng.standard_normal((N, d))
    return q, k, v, mc, dout


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


def _fd_grads(q, k, v, mc, grid, block, dout, fmap, norm):
    def loss(**kw):
        o = oca.mhla_causal_head64(kw.get("q", q), kw.get("k", k), kw.get("v", v), kw.get("mc", mc), grid, block,
                                   fmap, norm)
        return float(np.sum(o * dout))

    return [_fd(lambda y, n=n: loss(**{n: y}), x) for n, x in (("q", q), ("k", k), ("v", v), ("mc", mc))]


CASES = [((1, 4, 4), (1, 2, 2), 3), ((2, 2, 3), (1, 2, 3), 2), ((1, 1, 12), (1, 1, 4), 3), ((1, 1, 6), (1, 1, 6), 2)]


@pytest.mark.parametrize("norm", NORMS)
@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}-{c[1]}-d{c[2]}")
@pytest.mark.parametrize("fmap", ["elu1", "identity"])
def test_gradients_match_finite_differences(case, norm, fmap):
    grid, block, d = case
    q, k, v, mc, dout = _inputs(21, grid, block, d, positive=(fmap == "identity"))
    got = ocb.mhla_causal_head_backward64(q, k, v, mc, grid, block, dout, fmap, norm)
    want = _fd_grads(q, k, v, mc, grid, block, dout, fmap, norm)
    # (with a single block the DIVISIVE output does not depend on Mc at all:
    # dMc is compared on the scale of the other gradients)
    floor = 1e-3 * max(np.max(np.abs(w)) for w in want[:3])
    for name, g, w in zip("q k v mc".split(), got, want):
        err = np.max(np.abs(g - w)) / max(np.max(np.abs(w)), floor)
        assert err < 1e-6, f"d{name}: {err:.2e}"


@pytest.mark.parametrize("norm", NORMS)
@pytest.mark.parametrize("fmap", ["elu1", "relu"])
@pytest.mark.parametrize("case", [((1, 8, 8), (1, 4, 4), 8), ((2, 6, 4), (2, 3, 2), 5), ((1, 1, 30), (1, 1, 10), 4),
                                  ((1, 4, 4), (1, 4, 4), 6), ((2, 4, 6), (1, 2, 3), 3)],
                         ids=lambda c: f"{c[0]}-{c[1]}-d{c[2]}")
def test_recursion_equals_masked_matrix(case, norm, fmap):
    grid, block, d = case
    q, k, v, mc, dout = _inputs(7, grid, block, d)
    a = ocb.mhla_causal_head_backward64(q, k, v, mc, grid, block, dout, fmap, norm)
    b = ocb.mhla_causal_bruteforce_backward64(q, k, v, mc, grid, block, dout, fmap, norm)
    # (single block, DIVISIVE: dMc vanishes; compared on the scale of dv)
    floor = 1e-3 * np.max(np.abs(b[2]))
    for name, x, y in zip("q k v mc".split(), a, b):
        scale = max(np.max(np.abs(y)), floor)
        assert np.max(np.abs(x - y)) / scale < 1e-11, name


@pytest.mark.parametrize("norm", NORMS)
def test_no_gradient_above_the_diagonal_of_mc(norm):
    grid, block = (1, 6, 6), (1, 2, 3)
    q, k, v, mc, dout = _inputs(3, grid, block, 4)
    for fn in (ocb.mhla_causal_head_backward64, ocb.mhla_causal_bruteforce_backward64):
        dmc = fn(q, k, v, mc, grid, block, dout, "elu1", norm)[3]
        assert np.all(np.triu(dmc, 1) == 0.0)
        assert np.all(np.diag(dmc) != 0.0)


@pytest.mark.parametrize("norm", NORMS)
def test_an_output_reaches_only_earlier_tokens(norm):
    grid, block = (1, 4, 6), (1, 2, 3)
    q, k, v, mc, _ = _inputs(9, grid, block, 3)
    N = 24
    rng = np.random.default_rng(1)
    order = np.argsort(orc.block_of_token(grid, block) * N + np.arange(N), kind="stable")
    pos = np.empty(N, dtype=np.int64)
    pos[order] = np.arange(N)  # position of each token in (block, local) order
    for t in rng.choice(N, 4, replace=False):
        dout = np.zeros((N, 3))
        dout[t] = rng.standard_normal(3)
        dq, dk, dv, _ = ocb.mhla_causal_head_backward64(q, k, v, mc, grid, block, dout, "elu1", norm)
        assert np.all(np.delete(dq, t, axis=0) == 0.0)
        later = pos > pos[t]
        assert np.all(dk[later] == 0.0) and np.all(dv[later] == 0.0)
        assert np.any(dv[~later] != 0.0)


def test_single_block_none_is_textbook_causal_linear_attention():
    # M = 1, NONE: o_t = sum_{j<=t} (phq_t . phk_j) v_j, so dv_j = sum_{t>=j} (phq_t . phk_j) dO_t
    grid, block = (1, 1, 9), (1, 1, 9)
    q, k, v, _, dout = _inputs(4, grid, block, 3)
    mc = np.array([[0.7]])
    _, _, dv, dmc = ocb.mhla_causal_head_backward64(q, k, v, mc, grid, block, dout, "elu1", "none")
    pq, pk = orc.feature_map(q), orc.feature_map(k)
    want = np.zeros_like(v)
    for j in range(9):
        for t in range(j, 9):
            want[j] += 0.7 * (pq[t] @ pk[j]) * dout[t]
    np.testing.assert_allclose(dv, want, rtol=1e-12, atol=1e-12)
    # the output is linear in the single weight: dMc = loss / Mc
    o = oca.mhla_causal_head64(q, k, v, mc, grid, block, "elu1", "none")
    np.testing.assert_allclose(dmc[0, 0], np.sum(o * dout) / 0.7, rtol=1e-12)


def test_batched_gradients_sum_mc_over_heads():
    grid, block = (1, 4, 4), (1, 2, 2)
    rng = np.random.default_rng(2)
    q, k, v, dout = (rng.standard_normal((2, 3, 16, 4)) for _ in range(4))
    mc = rng.uniform(0.1, 1.0, (4, 4))
    dq, dk, dv, dmc = ocb.mhla_causal_backward64(q, k, v, mc, grid, block, dout, "elu1", "divisive")
    total = np.zeros((4, 4))
    for b in range(2):
        for h in range(3):
            g = ocb.mhla_causal_head_backward64(q[b, h], k[b, h], v[b, h], mc, grid, block, dout[b, h], "elu1",
                                                "divisive")
            np.testing.assert_array_equal(dq[b, h], g[0])
            total += g[3]
    np.testing.assert_allclose(dmc, total, rtol=1e-13)


def test_planted_mistake_in_the_mask_is_caught(monkeypatch):
    # a strict mask (a token no longer sees itself) in the explicit form
    grid, block, d = (1, 4, 4), (1, 2, 2), 3
    q, k, v, mc, dout = _inputs(21, grid, block, d)
    want = _fd_grads(q, k, v, mc, grid, block, dout, "elu1", "divisive")
    real = oca.causal_mask

    def strict(g, b):
        m = real(g, b)
        return m - np.eye(m.shape[0])

    monkeypatch.setattr(ocb, "causal_mask", strict)
    got = ocb.mhla_causal_bruteforce_backward64(q, k, v, mc, grid, block, dout, "elu1", "divisive")
    assert orc.relative_max_error(got[2], want[2]) > 1e-2


def test_planted_mistake_in_the_mala_count_gradient_is_caught(monkeypatch):
    # dropping dn~ (the running count's weight) leaves dq, dk, dv intact but
    # breaks the diagonal and the lower triangle of dMc
    grid, block, d = (1, 4, 4), (1, 2, 2), 3
    q, k, v, mc, dout = _inputs(21, grid, block, d)
    want = _fd_grads(q, k, v, mc, grid, block, dout, "elu1", "mala")
    real = ocb._token_grads

    def no_count(*args):
        dnum, ds, dvt, _ = real(*args)
        return dnum, ds, dvt, 0.0

    monkeypatch.setattr(ocb, "_token_grads", no_count)
    got = ocb.mhla_causal_head_backward64(q, k, v, mc, grid, block, dout, "elu1", "mala")
    assert orc.relative_max_error(got[2], want[2]) < 1e-6
    assert orc.relative_max_error(got[3], want[3]) > 1e-3
