"""Pins of the causal (block-ordered) MHLA oracle (CPU only).

Facts outside its own code: the masked explicit N x N form, textbook causal
linear attention at M = 1, the first token reproducing its own value, exact
causality (later tokens cannot change earlier outputs), agreement with the
non-causal oracle where the causal prefix is the whole visible set (the last
token of each block when Mc is lower triangular), MALA's unit row sums, and a
planted mistake (the diagonal weight of Mc dropped from the in-block term).
"""

import numpy as np
import pytest

from oracle import mhla_causal_oracle as occ
from oracle import mhla_oracle as orc

NORMS = ["divisive", "none", "mala"]
CASES = [((1, 1, 24), (1, 1, 6)), ((1, 6, 8), (1, 3, 2)), ((4, 4, 4), (2, 2, 2)), ((2, 3, 4), (2, 3, 4))]


def _inputs(seed, grid, d=4):
    rng = np.random.default_rng(seed)
    N = int(np.prod(grid))
    q, k, v = (rng.standard_normal((N, d)) for _ in range(3))
    return q, k, v


def _mc(seed, M):
    return np.random.default_rng(seed).uniform(0.1, 1.0, (M, M))


@pytest.mark.parametrize("norm", NORMS)
@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}-{c[1]}")
@pytest.mark.parametrize("fmap", ["elu1", "relu"])
def test_recursion_equals_masked_matrix(case, norm, fmap):
    grid, block = case
    q, k, v = _inputs(1, grid)
    M = int(np.prod([g // b for g, b in zip(grid, block)]))
    mc = _mc(2, M)
    a = occ.mhla_causal_head64(q, k, v, mc, grid, block, fmap, norm)
    b = occ.mhla_causal_bruteforce64(q, k, v, mc, grid, block, fmap, norm)
    assert orc.relative_max_error(a, b) < 1e-12


def test_mask_by_hand():
    # 1D, blocks of 2: the order is the sequence order
    np.testing.assert_array_equal(occ.causal_mask((1, 1, 4), (1, 1, 2)), np.tril(np.ones((4, 4))))
    # 2 x 2 grid of 1 x 2 blocks: block 0 = tokens 0, 1; block 1 = tokens 2, 3
    np.testing.assert_array_equal(occ.causal_mask((1, 2, 2), (1, 1, 2)), np.tril(np.ones((4, 4))))
    # 2 x 2 grid of 2 x 1 blocks: block 0 = tokens 0, 2; block 1 = tokens 1, 3
    want = np.array([[1, 0, 0, 0], [1, 1, 1, 0], [1, 0, 1, 0], [1, 1, 1, 1]], float)
    np.testing.assert_array_equal(occ.causal_mask((1, 2, 2), (1, 2, 1)), want)


def test_single_block_is_textbook_causal_linear_attention():
    grid, block = (1, 1, 20), (1, 1, 20)
    q, k, v = _inputs(3, grid)
    pq, pk = orc.feature_map(q), orc.feature_map(k)
    want = np.zeros_like(v)
    for t in range(20):
        w = np.array([pq[t] @ pk[j] for j in range(t + 1)])
        want[t] = (w @ v[: t + 1]) / w.sum()
    got = occ.mhla_causal_head64(q, k, v, np.array([[0.7]]), grid, block)
    assert orc.relative_max_error(got, want) < 1e-12


@pytest.mark.parametrize("norm", ["divisive", "mala"])
def test_first_token_returns_its_value(norm):
    grid, block = (1, 4, 4), (1, 2, 2)
    q, k, v = _inputs(4, grid)
    o = occ.mhla_causal_head64(q, k, v, _mc(5, 4), grid, block, norm=norm)
    np.testing.assert_allclose(o[0], v[0], rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("norm", NORMS)
def test_later_tokens_do_not_change_earlier_outputs(norm):
    grid, block = (1, 6, 8), (1, 3, 2)
    q, k, v = _inputs(6, grid)
    mc = _mc(7, 8)
    C = occ.causal_mask(grid, block)
    base = occ.mhla_causal_head64(q, k, v, mc, grid, block, norm=norm)
    t = 21
    later = np.nonzero(C[t] == 0)[0]          # tokens that come after t
    k2, v2 = k.copy(), v.copy()
    k2[later] += 3.0
    v2[later] -= 2.0
    o2 = occ.mhla_causal_head64(q, k2, v2, mc, grid, block, norm=norm)
    earlier = np.nonzero(C[t] == 1)[0]
    np.testing.assert_array_equal(o2[earlier], base[earlier])
    assert np.max(np.abs(o2[later] - base[later])) > 1e-3


@pytest.mark.parametrize("norm", NORMS)
def test_last_token_of_each_block_matches_non_causal_with_lower_triangular_mc(norm):
    grid, block = (4, 4, 4), (2, 2, 2)
    q, k, v = _inputs(8, grid)
    mc = np.tril(_mc(9, 8))
    causal = occ.mhla_causal_head64(q, k, v, mc, grid, block, norm=norm)
    full = orc.mhla_head64(q, k, v, mc, grid, block, norm=norm)
    bidx = orc.block_of_token(grid, block)
    last = [np.nonzero(bidx == b)[0][-1] for b in range(8)]
    assert orc.relative_max_error(causal[last], full[last]) < 1e-12
    # an earlier token of the same block sees less and differs
    assert np.max(np.abs(causal[last[3] - 1] - full[last[3] - 1])) > 1e-6


def test_mala_causal_rows_sum_to_one():
    grid, block = (1, 6, 8), (1, 3, 2)
    q, k, v = _inputs(10, grid)
    mc = _mc(11, 8)
    # with V = I (N columns) the output rows are the rows of the score matrix
    N = q.shape[0]
    P = occ.mhla_causal_bruteforce64(q, k, np.eye(N), mc, grid, block, norm="mala")
    np.testing.assert_allclose(P.sum(axis=1), 1.0, rtol=1e-12)
    C = occ.causal_mask(grid, block)
    assert np.all(P[C == 0] == 0.0)


def test_planted_mistake_is_caught(monkeypatch):
    grid, block = (1, 1, 12), (1, 1, 4)
    q, k, v = _inputs(12, grid)
    mc = _mc(13, 3)
    orig = occ.mhla_causal_head64

    def wrong(q, k, v, mc, grid, block, fmap="elu1", norm="divisive"):
        mc2 = np.array(mc, float)
        np.fill_diagonal(mc2, 1.0)            # in-block term without its Mc weight
        return orig(q, k, v, mc2, grid, block, fmap, norm)

    monkeypatch.setattr(occ, "mhla_causal_head64", wrong)
    a = occ.mhla_causal_head64(q, k, v, mc, grid, block)
    b = occ.mhla_causal_bruteforce64(q, k, v, mc, grid, block)
    assert orc.relative_max_error(a, b) > 1e-3
