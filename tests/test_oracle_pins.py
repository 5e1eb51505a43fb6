"""Pins of the float64 oracle to facts outside the oracle itself.

Each test ties an oracle function to something it cannot agree with by
construction: a hand-worked example, an explicit N x N construction written
with plain Python loops, special cases that reduce to textbook linear
attention, invariants the pages state (MALA's unit row sums, the rank bound,
magnitude cancellation) and exact symmetries.  The last group plants
mistakes in the oracle (on the CPU) and checks that a pin catches each one.
"""

import math
import os
from fractions import Fraction

import numpy as np
import pytest


from oracle import mhla_oracle as orc
from token_level_head_phi_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng_inputs(seed, N, d, scale=1.0):
    rng = np.random.default_rng(seed)
    return [scale * rng.standard_normal((N, d)) for _ in range(3)]


def _rand_mc(seed, M, positive=True):
    rng = np.random.default_rng(seed + 7)
    m = rng.uniform(0.05, 1.0, size=(M, M)) if positive else rng.standard_normal((M, M))
    return m / m.sum(axis=1, keepdims=True) if positive else m


# ---------------------------------------------------------------- phi, blocks

def test_feature_map_values():
    # ELU+1 with alpha = 1: x + 1 above zero, exp(x) at and below zero.
    x = np.array([2.0, 0.5, 0.0, -1.0, -3.0, -60.0])
    want = [3.0, 1.5, 1.0, math.exp(-1.0), math.exp(-3.0), math.exp(-60.0)]
    np.testing.assert_allclose(orc.feature_map(x), want, rtol=1e-15, atol=0)
    # continuous at 0, strictly positive, monotone
    assert abs(orc.feature_map(1e-12)[()] - 1.0) < 1e-11
    grid = np.linspace(-30, 30, 10001)
    f = orc.feature_map(grid)
    assert np.all(f > 0) and np.all(np.diff(f) > 0)
    np.testing.assert_array_equal(orc.feature_map(x, orc.IDENTITY), x)


def test_block_of_token_hand_listed():
    # 4x4 grid, 2x2 blocks: rows of the grid read left to right.
    assert orc.block_of_token((1, 4, 4), (1, 2, 2)).tolist() == [
        0, 0, 1, 1,
        0, 0, 1, 1,
        2, 2, 3, 3,
        2, 2, 3, 3]
    # 3D grid (T=2, 2x4), blocks (1, 2, 2): frames are separate block rows.
    assert orc.block_of_token((2, 2, 4), (1, 2, 2)).tolist() == [
        0, 0, 1, 1, 0, 0, 1, 1,
        2, 2, 3, 3, 2, 2, 3, 3]
    # temporal blocks of 2 frames, one spatial block per frame pair
    assert orc.block_of_token((4, 1, 2), (2, 1, 2)).tolist() == [0, 0, 0, 0, 1, 1, 1, 1]
    # 1D sequence, contiguous blocks
    assert orc.block_of_token((1, 1, 6), (1, 1, 2)).tolist() == [0, 0, 1, 1, 2, 2]
    # non-square 2D grid 2x6 with 2x3 blocks
    assert orc.block_of_token((1, 2, 6), (1, 2, 3)).tolist() == [0, 0, 0, 1, 1, 1, 0, 0, 0, 1, 1, 1]
    with pytest.raises(ValueError):
        orc.block_of_token((1, 5, 4), (1, 2, 2))


# ---------------------------------------------------------- worked example

def _load_worked_example():
    inputs, expect = {}, {}
    with open(os.path.join(GOLDEN, "worked_example_d2.txt")) as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            parts = line.split()
            if parts[0] == "input":
                inputs[parts[1]] = np.array([float(Fraction(p)) for p in parts[2:]])
            else:
                expect.setdefault(parts[0], {})[int(parts[1])] = [Fraction(p) for p in parts[2:]]
    q = inputs["q"].reshape(4, 2)
    k = inputs["k"].reshape(4, 2)
    v = inputs["v"].reshape(4, 2)
    mc = inputs["mc"].reshape(2, 2)
    return q, k, v, mc, expect


@pytest.mark.parametrize("norm", orc.NORMS)
def test_worked_example_hand_derived(norm):
    q, k, v, mc, expect = _load_worked_example()
    for fn in (orc.mhla_head64, orc.mhla_bruteforce64):
        o = fn(q, k, v, mc, (1, 1, 4), (1, 1, 2), norm=norm)
        for t, row in expect[norm].items():
            np.testing.assert_allclose(o[t], [float(x) for x in row], rtol=1e-13, atol=1e-14)


# ----------------------------------------------- explicit construction (loops)

def _loop_output(q, k, v, mc, grid, block, norm, fmap=orc.ELU1):
    """Token-level expansion of key design 2 written with Python loops.

    For query t in block i: weights w_j = Mc[i, b(j)] * sum_k phi(q_t)[k] phi(k_j)[k].
    """
    bidx = orc.block_of_token(grid, block).tolist()
    pq = orc.feature_map(q, fmap)
    pk = orc.feature_map(k, fmap)
    N, d = q.shape
    out = np.zeros((N, v.shape[1]))
    for t in range(N):
        i = bidx[t]
        w = [mc[i][bidx[j]] * sum(pq[t][a] * pk[j][a] for a in range(d)) for j in range(N)]
        s = sum(w)
        if norm == orc.MALA:
            nt = sum(mc[i][bidx[j]] for j in range(N))
            w = [(1.0 + 1.0 / s) * w[j] - (s / nt) * mc[i][bidx[j]] for j in range(N)]
        for c in range(v.shape[1]):
            acc = sum(w[j] * v[j][c] for j in range(N))
            out[t][c] = acc / s if norm == orc.DIVISIVE else acc
    return out


CASES = [
    # grid, block, d
    ((1, 1, 12), (1, 1, 4), 3),
    ((1, 6, 6), (1, 3, 3), 4),
    ((2, 4, 4), (1, 2, 2), 2),
    ((4, 2, 6), (2, 2, 3), 5),
    ((1, 2, 6), (1, 2, 3), 3),
]


@pytest.mark.parametrize("norm", orc.NORMS)
@pytest.mark.parametrize("case", CASES)
def test_factored_equals_loop_expansion(case, norm):
    grid, block, d = case
    N = grid[0] * grid[1] * grid[2]
    M = N // (block[0] * block[1] * block[2])
    q, k, v = _rng_inputs(hash((grid, block, d)) % 1000, N, d)
    mc = _rand_mc(3, M)
    want = _loop_output(q, k, v, mc, grid, block, norm)
    got = orc.mhla_head64(q, k, v, mc, grid, block, norm=norm)
    brute = orc.mhla_bruteforce64(q, k, v, mc, grid, block, norm=norm)
    assert orc.relative_max_error(got, want) < 1e-12
    assert orc.relative_max_error(brute, want) < 1e-12


@pytest.mark.parametrize("norm", orc.NORMS)
def test_factored_equals_bruteforce_tiny_config(norm):
    w = wl.WORKLOADS["tiny_f32"]
    q, k, v = wl.head_inputs(w, 0)
    mc = wl.make_mc(w)
    got = orc.mhla_head64(q, k, v, mc, w.grid, w.block, norm=norm)
    brute = orc.mhla_bruteforce64(q, k, v, mc, w.grid, w.block, norm=norm)
    assert orc.relative_max_error(got, brute) < 1e-12


def test_factored_equals_bruteforce_deit_head():
    w = wl.WORKLOADS["deit_t"]
    q, k, v = wl.head_inputs(w, 5)
    mc = wl.make_mc(w)
    for norm in orc.NORMS:
        got = orc.mhla_head64(q, k, v, mc, w.grid, w.block, norm=norm)
        brute = orc.mhla_bruteforce64(q, k, v, mc, w.grid, w.block, norm=norm)
        assert orc.relative_max_error(got, brute) < 1e-11


# --------------------------------------------------------- special cases

def _global_la_loops(q, k, v, fmap=orc.ELU1):
    """Textbook linear attention (MHLA page background): o_t =
    sum_j (phi(q_t).phi(k_j)) v_j / sum_j phi(q_t).phi(k_j), by loops."""
    pq, pk = orc.feature_map(q, fmap), orc.feature_map(k, fmap)
    N = q.shape[0]
    out = np.zeros((N, v.shape[1]))
    for t in range(N):
        w = [float(np.dot(pq[t], pk[j])) for j in range(N)]
        out[t] = sum(w[j] * v[j] for j in range(N)) / sum(w)
    return out


def test_single_block_is_global_linear_attention():
    q, k, v = _rng_inputs(11, 40, 4)
    want = _global_la_loops(q, k, v)
    for m in (1.0, 0.3, 7.0):  # any positive scalar Mc cancels
        got = orc.mhla_head64(q, k, v, np.array([[m]]), (1, 1, 40), (1, 1, 40))
        assert orc.relative_max_error(got, want) < 1e-12


def test_identity_mixing_is_block_local():
    grid, block, d = (1, 6, 6), (1, 3, 2), 3
    N = 36
    q, k, v = _rng_inputs(12, N, d)
    bidx = orc.block_of_token(grid, block)
    M = int(bidx.max()) + 1
    got = orc.mhla_head64(q, k, v, np.eye(M), grid, block)
    for b in range(M):
        sel = bidx == b
        want = _global_la_loops(q[sel], k[sel], v[sel])
        assert orc.relative_max_error(got[sel], want) < 1e-12


def test_uniform_mixing_is_global_for_any_partition():
    q, k, v = _rng_inputs(13, 48, 4)
    want = _global_la_loops(q, k, v)
    for grid, block in [((1, 1, 48), (1, 1, 6)), ((1, 6, 8), (1, 3, 4)), ((3, 4, 4), (1, 2, 2))]:
        M = 48 // (block[0] * block[1] * block[2])
        got = orc.mhla_head64(q, k, v, np.full((M, M), 0.37), grid, block)
        assert orc.relative_max_error(got, want) < 1e-12


def test_divisive_invariant_to_positive_row_scaling_of_mc():
    grid, block = (1, 8, 8), (1, 4, 4)
    q, k, v = _rng_inputs(14, 64, 8)
    mc = _rand_mc(5, 4)
    scale = np.array([0.5, 3.0, 1.0, 11.0])[:, None]
    a = orc.mhla_head64(q, k, v, mc, grid, block)
    b = orc.mhla_head64(q, k, v, mc * scale, grid, block)
    assert orc.relative_max_error(b, a) < 1e-13


# ------------------------------------------------------------------ MALA

def test_mala_rows_sum_to_one():
    for grid, block in [((1, 1, 32), (1, 1, 32)), ((1, 8, 8), (1, 4, 4)), ((2, 4, 4), (1, 2, 2))]:
        N = grid[0] * grid[1] * grid[2]
        M = N // (block[0] * block[1] * block[2])
        q, k, _ = _rng_inputs(15 + N, N, 6)
        P = orc.mala_scores64(q, k, _rand_mc(2, M), grid, block)
        np.testing.assert_allclose(P.sum(axis=1), 1.0, rtol=0, atol=1e-12)


def test_mala_single_block_is_page_formula():
    """M = 1, Mc = [[1]]: Y_i = beta phi(Q_i) sum_j phi(K_j)^T V_j - gamma sum_j V_j,
    beta = 1 + 1/(phi(Q_i) sum_m phi(K_m)^T), gamma = phi(Q_i) sum_m phi(K_m)^T / N."""
    N, d = 30, 4
    q, k, v = _rng_inputs(16, N, d)
    pq, pk = orc.feature_map(q), orc.feature_map(k)
    ksum = [sum(pk[m][a] for m in range(N)) for a in range(d)]
    kv = [[sum(pk[j][a] * v[j][c] for j in range(N)) for c in range(d)] for a in range(d)]
    vsum = [sum(v[j][c] for j in range(N)) for c in range(d)]
    want = np.zeros((N, d))
    for i in range(N):
        s = sum(pq[i][a] * ksum[a] for a in range(d))
        beta, gamma = 1.0 + 1.0 / s, s / N
        for c in range(d):
            want[i][c] = beta * sum(pq[i][a] * kv[a][c] for a in range(d)) - gamma * vsum[c]
    got = orc.mhla_head64(q, k, v, np.array([[1.0]]), (1, 1, N), (1, 1, N), norm=orc.MALA)
    assert orc.relative_max_error(got, want) < 1e-12


def test_mala_magnitude_sharpens_scores():
    """Scaling ||phi(Q_i)|| by a > 1 raises the high/low score ratio (MALA page)."""
    N, d = 24, 4
    rng = np.random.default_rng(17)
    q = rng.uniform(0.2, 1.5, (N, d))
    k = rng.uniform(0.2, 1.5, (N, d))
    grid = block = (1, 1, N)
    P1 = orc.mala_scores64(q, k, np.array([[1.0]]), grid, block, fmap=orc.IDENTITY)
    P2 = orc.mala_scores64(3.0 * q, k, np.array([[1.0]]), grid, block, fmap=orc.IDENTITY)
    for i in range(N):
        hi, lo = np.argmax(P1[i]), np.argmin(P1[i])
        if P1[i, lo] > 0:
            assert P2[i, hi] / P2[i, lo] > P1[i, hi] / P1[i, lo]
    # divisive linear attention ignores the magnitude entirely
    v = rng.standard_normal((N, d))
    a = orc.mhla_head64(q, k, v, np.array([[1.0]]), grid, block, fmap=orc.IDENTITY)
    b = orc.mhla_head64(3.0 * q, k, v, np.array([[1.0]]), grid, block, fmap=orc.IDENTITY)
    assert orc.relative_max_error(b, a) < 1e-13


# ------------------------------------------------------------ symmetries

@pytest.mark.parametrize("norm", [orc.DIVISIVE, orc.MALA])
def test_constant_values_pass_through(norm):
    grid, block = (2, 4, 4), (1, 2, 2)
    q, k, _ = _rng_inputs(18, 32, 5)
    c = np.array([0.25, -1.5, 3.0, 0.0, 2.0])
    v = np.tile(c, (32, 1))
    got = orc.mhla_head64(q, k, v, _rand_mc(4, 8), grid, block, norm=norm)
    np.testing.assert_allclose(got, v, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("norm", orc.NORMS)
def test_permutation_within_blocks(norm):
    grid, block = (1, 6, 6), (1, 3, 3)
    q, k, v = _rng_inputs(19, 36, 4)
    mc = _rand_mc(6, 4)
    bidx = orc.block_of_token(grid, block)
    base = orc.mhla_head64(q, k, v, mc, grid, block, norm=norm)
    rng = np.random.default_rng(0)
    perm = np.arange(36)
    for b in range(4):
        idx = np.flatnonzero(bidx == b)
        perm[idx] = rng.permutation(idx)
    # keys/values shuffled inside their blocks: outputs unchanged
    o1 = orc.mhla_head64(q, k[perm], v[perm], mc, grid, block, norm=norm)
    assert orc.relative_max_error(o1, base) < 1e-12
    # queries shuffled inside their blocks: outputs shuffled the same way
    o2 = orc.mhla_head64(q[perm], k, v, mc, grid, block, norm=norm)
    assert orc.relative_max_error(o2, base[perm]) < 1e-12


@pytest.mark.parametrize("norm", orc.NORMS)
def test_linear_in_values(norm):
    grid, block = (1, 4, 8), (1, 2, 4)
    q, k, v1 = _rng_inputs(20, 32, 3)
    v2 = np.random.default_rng(21).standard_normal((32, 3))
    mc = _rand_mc(7, 4)
    f = lambda vv: orc.mhla_head64(q, k, vv, mc, grid, block, norm=norm)  # noqa: E731
    assert orc.relative_max_error(f(2.0 * v1 - 0.5 * v2), 2.0 * f(v1) - 0.5 * f(v2)) < 1e-12


# ------------------------------------------------------------------ rank

def test_rank_bound_and_collapse():
    """Key design 1: rank(A_lin) <= d, rank(A_MHLA) <= min(N, sum_b min(n_b, d))."""
    grid, block, d = (1, 8, 8), (1, 4, 4), 4
    q, k, _ = _rng_inputs(22, 64, d)
    mc = _rand_mc(8, 4)
    A = orc.attention_matrix64(q, k, mc, grid, block)
    bound = orc.rank_bound(grid, block, d)
    assert bound == 16
    r = orc.numerical_rank(A)
    assert r <= bound
    assert r == bound  # generic inputs reach it
    A_lin = orc.attention_matrix64(q, k, np.array([[1.0]]), grid, grid)
    assert orc.numerical_rank(A_lin) <= d
    # small blocks: n_b < d caps each block's contribution
    assert orc.rank_bound((1, 1, 12), (1, 1, 2), 4) == 12
    assert orc.rank_bound((1, 1, 12), (1, 1, 6), 4) == 8


# ------------------------------------------------- planted mistakes caught

def _pins_pass():
    """Worked example + loop expansion on one case; True when both hold."""
    try:
        for norm in orc.NORMS:
            test_worked_example_hand_derived(norm)
            test_factored_equals_loop_expansion(CASES[1], norm)
            test_factored_equals_loop_expansion(CASES[2], norm)
        test_mala_rows_sum_to_one()
    except AssertionError:
        return False
    return True


def test_pins_pass_unmodified():
    assert _pins_pass()


@pytest.mark.parametrize("mistake", ["mc_transposed", "summary_transposed", "no_denominator",
                                     "mala_gamma_sign", "phi_without_plus_one", "block_index_swapped"])
def test_planted_mistake_is_caught(monkeypatch, mistake):
    if mistake == "mc_transposed":
        orig = orc.mix
        monkeypatch.setattr(orc, "mix", lambda mc, *a: orig(np.asarray(mc).T, *a))
    elif mistake == "summary_transposed":
        orig = orc.block_summaries

        def bad(phik, v, bidx, M):
            S, z, vs, n = orig(phik, v, bidx, M)
            return S.transpose(0, 2, 1).copy(), z, vs, n
        monkeypatch.setattr(orc, "block_summaries", bad)
    elif mistake == "no_denominator":
        orig = orc.head_output
        monkeypatch.setattr(orc, "head_output",
                            lambda pq, b, St, zt, vt, nt, norm: orig(pq, b, St, zt, vt, nt,
                                                                     orc.NONE if norm == orc.DIVISIVE else norm))
    elif mistake == "mala_gamma_sign":
        orig = orc.head_output
        monkeypatch.setattr(orc, "head_output",
                            lambda pq, b, St, zt, vt, nt, norm: orig(pq, b, St, zt, -vt if norm == orc.MALA else vt,
                                                                     nt, norm))
    elif mistake == "phi_without_plus_one":
        orig = orc.feature_map
        monkeypatch.setattr(orc, "feature_map",
                            lambda x, kind=orc.ELU1: orig(x, kind) - (1.0 if kind == orc.ELU1 else 0.0))
    elif mistake == "block_index_swapped":
        orig = orc.block_of_token
        monkeypatch.setattr(orc, "block_of_token", lambda g, b: orig(g, b)[::-1].copy())
    caught = not _pins_pass()
    if mistake == "phi_without_plus_one":
        with pytest.raises(AssertionError):
            test_feature_map_values()
        caught = True
    if mistake == "block_index_swapped":
        with pytest.raises(AssertionError):
            test_block_of_token_hand_listed()
        caught = True
    assert caught
