"""Pins of per-head mixing matrices (Mc [H, M, M], one per head, shared over
the batch) in the batched oracle entry points (CPU only): H identical copies
reproduce the shared-Mc results, each head of a per-head call equals a
single-head call with its own matrix, and dMc [H, M, M] sums over the batch
only -- its sum over heads is the shared-Mc gradient when the copies agree."""

import numpy as np

from oracle import mhla_backward_oracle as orb
from oracle import mhla_causal_oracle as occ
from oracle import mhla_oracle as orc

GRID, BLOCK, D = (1, 4, 6), (1, 2, 3), 3


def _inputs(seed, B=2, H=3):
    rng = np.random.default_rng(seed)
    N = int(np.prod(GRID))
    q, k, v, g = (rng.standard_normal((B, H, N, D)) for _ in range(4))
    mcs = rng.uniform(0.1, 1.0, (H, 4, 4))
    return q, k, v, g, mcs


def test_identical_copies_reproduce_shared_mc():
    q, k, v, g, mcs = _inputs(1)
    shared = mcs[0]
    copies = np.stack([shared] * 3)
    for norm in ("divisive", "none", "mala"):
        np.testing.assert_array_equal(orc.mhla_forward64(q, k, v, copies, GRID, BLOCK, norm=norm),
                                      orc.mhla_forward64(q, k, v, shared, GRID, BLOCK, norm=norm))
        np.testing.assert_array_equal(occ.mhla_causal_forward64(q, k, v, copies, GRID, BLOCK, norm=norm),
                                      occ.mhla_causal_forward64(q, k, v, shared, GRID, BLOCK, norm=norm))
    a = orb.mhla_backward64(q, k, v, copies, GRID, BLOCK, g)
    b = orb.mhla_backward64(q, k, v, shared, GRID, BLOCK, g)
    for x, y in zip(a[:3], b[:3]):
        np.testing.assert_array_equal(x, y)
    assert a[3].shape == (3, 4, 4)
    np.testing.assert_allclose(a[3].sum(axis=0), b[3], rtol=1e-12)


def test_each_head_uses_its_own_matrix():
    q, k, v, g, mcs = _inputs(2)
    o = orc.mhla_forward64(q, k, v, mcs, GRID, BLOCK)
    for b in range(2):
        for h in range(3):
            want = orc.mhla_head64(q[b, h], k[b, h], v[b, h], mcs[h], GRID, BLOCK)
            np.testing.assert_array_equal(o[b, h], want)
    # the heads' matrices differ, so reusing head 0's matrix changes heads 1, 2
    wrong = orc.mhla_forward64(q, k, v, np.stack([mcs[0]] * 3), GRID, BLOCK)
    assert np.max(np.abs(wrong[:, 1:] - o[:, 1:])) > 1e-6


def test_per_head_gradient_sums_over_batch_only():
    q, k, v, g, mcs = _inputs(3)
    dmc = orb.mhla_backward64(q, k, v, mcs, GRID, BLOCK, g)[3]
    for h in range(3):
        want = sum(orb.mhla_head_backward64(q[b, h], k[b, h], v[b, h], mcs[h], GRID, BLOCK, g[b, h])[3]
                   for b in range(2))
        np.testing.assert_allclose(dmc[h], want, rtol=1e-13)
