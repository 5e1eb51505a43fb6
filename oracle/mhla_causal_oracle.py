"""Float64 CPU oracle for causal (block-ordered) MHLA.

TEST INFRASTRUCTURE ONLY, like ``mhla_oracle``: only ``tests/`` (and the
benchmark's CPU-baseline leg) use it; it shares no code with the CUDA library
and imports nothing but numpy and the forward oracle.

The MHLA page mentions a chunkwise, streaming form of the method for
autoregressive use (key design 2's long-sequence remarks, and the summaries
being additive) but defines no causal variant, so this module takes the
plainest reading that the rest of the method supports:

  * tokens are ordered by (block index, position inside the block), blocks in
    raster order of the block grid and tokens in raster order inside a block
    (for a 1D sequence this is the sequence order);
  * query t in block i sees token j iff j comes no later than t in that order;
    the pair is weighted as in the non-causal method, A[t, j] =
    Mc[i, b(j)] phi(q_t) . phi(k_j): earlier blocks b < i through the strict
    lower triangle of Mc, block i itself through Mc[i, i] and only its tokens
    up to t;
  * every norm uses the same causal sums: with the prefix states
    S~_t = sum_{b<i} Mc[i,b] S_b + Mc[i,i] sum_{j in i, j <= t} phi(k_j) v_j^T
    (z~_t, v~_t, n~_t likewise), DIVISIVE o = phi(q)^T S~_t / phi(q)^T z~_t,
    NONE o = phi(q)^T S~_t, MALA o = beta phi(q)^T S~_t - gamma v~_t with
    s = phi(q)^T z~_t, beta = 1 + 1/s, gamma = s / n~_t (rows of the score
    matrix still sum to 1); s = 0 gives o = 0 as in the non-causal oracle.

``mhla_causal_head64`` runs the prefix recursion token by token;
``mhla_causal_bruteforce64`` masks the explicit N x N matrix instead.
"""

from __future__ import annotations

import numpy as np

from .mhla_oracle import (DIVISIVE, ELU1, MALA, NONE, block_of_token, block_summaries, feature_map, head_mc, mix)


def causal_mask(grid, block) -> np.ndarray:
    """C[t, j] = 1 iff token j comes no later than token t in (block, local) order."""
    bidx = block_of_token(grid, block)
    N = bidx.shape[0]
    # position inside the block: tokens of a block, taken in increasing global
    # index, are in raster order inside the block
    local = np.zeros(N, dtype=np.int64)
    for b in range(int(bidx.max()) + 1):
        sel = np.nonzero(bidx == b)[0]
        local[sel] = np.arange(sel.shape[0])
    key = bidx * N + local
    return (key[None, :] <= key[:, None]).astype(np.float64)


def _token_output(pq, St, zt, vt, nt, norm):
    num = pq @ St
    if norm == NONE:
        return num
    s = pq @ zt
    if s == 0.0:
        return np.zeros_like(num)
    if norm == DIVISIVE:
        return num / s
    if norm == MALA:
        return (1.0 + 1.0 / s) * num - (s / nt) * vt
    raise ValueError(f"unknown norm {norm!r}")


def mhla_causal_head64(q, k, v, mc, grid, block, fmap: str = ELU1, norm: str = DIVISIVE) -> np.ndarray:
    """Causal MHLA of one head by the prefix recursion: q, k, v [N, d] -> o [N, d]."""
    bidx = block_of_token(grid, block)
    M = int(bidx.max()) + 1
    mc = np.asarray(mc, dtype=np.float64)
    phq = feature_map(q, fmap)
    phk = feature_map(k, fmap)
    v = np.asarray(v, dtype=np.float64)
    S, z, vs, n = block_summaries(phk, v, bidx, M)
    # earlier blocks only: the strict lower triangle of Mc
    Sp, zp, vp, npre = mix(np.tril(mc, -1), S, z, vs, n)
    out = np.zeros((q.shape[0], v.shape[1]))
    for i in range(M):
        w = mc[i, i]
        rS = np.zeros_like(S[0])
        rz = np.zeros_like(z[0])
        rv = np.zeros_like(vs[0])
        rn = 0.0
        for t in np.nonzero(bidx == i)[0]:
            rS += np.outer(phk[t], v[t])
            rz += phk[t]
            rv += v[t]
            rn += 1.0
            out[t] = _token_output(phq[t], Sp[i] + w * rS, zp[i] + w * rz, vp[i] + w * rv, npre[i] + w * rn, norm)
    return out


def mhla_causal_bruteforce64(q, k, v, mc, grid, block, fmap: str = ELU1, norm: str = DIVISIVE) -> np.ndarray:
    """Causal MHLA of one head from the masked explicit matrix.

    A = C * W * (phi(q) phi(k)^T), W[t,j] = Mc[b(t), b(j)], C the causal mask;
    DIVISIVE o = (A V) / (A 1); NONE o = A V; MALA P = beta A - gamma (C * W)
    with s = A 1, beta = 1 + 1/s, gamma = s / ((C * W) 1), o = P V.
    """
    bidx = block_of_token(grid, block)
    mc = np.asarray(mc, dtype=np.float64)
    C = causal_mask(grid, block)
    W = C * mc[bidx][:, bidx]
    A = W * (feature_map(q, fmap) @ feature_map(k, fmap).T)
    v = np.asarray(v, dtype=np.float64)
    if norm == NONE:
        return A @ v
    s = A.sum(axis=1)
    live = s != 0.0
    inv = np.divide(1.0, s, out=np.zeros_like(s), where=live)
    if norm == DIVISIVE:
        return np.where(live[:, None], (A @ v) * inv[:, None], 0.0)
    if norm == MALA:
        P = (1.0 + inv)[:, None] * A - (s / W.sum(axis=1))[:, None] * W
        return np.where(live[:, None], P @ v, 0.0)
    raise ValueError(f"unknown norm {norm!r}")


def mhla_causal_forward64(q, k, v, mc, grid, block, fmap: str = ELU1, norm: str = DIVISIVE) -> np.ndarray:
    """Causal MHLA over [B, H, N, d] (or [N, d]) inputs, float64 out."""
    q = np.asarray(q)
    if q.ndim == 2:
        return mhla_causal_head64(q, k, v, mc, grid, block, fmap, norm)
    out = np.zeros(q.shape, dtype=np.float64)
    for bi in range(q.shape[0]):
        for hi in range(q.shape[1]):
            out[bi, hi] = mhla_causal_head64(q[bi, hi], k[bi, hi], v[bi, hi], head_mc(mc, hi), grid, block, fmap,
                                             norm)
    return out


__all__ = ["causal_mask", "mhla_causal_head64", "mhla_causal_bruteforce64", "mhla_causal_forward64"]
