"""Float64 CPU oracle for the token-level multi-head linear attention forward.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` use it.  It shares no code with the CUDA library and imports
nothing but numpy.

What it follows (pages are cited by title and section):

* "MHLA: Restoring Expressivity of Linear Attention via Token-Level
  Multi-Head" (ICLR 2026 notes) -- section "overall framework" (split the N
  tokens into M non-overlapping blocks on the 2D/3D grid; local summaries
  S_b = sum_{j in b} phi(K_j) V_j^T and z_b = sum_{j in b} phi(K_j)), the
  flowchart's output node o = q~^T S~_i / q~^T z~_i, key design 2
  ("Multi-Head Mixing": S~_i = sum_b Mc[i,b] S_b, z~_i = sum_b Mc[i,b] z_b,
  the token-level expansion q~^T S~_i = sum_t Mc[i,b(t)] (q~^T K~_t) V_t^T,
  and dropping the normaliser for long sequences), key design 1 (rank
  bounds), and the background section (positive feature map phi,
  Sim(Q_i, K_j) ~ phi(Q_i) phi(K_j)^T).
* "Rectifying Magnitude Neglect in Linear Attention" (ICCV 2025 notes) --
  section "key designs": Attn(Q_i,K_j) = beta phi(Q_i) phi(K_j)^T - gamma,
  beta = 1 + 1/(phi(Q_i) sum_m phi(K_m)^T), gamma = phi(Q_i) sum_m
  phi(K_m)^T / N, rows sum to 1, and the linear form
  Y_i = beta phi(Q_i) sum_j phi(K_j)^T V_j - gamma sum_j V_j; the ablation
  that names ELU+1 among the feature maps.

Readings taken where the pages are silent (each is listed in the design notes):
  * the output display equation of key design 2 is lost in the page text; the
    flowchart's o = q~^T S~_i / q~^T z~_i is used;
  * phi = ELU(x) + 1 with alpha = 1, applied to Q and K only; no 1/sqrt(d);
  * one Mc [M, M] shared by every batch and head; row = query block;
  * tokens and blocks are numbered in raster order of (T, Hg, Wg);
  * MALA combined with block mixing: every global sum of the MALA page is
    replaced by its Mc-mixed counterpart (sum phi(K)^T V -> S~_i,
    sum phi(K) -> z~_i, sum V -> v~_i, N -> n~_i = sum_b Mc[i,b] n_b); at
    M = 1 with Mc = [[1]] this is the MALA page's formula;
  * no epsilon in any denominator; where a query's denominator
    s = phi(q)^T z~_i is exactly zero (possible with ReLU features, or with a
    zero row of Mc) its output is zero under DIVISIVE and MALA: with
    nonnegative features and Mc, s = 0 forces phi(q)^T S~_i = 0, so this is
    the value the customary guard num / (s + eps) takes for every eps > 0;
  * the MALA page's ablation names ELU+1, ReLU and exp as interchangeable
    feature maps; ReLU is max(x, 0) and exp is e^x elementwise, evaluated
    without any shift (inputs whose exponential overflows are the caller's).

Parity pins (tests/test_oracle_pins.py) tie every function here to facts
outside this file: a hand-derived worked example, the explicit N x N
construction, the M = 1 and Mc = I special cases, MALA's unit row sums,
constant-V, magnitude cancellation, permutation and linearity symmetries,
and the rank bound.
"""

from __future__ import annotations

from typing import Sequence, Tuple

import numpy as np

DIVISIVE = "divisive"
MALA = "mala"
NONE = "none"
NORMS = (DIVISIVE, MALA, NONE)

ELU1 = "elu1"
IDENTITY = "identity"
RELU = "relu"
EXP = "exp"
FEATURE_MAPS = (ELU1, IDENTITY, RELU, EXP)


def feature_map(x, kind: str = ELU1) -> np.ndarray:
    """phi applied elementwise.

    ELU+1 (alpha = 1): x + 1 for x > 0, exp(x) otherwise -- the positive
    feature map of the MHLA page's background section and one of the maps the
    MALA page's ablation names; RELU (max(x, 0)) and EXP (e^x) are the other
    two maps of that ablation.  IDENTITY is phi(x) = x, used only by tests
    that need exact control of phi (the caller keeps features positive).
    """
    x = np.asarray(x, dtype=np.float64)
    if kind == ELU1:
        return np.where(x > 0.0, x + 1.0, np.exp(np.minimum(x, 0.0)))
    if kind == IDENTITY:
        return x.copy()
    if kind == RELU:
        return np.maximum(x, 0.0)
    if kind == EXP:
        return np.exp(x)
    raise ValueError(f"unknown feature map {kind!r}")


def block_of_token(grid: Sequence[int], block: Sequence[int]) -> np.ndarray:
    """Block number b(t) of every token t, tokens and blocks in raster order.

    The MHLA page ("overall framework") splits the tokens into M
    non-overlapping blocks defined on the 2D/3D grid, not on the flattened
    sequence.  Token t = (tau*Hg + y)*Wg + x belongs to block
    ((tau//bt)*(Hg//bh) + y//bh)*(Wg//bw) + x//bw.
    """
    T, Hg, Wg = (int(g) for g in grid)
    bt, bh, bw = (int(b) for b in block)
    if min(T, Hg, Wg, bt, bh, bw) < 1 or T % bt or Hg % bh or Wg % bw:
        raise ValueError(f"block {tuple(block)} does not tile grid {tuple(grid)}")
    tau, y, x = np.meshgrid(np.arange(T), np.arange(Hg), np.arange(Wg), indexing="ij")
    b = ((tau // bt) * (Hg // bh) + y // bh) * (Wg // bw) + x // bw
    return b.ravel().astype(np.int64)


def block_summaries(phik: np.ndarray, v: np.ndarray, bidx: np.ndarray, M: int):
    """Per-block local summaries of one head (MHLA page, "overall framework").

    S_b = sum_{j in b} phi(K_j) V_j^T  [M, d, d]  (row index = feature of phi(K))
    z_b = sum_{j in b} phi(K_j)        [M, d]
    v_b = sum_{j in b} V_j             [M, d]   (needed by the MALA norm)
    n_b = |b|                          [M]
    """
    d = phik.shape[1]
    S = np.zeros((M, d, d))
    z = np.zeros((M, d))
    vs = np.zeros((M, v.shape[1]))
    n = np.zeros(M)
    for b in range(M):
        sel = bidx == b
        S[b] = phik[sel].T @ v[sel]
        z[b] = phik[sel].sum(axis=0)
        vs[b] = v[sel].sum(axis=0)
        n[b] = np.count_nonzero(sel)
    return S, z, vs, n


def mix(mc: np.ndarray, S, z, vs, n):
    """Multi-Head Mixing (MHLA page, key design 2): one product of Mc with the
    stack of block summaries.  S~_i = sum_b Mc[i,b] S_b and likewise for z, v, n.
    """
    mc = np.asarray(mc, dtype=np.float64)
    M = mc.shape[0]
    St = (mc @ S.reshape(M, -1)).reshape(S.shape)
    return St, mc @ z, mc @ vs, mc @ n


def head_output(phiq: np.ndarray, bidx: np.ndarray, St, zt, vt, nt, norm: str) -> np.ndarray:
    """Output of every query of one head, query t in block i = b(t).

    DIVISIVE: o = phi(q)^T S~_i / phi(q)^T z~_i  (MHLA flowchart output node)
    NONE:     o = phi(q)^T S~_i                  (key design 2, normaliser dropped)
    MALA:     s = phi(q)^T z~_i, beta = 1 + 1/s, gamma = s / n~_i,
              o = beta phi(q)^T S~_i - gamma v~_i  (MALA page, linear form,
              global sums replaced by their mixed counterparts)
    A query with s = 0 gets o = 0 under DIVISIVE and MALA (module notes).
    """
    out = np.zeros((phiq.shape[0], St.shape[2]))
    for i in range(St.shape[0]):
        rows = bidx == i
        pq = phiq[rows]
        num = pq @ St[i]
        if norm == NONE:
            out[rows] = num
            continue
        s = pq @ zt[i]
        live = s != 0.0
        inv = np.divide(1.0, s, out=np.zeros_like(s), where=live)
        if norm == DIVISIVE:
            res = num * inv[:, None]
        elif norm == MALA:
            gamma = s / nt[i]
            res = (1.0 + inv)[:, None] * num - gamma[:, None] * vt[i][None, :]
        else:
            raise ValueError(f"unknown norm {norm!r}")
        out[rows] = np.where(live[:, None], res, 0.0)
    return out


def mhla_head64(q, k, v, mc, grid, block, fmap: str = ELU1, norm: str = DIVISIVE) -> np.ndarray:
    """Factored MHLA forward of one (batch, head): q, k, v [N, d] -> o [N, d]."""
    bidx = block_of_token(grid, block)
    M = int(bidx.max()) + 1
    mc = np.asarray(mc, dtype=np.float64)
    if mc.shape != (M, M):
        raise ValueError(f"Mc must be [{M}, {M}], got {mc.shape}")
    phiq = feature_map(q, fmap)
    phik = feature_map(k, fmap)
    v = np.asarray(v, dtype=np.float64)
    S, z, vs, n = block_summaries(phik, v, bidx, M)
    St, zt, vt, nt = mix(mc, S, z, vs, n)
    return head_output(phiq, bidx, St, zt, vt, nt, norm)


def head_mc(mc, hi: int) -> np.ndarray:
    """The mixing matrix of head hi: mc itself when it is [M, M] (one matrix
    shared by every head), mc[hi] when it is [H, M, M] (one per head, shared
    over the batch)."""
    mc = np.asarray(mc)
    return mc[hi] if mc.ndim == 3 else mc


def mhla_forward64(q, k, v, mc, grid, block, fmap: str = ELU1, norm: str = DIVISIVE) -> np.ndarray:
    """Factored MHLA forward over [B, H, N, d] (or [N, d]) inputs, float64 out.

    mc is [M, M] (shared) or [H, M, M] (per head)."""
    q = np.asarray(q)
    if q.ndim == 2:
        return mhla_head64(q, k, v, mc, grid, block, fmap, norm)
    k = np.asarray(k)
    v = np.asarray(v)
    out = np.zeros(q.shape, dtype=np.float64)
    for bi in range(q.shape[0]):
        for hi in range(q.shape[1]):
            out[bi, hi] = mhla_head64(q[bi, hi], k[bi, hi], v[bi, hi], head_mc(mc, hi), grid, block, fmap, norm)
    return out


def attention_matrix64(q, k, mc, grid, block, fmap: str = ELU1) -> np.ndarray:
    """Explicit unnormalised MHLA attention matrix of one head [N, N].

    A[t, j] = Mc[b(t), b(j)] * phi(q_t) . phi(k_j) -- the token-level
    expansion of key design 2 (block selection times intra-block reweighting).
    """
    bidx = block_of_token(grid, block)
    mc = np.asarray(mc, dtype=np.float64)
    return mc[bidx][:, bidx] * (feature_map(q, fmap) @ feature_map(k, fmap).T)


def mhla_bruteforce64(q, k, v, mc, grid, block, fmap: str = ELU1, norm: str = DIVISIVE) -> np.ndarray:
    """O(N^2) construction of one head's output from the explicit matrix.

    Never forms a block summary: it builds A (attention_matrix64) and
      DIVISIVE: o = (A V) / (A 1)
      NONE:     o = A V
      MALA:     P[t,j] = beta_t A[t,j] - gamma_t Mc[b(t),b(j)] with
                s_t = sum_j A[t,j], beta_t = 1 + 1/s_t,
                gamma_t = s_t / sum_j Mc[b(t),b(j)];  o = P V.
    """
    A = attention_matrix64(q, k, mc, grid, block, fmap)
    v = np.asarray(v, dtype=np.float64)
    if norm == NONE:
        return A @ v
    s = A.sum(axis=1)
    if norm == DIVISIVE:
        live = s != 0.0
        return np.where(live[:, None], A @ v, 0.0) * np.divide(1.0, s, out=np.zeros_like(s), where=live)[:, None]
    if norm == MALA:
        return mala_scores64(q, k, mc, grid, block, fmap) @ v
    raise ValueError(f"unknown norm {norm!r}")


def mala_scores64(q, k, mc, grid, block, fmap: str = ELU1) -> np.ndarray:
    """Explicit MALA score matrix P [N, N] with block mixing (see mhla_bruteforce64).

    With a single block and Mc = [[1]] this is the MALA page's
    Attn(Q_i, K_j) = beta phi(Q_i) phi(K_j)^T - gamma, whose rows sum to 1.
    """
    bidx = block_of_token(grid, block)
    mc = np.asarray(mc, dtype=np.float64)
    W = mc[bidx][:, bidx]
    A = W * (feature_map(q, fmap) @ feature_map(k, fmap).T)
    s = A.sum(axis=1)
    live = s != 0.0
    beta = 1.0 + np.divide(1.0, s, out=np.zeros_like(s), where=live)
    gamma = s / W.sum(axis=1)
    # a query with s = 0 has a zero score row (module notes)
    return np.where(live[:, None], beta[:, None] * A - gamma[:, None] * W, 0.0)


def rank_bound(grid, block, d: int) -> int:
    """Upper bound on rank(A_MHLA) from key design 1: min(N, sum_b min(n_b, d))."""
    bidx = block_of_token(grid, block)
    counts = np.bincount(bidx)
    return int(min(bidx.size, sum(min(int(c), d) for c in counts)))


def numerical_rank(A: np.ndarray, rtol: float = 1e-9) -> int:
    """Number of singular values above rtol * sigma_max."""
    s = np.linalg.svd(np.asarray(A, dtype=np.float64), compute_uv=False)
    if s.size == 0 or s[0] == 0.0:
        return 0
    return int(np.count_nonzero(s > rtol * s[0]))


def relative_max_error(got, want) -> float:
    """max|got - want| / max|want|, the parity measure of the GPU tests."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    scale = np.max(np.abs(want)) if want.size else 0.0
    if want.size == 0:
        return 0.0
    return float(np.max(np.abs(got - want)) / (scale if scale > 0 else 1.0))


__all__ = [
    "DIVISIVE", "MALA", "NONE", "NORMS", "ELU1", "IDENTITY", "RELU", "EXP", "FEATURE_MAPS", "feature_map",
    "block_of_token", "block_summaries", "mix", "head_output", "mhla_head64",
    "mhla_forward64", "attention_matrix64", "mhla_bruteforce64", "mala_scores64",
    "rank_bound", "numerical_rank", "relative_max_error", "head_mc",
]
