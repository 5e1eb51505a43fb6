"""Float64 CPU oracle for the gradients of the MHLA forward pass.

TEST INFRASTRUCTURE ONLY, like ``mhla_oracle``: only ``tests/`` (and the
benchmark's CPU-baseline leg) use it; it shares no code with the CUDA library
and imports nothing but numpy and the forward oracle.

What it differentiates is the forward of ``mhla_oracle`` ("MHLA: Restoring
Expressivity of Linear Attention via Token-Level Multi-Head", overall
framework, flowchart output node and key design 2; "Rectifying Magnitude
Neglect in Linear Attention", key designs, for the MALA norm).  The MHLA page
says Mc is learned end to end together with the rest of the network, which
needs the gradients with respect to Q, K, V and Mc; the pages print no
formula for them, so they are the plain chain rule of the forward steps:

  forward (one head; token t in query block i = b(t), token j in block b):
    phq = phi(q), phk = phi(k)
    S_b = sum_j phk_j v_j^T,  z_b = sum_j phk_j,  v_b = sum_j v_j,  n_b = |b|
    S~_i = sum_b Mc[i,b] S_b  (and z~, v~, n~ likewise)
    num_t = phq_t^T S~_i,  s_t = phq_t . z~_i
    DIVISIVE o_t = num_t / s_t;  NONE o_t = num_t;
    MALA     o_t = (1 + 1/s_t) num_t - (s_t / n~_i) v~_i

  backward, given dO (the gradient of the loss with respect to o):
    output step:  dnum_t, ds_t from the norm; dphq_t = S~_i dnum_t + z~_i ds_t
                  dS~_i = sum_t phq_t dnum_t^T, dz~_i = sum_t ds_t phq_t
                  (MALA also dv~_i = -sum_t gamma_t dO_t and dn~_i)
    mixing:       dS_b = sum_i Mc[i,b] dS~_i (z, v likewise)
                  dMc[i,b] = <dS~_i, S_b> + <dz~_i, z_b> + <dv~_i, v_b> + dn~_i n_b
    summaries:    dphk_j = dS_b v_j + dz_b,  dv_j = dS_b^T phk_j + dv_b
    feature map:  dq = dphq * phi'(q), dk = dphk * phi'(k)

A query whose denominator s is exactly zero has output 0 (the forward
oracle's rule); its output is then constant and it contributes nothing to
any gradient.  phi' of ReLU is taken as 0 at x = 0 (a subgradient).

``mhla_bruteforce_backward64`` differentiates the explicit N x N form instead
(A[t,j] = Mc[b(t),b(j)] phq_t . phk_j), never forming a summary; tests pin
both against each other and against finite differences of the forward.
"""

from __future__ import annotations

import numpy as np

from .mhla_oracle import (DIVISIVE, ELU1, EXP, IDENTITY, MALA, NONE, RELU, block_of_token, block_summaries,
                          feature_map, head_mc, mix)


def feature_map_grad(x, kind: str = ELU1) -> np.ndarray:
    """phi'(x): 1 for x > 0 and exp(x) otherwise (ELU+1, alpha = 1); 1 for
    IDENTITY; 1 for x > 0 and 0 otherwise (ReLU); exp(x) (exp).

    At x = 0 both sides of ELU+1 give 1, so it is differentiable everywhere.
    """
    x = np.asarray(x, dtype=np.float64)
    if kind == ELU1:
        return np.where(x > 0.0, 1.0, np.exp(np.minimum(x, 0.0)))
    if kind == IDENTITY:
        return np.ones_like(x)
    if kind == RELU:
        return np.where(x > 0.0, 1.0, 0.0)
    if kind == EXP:
        return np.exp(x)
    raise ValueError(f"unknown feature map {kind!r}")


def mhla_head_backward64(q, k, v, mc, grid, block, dout, fmap: str = ELU1, norm: str = DIVISIVE):
    """Gradients of one head's factored forward: returns (dq, dk, dv, dmc)."""
    bidx = block_of_token(grid, block)
    M = int(bidx.max()) + 1
    mc = np.asarray(mc, dtype=np.float64)
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    dout = np.asarray(dout, dtype=np.float64)
    phq = feature_map(q, fmap)
    phk = feature_map(k, fmap)
    S, z, vs, n = block_summaries(phk, v, bidx, M)
    St, zt, vt, nt = mix(mc, S, z, vs, n)

    d, dv_dim = S.shape[1], S.shape[2]
    dphq = np.zeros_like(phq)
    dSt = np.zeros_like(St)
    dzt = np.zeros_like(zt)
    dvt = np.zeros_like(vt)
    dnt = np.zeros_like(nt)
    for i in range(M):
        rows = bidx == i
        pq = phq[rows]
        g = dout[rows]
        num = pq @ St[i]
        if norm == NONE:
            dnum = g
            ds = np.zeros(pq.shape[0])
        else:
            s = pq @ zt[i]
            # queries with s = 0 have a constant (zero) output: no gradient
            live = s != 0.0
            g = np.where(live[:, None], g, 0.0)
            inv = np.divide(1.0, s, out=np.zeros_like(s), where=live)
            if norm == DIVISIVE:
                o = num * inv[:, None]
                dnum = g * inv[:, None]
                ds = -np.sum(g * o, axis=1) * inv
            elif norm == MALA:
                beta = 1.0 + inv
                gamma = s / nt[i]
                dnum = beta[:, None] * g
                dbeta = np.sum(g * num, axis=1)
                dgamma = -(g @ vt[i])
                ds = -dbeta * inv ** 2 + dgamma / nt[i]
                dvt[i] = -(gamma[:, None] * g).sum(axis=0)
                dnt[i] = -np.sum(dgamma * s) / nt[i] ** 2
            else:
                raise ValueError(f"unknown norm {norm!r}")
        dphq[rows] = dnum @ St[i].T + ds[:, None] * zt[i][None, :]
        dSt[i] = pq.T @ dnum
        dzt[i] = pq.T @ ds

    # mixing: each summary gathers the gradients of every query block that mixed it
    dS = (mc.T @ dSt.reshape(M, -1)).reshape(M, d, dv_dim)
    dz = mc.T @ dzt
    dvs = mc.T @ dvt
    dmc = (dSt.reshape(M, -1) @ S.reshape(M, -1).T + dzt @ z.T + dvt @ vs.T + np.outer(dnt, n))

    dphk = np.zeros_like(phk)
    dv = np.zeros_like(v)
    for b in range(M):
        sel = bidx == b
        dphk[sel] = v[sel] @ dS[b].T + dz[b][None, :]
        dv[sel] = phk[sel] @ dS[b] + dvs[b][None, :]
    return dphq * feature_map_grad(q, fmap), dphk * feature_map_grad(k, fmap), dv, dmc


def mhla_bruteforce_backward64(q, k, v, mc, grid, block, dout, fmap: str = ELU1, norm: str = DIVISIVE):
    """Gradients of the explicit O(N^2) form (see mhla_bruteforce64): (dq, dk, dv, dmc).

    A = W * (phq phk^T) with W[t,j] = Mc[b(t),b(j)].
      DIVISIVE: o = P V, P = A / rowsum(A);  NONE: o = A V;
      MALA: P = beta A - gamma W, s = rowsum(A), beta = 1 + 1/s,
            gamma = s / rowsum(W);  o = P V.
    """
    bidx = block_of_token(grid, block)
    M = int(bidx.max()) + 1
    mc = np.asarray(mc, dtype=np.float64)
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    dout = np.asarray(dout, dtype=np.float64)
    phq = feature_map(q, fmap)
    phk = feature_map(k, fmap)
    W = mc[bidx][:, bidx]
    G = phq @ phk.T
    A = W * G
    if norm == NONE:
        dv = A.T @ dout
        dA = dout @ v.T
        dW = np.zeros_like(W)
    elif norm == DIVISIVE:
        s = A.sum(axis=1)
        live = s != 0.0
        inv = np.divide(1.0, s, out=np.zeros_like(s), where=live)
        P = A * inv[:, None]
        o = P @ v
        dv = P.T @ dout
        dA = (dout @ v.T - np.sum(dout * o, axis=1)[:, None]) * inv[:, None]
        dW = np.zeros_like(W)
    elif norm == MALA:
        s = A.sum(axis=1)
        live = s != 0.0
        inv = np.divide(1.0, s, out=np.zeros_like(s), where=live)
        w = W.sum(axis=1)
        beta = 1.0 + inv
        gamma = s / w
        P = np.where(live[:, None], beta[:, None] * A - gamma[:, None] * W, 0.0)
        dv = P.T @ dout
        dP = np.where(live[:, None], dout @ v.T, 0.0)
        dbeta = np.sum(dP * A, axis=1)
        dgamma = -np.sum(dP * W, axis=1)
        ds = -dbeta * inv ** 2 + dgamma / w
        dw = -dgamma * s / w ** 2
        dA = beta[:, None] * dP + ds[:, None]
        dW = -gamma[:, None] * dP + dw[:, None]
    else:
        raise ValueError(f"unknown norm {norm!r}")
    dW = dW + dA * G
    dG = dA * W
    dphq = dG @ phk
    dphk = dG.T @ phq
    dmc = np.zeros((M, M))
    np.add.at(dmc, (bidx[:, None], bidx[None, :]), dW)
    return dphq * feature_map_grad(q, fmap), dphk * feature_map_grad(k, fmap), dv, dmc


def mhla_backward64(q, k, v, mc, grid, block, dout, fmap: str = ELU1, norm: str = DIVISIVE):
    """Gradients over [B, H, N, d] inputs: dq, dk, dv [B, H, N, d] and dmc
    shaped like mc -- [M, M] summed over every (batch, head) when one Mc is
    shared, [H, M, M] summed over the batch when each head has its own."""
    q = np.asarray(q)
    if q.ndim == 2:
        return mhla_head_backward64(q, k, v, mc, grid, block, dout, fmap, norm)
    k, v, dout = np.asarray(k), np.asarray(v), np.asarray(dout)
    dq = np.zeros(q.shape)
    dk = np.zeros(q.shape)
    dv = np.zeros(v.shape)
    dmc = np.zeros(np.asarray(mc).shape)
    for bi in range(q.shape[0]):
        for hi in range(q.shape[1]):
            g = mhla_head_backward64(q[bi, hi], k[bi, hi], v[bi, hi], head_mc(mc, hi), grid, block, dout[bi, hi],
                                     fmap, norm)
            dq[bi, hi], dk[bi, hi], dv[bi, hi] = g[0], g[1], g[2]
            if dmc.ndim == 3:
                dmc[hi] += g[3]
            else:
                dmc += g[3]
    return dq, dk, dv, dmc


__all__ = ["feature_map_grad", "mhla_head_backward64", "mhla_bruteforce_backward64", "mhla_backward64"]
