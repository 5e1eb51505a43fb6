"""Float64 CPU oracle for the gradients of the causal (block-ordered) MHLA forward.

TEST INFRASTRUCTURE ONLY, like ``mhla_oracle``: only ``tests/`` use it; it
shares no code with the CUDA library and imports nothing but numpy and the
other oracle modules.

What it differentiates is ``mhla_causal_oracle``: the causal reading of
"MHLA: Restoring Expressivity of Linear Attention via Token-Level
Multi-Head" (key design 2's chunkwise, streaming remarks; the summaries are
additive), with the MALA norm of "Rectifying Magnitude Neglect in Linear
Attention" (key designs).  The pages print no gradient; these are the chain
rule of the causal forward steps (query t in block i, w = Mc[i, i]):

  forward:   Sp_i = sum_{b<i} Mc[i,b] S_b  (zp, vp, np likewise)
             R_t  = sum_{j in i, j <= t} phk_j v_j^T  (rz_t, rv_t, rn_t likewise)
             S~_t = Sp_i + w R_t,  z~_t = zp_i + w rz_t,  v~_t, n~_t likewise
             o_t  = the norm of phq_t^T S~_t and s_t = phq_t . z~_t

  backward, given dO:
    per token: dnum_t, ds_t (and MALA dv~_t, dn~_t) from the norm, exactly as
               in the non-causal backward; dphq_t = S~_t dnum_t + z~_t ds_t;
               the state gradient dS~_t = phq_t dnum_t^T, dz~_t = ds_t phq_t
    prefix:    dSp_i = sum_{t in i} dS~_t (z, v, n likewise);
               dS_b = sum_{i>b} Mc[i,b] dSp_i;
               dMc[i,b] (b < i) = <dSp_i, S_b> + <dzp_i, z_b> + <dvp_i, v_b> + dnp_i n_b
    in block:  token j of block i feeds every S~_t with t >= j, so with the
               suffix sums GS_j = sum_{t>=j} dS~_t (Gz_j, Gv_j likewise)
               dphk_j += w (GS_j v_j + Gz_j),  dv_j += w (GS_j^T phk_j + Gv_j);
               dMc[i,i] = sum_t <dS~_t, R_t> + <dz~_t, rz_t> + <dv~_t, rv_t> + dn~_t rn_t
    summaries: dphk_j += dS_b v_j + dz_b,  dv_j += dS_b^T phk_j + dv_b
    map:       dq = dphq * phi'(q),  dk = dphk * phi'(k)
  Mc above the diagonal does not enter the causal output: its gradient is 0.
  A query whose denominator s is exactly zero has output 0 and contributes
  nothing (the forward oracle's rule).

``mhla_causal_head_backward64`` follows the prefix recursion token by token;
``mhla_causal_bruteforce_backward64`` differentiates the masked explicit
N x N form instead.
"""

from __future__ import annotations

import numpy as np

from .mhla_backward_oracle import feature_map_grad
from .mhla_causal_oracle import causal_mask
from .mhla_oracle import DIVISIVE, ELU1, MALA, NONE, block_of_token, block_summaries, feature_map, head_mc, mix


def _token_grads(pq, g, St, zt, vt, nt, norm):
    """dnum, ds, dv~, dn~ of one query from its state and dO (g)."""
    num = pq @ St
    zero = np.zeros_like(vt)
    if norm == NONE:
        return g, 0.0, zero, 0.0
    s = float(pq @ zt)
    if s == 0.0:
        return np.zeros_like(num), 0.0, zero, 0.0
    inv = 1.0 / s
    if norm == DIVISIVE:
        o = num * inv
        return g * inv, -float(g @ o) * inv, zero, 0.0
    if norm == MALA:
        beta = 1.0 + inv
        gamma = s / nt
        dbeta = float(g @ num)
        dgamma = -float(g @ vt)
        ds = -dbeta * inv * inv + dgamma / nt
        return beta * g, ds, -gamma * g, -dgamma * s / (nt * nt)
    raise ValueError(f"unknown norm {norm!r}")


def mhla_causal_head_backward64(q, k, v, mc, grid, block, dout, fmap: str = ELU1, norm: str = DIVISIVE):
    """Gradients of one head's causal forward by the prefix recursion: (dq, dk, dv, dmc)."""
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
    lower = np.tril(mc, -1)
    Sp, zp, vp, npre = mix(lower, S, z, vs, n)

    dphq = np.zeros_like(phq)
    dphk = np.zeros_like(phk)
    dv = np.zeros_like(v)
    dSp = np.zeros_like(Sp)
    dzp = np.zeros_like(zp)
    dvp = np.zeros_like(vp)
    dnp = np.zeros_like(npre)
    dmc = np.zeros((M, M))
    for i in range(M):
        w = mc[i, i]
        toks = np.nonzero(bidx == i)[0]
        R = np.zeros_like(S[0])
        rz = np.zeros_like(z[0])
        rv = np.zeros_like(vs[0])
        rn = 0.0
        per_token = []
        for t in toks:
            R += np.outer(phk[t], v[t])
            rz += phk[t]
            rv += v[t]
            rn += 1.0
            St, zt, vt, nt = Sp[i] + w * R, zp[i] + w * rz, vp[i] + w * rv, npre[i] + w * rn
            dnum, ds, dvt, dnt = _token_grads(phq[t], dout[t], St, zt, vt, nt, norm)
            dphq[t] = St @ dnum + ds * zt
            dSt = np.outer(phq[t], dnum)
            dzt = ds * phq[t]
            dSp[i] += dSt
            dzp[i] += dzt
            dvp[i] += dvt
            dnp[i] += dnt
            dmc[i, i] += np.sum(dSt * R) + dzt @ rz + dvt @ rv + dnt * rn
            per_token.append((dSt, dzt, dvt))
        # in-block terms: suffix sums over the queries at or after each token
        GS = np.zeros_like(S[0])
        Gz = np.zeros_like(z[0])
        Gv = np.zeros_like(vs[0])
        for pos in range(len(toks) - 1, -1, -1):
            j = toks[pos]
            dSt, dzt, dvt = per_token[pos]
            GS += dSt
            Gz += dzt
            Gv += dvt
            dphk[j] += w * (GS @ v[j] + Gz)
            dv[j] += w * (GS.T @ phk[j] + Gv)

    # earlier blocks, through the strict lower triangle of Mc
    dS = (lower.T @ dSp.reshape(M, -1)).reshape(S.shape)
    dz = lower.T @ dzp
    dvs = lower.T @ dvp
    strict = np.tril(np.ones((M, M)), -1)
    dmc += strict * (dSp.reshape(M, -1) @ S.reshape(M, -1).T + dzp @ z.T + dvp @ vs.T + np.outer(dnp, n))
    for b in range(M):
        sel = bidx == b
        dphk[sel] += v[sel] @ dS[b].T + dz[b][None, :]
        dv[sel] += phk[sel] @ dS[b] + dvs[b][None, :]
    return dphq * feature_map_grad(q, fmap), dphk * feature_map_grad(k, fmap), dv, dmc


def mhla_causal_bruteforce_backward64(q, k, v, mc, grid, block, dout, fmap: str = ELU1, norm: str = DIVISIVE):
    """Gradients of the masked explicit form (see mhla_causal_bruteforce64): (dq, dk, dv, dmc).

    A = W * (phq phk^T) with W = C * Mc[b(t), b(j)] and C the causal mask;
    DIVISIVE P = A / rowsum(A); NONE P = A; MALA P = beta A - gamma W with
    s = rowsum(A), beta = 1 + 1/s, gamma = s / rowsum(W); o = P V.
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
    C = causal_mask(grid, block)
    W = C * mc[bidx][:, bidx]
    G = phq @ phk.T
    A = W * G
    if norm == NONE:
        dvv = A.T @ dout
        dA = dout @ v.T
        dW = np.zeros_like(W)
    elif norm == DIVISIVE:
        s = A.sum(axis=1)
        live = s != 0.0
        inv = np.divide(1.0, s, out=np.zeros_like(s), where=live)
        P = A * inv[:, None]
        o = P @ v
        dvv = P.T @ dout
        dA = (dout @ v.T - np.sum(dout * o, axis=1)[:, None]) * inv[:, None]
        dW = np.zeros_like(W)
    elif norm == MALA:
        s = A.sum(axis=1)
        live = s != 0.0
        inv = np.divide(1.0, s, out=np.zeros_like(s), where=live)
        wsum = W.sum(axis=1)
        beta = 1.0 + inv
        gamma = s / wsum
        P = np.where(live[:, None], beta[:, None] * A - gamma[:, None] * W, 0.0)
        dvv = P.T @ dout
        dP = np.where(live[:, None], dout @ v.T, 0.0)
        dbeta = np.sum(dP * A, axis=1)
        dgamma = -np.sum(dP * W, axis=1)
        ds = -dbeta * inv ** 2 + dgamma / wsum
        dw = -dgamma * s / wsum ** 2
        dA = beta[:, None] * dP + ds[:, None]
        dW = -gamma[:, None] * dP + dw[:, None]
    else:
        raise ValueError(f"unknown norm {norm!r}")
    dW = dW + dA * G
    dG = dA * W
    dphq = dG @ phk
    dphk = dG.T @ phq
    dmc = np.zeros((M, M))
    # W[t, j] = C[t, j] Mc[b(t), b(j)]: only unmasked pairs reach Mc
    np.add.at(dmc, (bidx[:, None], bidx[None, :]), C * dW)
    return dphq * feature_map_grad(q, fmap), dphk * feature_map_grad(k, fmap), dvv, dmc


def mhla_causal_backward64(q, k, v, mc, grid, block, dout, fmap: str = ELU1, norm: str = DIVISIVE):
    """Causal gradients over [B, H, N, d] inputs: dq, dk, dv [B, H, N, d] and
    dmc shaped like mc (summed over every (batch, head) for one shared Mc, over
    the batch for one Mc per head)."""
    q = np.asarray(q)
    if q.ndim == 2:
        return mhla_causal_head_backward64(q, k, v, mc, grid, block, dout, fmap, norm)
    k, v, dout = np.asarray(k), np.asarray(v), np.asarray(dout)
    dq = np.zeros(q.shape)
    dk = np.zeros(q.shape)
    dv = np.zeros(v.shape)
    dmc = np.zeros(np.asarray(mc).shape)
    for bi in range(q.shape[0]):
        for hi in range(q.shape[1]):
            g = mhla_causal_head_backward64(q[bi, hi], k[bi, hi], v[bi, hi], head_mc(mc, hi), grid, block,
                                            dout[bi, hi], fmap, norm)
            dq[bi, hi], dk[bi, hi], dv[bi, hi] = g[0], g[1], g[2]
            if dmc.ndim == 3:
                dmc[hi] += g[3]
            else:
                dmc += g[3]
    return dq, dk, dv, dmc


__all__ = ["mhla_causal_head_backward64", "mhla_causal_bruteforce_backward64", "mhla_causal_backward64"]
