// Backward pass of the block-ordered causal MHLA on the CUDA cores (float32
// arithmetic, every head dimension, bf16 or float32 tensors).
//
// The causal form ("MHLA: Restoring Expressivity of Linear Attention via
// Token-Level Multi-Head", key design 2 with its chunkwise, streaming
// remarks; the pages define no causal variant, this is the block-ordered
// reading of the forward kernels): query t of block i, w = Mc[i, i],
//     S~_t = Sp_i + w R_t,  Sp_i = sum_{b<i} Mc[i,b] S_b,
//     R_t = sum_{j in i, j <= t} phi(k_j) v_j^T          (z, v, n likewise)
// and o_t the norm of phi(q_t)^T S~_t and s_t = phi(q_t) . z~_t.  Its
// gradients are the chain rule of these steps:
//   per token: dnum_t, ds_t (MALA: dv~_t = -gamma_t dO_t, dn~_t) from the
//              norm as in the non-causal backward; dphi(q_t) = S~_t dnum_t +
//              z~_t ds_t; the state gradient dS~_t = phi(q_t) dnum_t^T,
//              dz~_t = ds_t phi(q_t)
//   prefix:    dSp_i = sum_t dS~_t (z, v, n likewise), which the non-causal
//              mixing, Mc and summary steps take from here with Mc's strict
//              lower triangle
//   in block:  dphi(k_j) += w (GS_j v_j + Gz_j), dv_j += w (GS_j^T phi(k_j)
//              + Gv_j) with the suffix sums GS_j = sum_{t >= j} dS~_t (Gz,
//              Gv likewise);
//              dMc[i,i] = sum_t <dS~_t, R_t> + <dz~_t, rz_t> + <dv~_t, rv_t>
//              + dn~_t rn_t.
// Two kernels, one CTA per (block, head) each:
//   causal_bwd_fwd  walks the block forwards in tiles (the running in-block
//                   state R and the masked in-tile scores, as the forward
//                   kernel does): dq, the block's dSp (into the piece-0 row
//                   of the partials), dn~, the diagonal term of dMc and, per
//                   token, dnum_t, ds_t, gamma_t for the second kernel
//   causal_bwd_rev  walks it backwards with the suffix sums GS, Gz, Gv: the
//                   in-block parts of dphi(k) and dv (before phi'), which the
//                   summary step adds to its own
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "backward.h"
#include "common.cuh"

namespace mhla {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

template <int D>
struct TileTokens {
  static constexpr int value = D <= 64 ? 32 : 16;
};

// Rows of the D-wide shared arrays are D + 1 floats apart, so that a warp
// reading one column of D consecutive rows hits 32 different banks.
template <int D>
constexpr size_t fwd_smem_floats() {
  constexpr int TQ = TileTokens<D>::value, LD = D + 1;
  return 2 * D * LD + 4 * D + 5 * TQ * LD + TQ * TQ + 2 * TQ + 2 * kWarps;
}

template <int D>
constexpr size_t rev_smem_floats() {
  constexpr int TQ = TileTokens<D>::value, LD = D + 1;
  return D * LD + 2 * D + 5 * TQ * LD + 2 * TQ * TQ + TQ;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

__device__ __forceinline__ float phi_grad(float x, int fmap) { return phi_deriv(x, phi_apply(x, fmap), fmap); }

// Shared memory: Sp_i (D*D), R (D*D), zp, vp, rz, rv (D each) | tiles of
// phi(q), phi(k), v, dO, dnum (TQ*D each) | in-tile scores, later the
// in-tile dq weights (TQ*TQ) | ds, gamma (TQ) | per-warp sums of the
// diagonal term and of dn~.
template <int D, typename T>
__global__ void __launch_bounds__(kThreads)
causal_bwd_fwd_kernel(Plan p, const T* __restrict__ Q, const T* __restrict__ K, const T* __restrict__ V,
                      const T* __restrict__ dO, const float* __restrict__ mixed,
                      const float* __restrict__ rowsum_lower, const float* __restrict__ mc, T* __restrict__ dQ,
                      float* __restrict__ dmixp, float* __restrict__ dnp, float* __restrict__ diag,
                      float* __restrict__ tokbuf) {
  constexpr int TQ = TileTokens<D>::value, LD = D + 1;
  constexpr int PER = (D * D + kThreads - 1) / kThreads;
  extern __shared__ float sm[];
  float* sP = sm;               // Sp_i
  float* sR = sP + D * LD;      // in-block state R (without w)
  float* zP = sR + D * LD;
  float* vP = zP + D;
  float* zR = vP + D;
  float* vR = zR + D;
  float* sq = vR + D;           // phi(q)
  float* sk = sq + TQ * LD;     // phi(k)
  float* sx = sk + TQ * LD;     // v
  float* sg = sx + TQ * LD;     // dO
  float* sdn = sg + TQ * LD;    // dnum
  float* sa = sdn + TQ * LD;    // TQ*TQ
  float* sds = sa + TQ * TQ;    // ds
  float* sgm = sds + TQ;        // gamma
  float* sdg = sgm + TQ;        // per-warp sums: diagonal term [kWarps], dn~ [kWarps]
  const int u = blockIdx.y, i = blockIdx.x;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int jm = mc_index(p, u);
  const float w = mc[((size_t)jm * p.M + i) * p.M + i];
  const float* mrow = mixed + ((size_t)u * p.M + i) * p.R;
  for (int e = tid; e < D * D; e += kThreads) {
    sP[e / D * LD + e % D] = mrow[e];
    sR[e / D * LD + e % D] = 0.f;
  }
  for (int e = tid; e < D; e += kThreads) {
    zP[e] = mrow[D * D + e];
    vP[e] = mrow[D * D + D + e];
    zR[e] = 0.f;
    vR[e] = 0.f;
  }
  const float n_pre = (float)p.nb * rowsum_lower[jm * p.M + i];
  const bool mala = p.norm == MHLA_NORM_MALA;

  float acc[PER];
#pragma unroll
  for (int m = 0; m < PER; ++m) acc[m] = 0.f;
  float zacc = 0.f, vacc = 0.f, nacc = 0.f, dacc = 0.f;
  float rn = 0.f;  // tokens of the block before the tile

  for (int l0 = 0; l0 < p.nb; l0 += TQ) {
    const int cnt = min(TQ, p.nb - l0);
    __syncthreads();
    for (int e = tid; e < TQ * D; e += kThreads) {
      const int tt = e / D, f = e % D;
      float qx = 0.f, kx = 0.f, vx = 0.f, gx = 0.f;
      if (tt < cnt) {
        const size_t off = tok_off(p, u, block_token(p, i, l0 + tt)) + f;
        qx = phi_apply(to_f32(Q[off]), p.fmap);
        kx = phi_apply(to_f32(K[off]), p.fmap);
        vx = to_f32(V[off]);
        gx = to_f32(dO[off]);
      }
      sq[tt * LD + f] = qx;
      sk[tt * LD + f] = kx;
      sx[tt * LD + f] = vx;
      sg[tt * LD + f] = gx;
    }
    __syncthreads();
    // masked in-tile scores a[t][j] = phi(q_t) . phi(k_j), j <= t
    for (int e = tid; e < TQ * TQ; e += kThreads) {
      const int tt = e / TQ, jj = e % TQ;
      float a = 0.f;
      if (jj <= tt && tt < cnt)
        for (int f = 0; f < D; ++f) a = fmaf(sq[tt * LD + f], sk[jj * LD + f], a);
      sa[e] = a;
    }
    __syncthreads();
    // one warp per query: its state, norm gradients and diagonal term
    for (int tt = warp; tt < cnt; tt += kWarps) {
      float sp = 0.f, sin = 0.f;
      for (int f = lane; f < D; f += 32) {
        sp = fmaf(sq[tt * LD + f], zP[f], sp);
        sin = fmaf(sq[tt * LD + f], zR[f], sin);
      }
      for (int jj = lane; jj <= tt; jj += 32) sin += sa[tt * TQ + jj];
      sp = warp_sum(sp);
      sin = warp_sum(sin);                      // phi(q_t) . rz_t
      const float s = fmaf(w, sin, sp);
      const float rnt = rn + (float)(tt + 1);   // rn_t
      const float nt = fmaf(w, rnt, n_pre);
      const bool live = p.norm == MHLA_NORM_NONE || s != 0.f;
      const float coef =
          !live ? 0.f : (p.norm == MHLA_NORM_DIVISIVE ? 1.f / s : (mala ? 1.f + 1.f / s : 1.f));  // dnum / dO
      float gnum = 0.f, gvt = 0.f, gain = 0.f, gvin = 0.f;
      for (int c = lane; c < D; c += 32) {
        float ap = 0.f, ar = 0.f, loc = 0.f, vloc = 0.f;
        for (int f = 0; f < D; ++f) {
          const float x = sq[tt * LD + f];
          ap = fmaf(x, sP[f * LD + c], ap);
          ar = fmaf(x, sR[f * LD + c], ar);
        }
        for (int jj = 0; jj <= tt; ++jj) {
          loc = fmaf(sa[tt * TQ + jj], sx[jj * LD + c], loc);
          vloc += sx[jj * LD + c];
        }
        const float ain = ar + loc;                 // phi(q_t)^T R_t, column c
        const float num = fmaf(w, ain, ap);
        const float vin = vR[c] + vloc;             // rv_t
        const float vt = fmaf(w, vin, vP[c]);
        const float g = sg[tt * LD + c];
        gnum = fmaf(g, num, gnum);
        gvt = fmaf(g, vt, gvt);
        gain = fmaf(g, ain, gain);
        gvin = fmaf(g, vin, gvin);
        sdn[tt * LD + c] = coef * g;
      }
      gnum = warp_sum(gnum);
      gvt = warp_sum(gvt);
      gain = warp_sum(gain);
      gvin = warp_sum(gvin);
      float ds = 0.f, gamma = 0.f, dnt = 0.f;
      if (live && p.norm == MHLA_NORM_DIVISIVE) {
        ds = -gnum / (s * s);
      } else if (live && mala) {
        const float dgamma = -gvt;
        ds = -gnum / (s * s) + dgamma / nt;
        gamma = s / nt;
        dnt = -dgamma * s / (nt * nt);
      }
      if (lane == 0) {
        sds[tt] = ds;
        sgm[tt] = gamma;
        // <dS~_t, R_t> + ds_t (phi(q_t) . rz_t) + <dv~_t, rv_t> + dn~_t rn_t
        dacc += coef * gain + ds * sin - gamma * gvin + dnt * rnt;
        nacc += dnt;
      }
    }
    __syncthreads();
    // in-tile dq weights E[t][j] = v_j . dnum_t + ds_t, j <= t
    for (int e = tid; e < TQ * TQ; e += kThreads) {
      const int tt = e / TQ, jj = e % TQ;
      float a = 0.f;
      if (jj <= tt && tt < cnt) {
        a = sds[tt];
        for (int c = 0; c < D; ++c) a = fmaf(sx[jj * LD + c], sdn[tt * LD + c], a);
      }
      sa[e] = a;
    }
    __syncthreads();
    // dq_t = ((Sp + w R) dnum_t + (zp + w rz) ds_t + w sum_{j<=t} E[t][j] phi(k_j)) phi'(q_t)
    for (int e = tid; e < cnt * D; e += kThreads) {
      const int tt = e / D, k = e % D;
      float a = 0.f;
      for (int c = 0; c < D; ++c) a = fmaf(fmaf(w, sR[k * LD + c], sP[k * LD + c]), sdn[tt * LD + c], a);
      a = fmaf(fmaf(w, zR[k], zP[k]), sds[tt], a);
      float loc = 0.f;
      for (int jj = 0; jj <= tt; ++jj) loc = fmaf(sa[tt * TQ + jj], sk[jj * LD + k], loc);
      a = fmaf(w, loc, a);
      const size_t off = tok_off(p, u, block_token(p, i, l0 + tt)) + k;
      dQ[off] = from_f32<T>(a * phi_grad(to_f32(Q[off]), p.fmap));
    }
    // dSp += phi(q_t) dnum_t^T, dzp += ds_t phi(q_t), dvp += -gamma_t dO_t
    for (int tt = 0; tt < cnt; ++tt) {
#pragma unroll
      for (int m = 0; m < PER; ++m) {
        const int e = tid + m * kThreads;
        if (e < D * D) acc[m] = fmaf(sq[tt * LD + e / D], sdn[tt * LD + e % D], acc[m]);
      }
      if (tid < D) zacc = fmaf(sds[tt], sq[tt * LD + tid], zacc);
      else if (tid < 2 * D && mala) vacc = fmaf(-sgm[tt], sg[tt * LD + tid - D], vacc);
    }
    // per token for the reverse walk: dnum (D), ds, gamma
    for (int e = tid; e < cnt * (D + 2); e += kThreads) {
      const int tt = e / (D + 2), c = e % (D + 2);
      const float x = c < D ? sdn[tt * LD + c] : (c == D ? sds[tt] : sgm[tt]);
      tokbuf[((size_t)u * p.N + block_token(p, i, l0 + tt)) * (D + 2) + c] = x;
    }
    __syncthreads();
    // advance the in-block state by the whole tile
    for (int e = tid; e < D * D; e += kThreads) {
      const int f = e / D, c = e % D;
      float a = 0.f;
      for (int jj = 0; jj < cnt; ++jj) a = fmaf(sk[jj * LD + f], sx[jj * LD + c], a);
      sR[f * LD + c] += a;
    }
    if (tid < D) {
      float a = 0.f;
      for (int jj = 0; jj < cnt; ++jj) a += sk[jj * LD + tid];
      zR[tid] += a;
    } else if (tid < 2 * D) {
      float a = 0.f;
      for (int jj = 0; jj < cnt; ++jj) a += sx[jj * LD + tid - D];
      vR[tid - D] += a;
    }
    rn += (float)cnt;
  }
  // the block's prefix gradient goes to its first piece row; the other
  // pieces of the block carry nothing
  const size_t row0 = (size_t)u * p.M * p.splits + (size_t)i * p.splits;
  for (int sp = 1; sp < p.splits; ++sp) {
    float* o = dmixp + (row0 + sp) * p.R;
    for (int e = tid; e < p.R; e += kThreads) o[e] = 0.f;
    if (tid == 0) dnp[row0 + sp] = 0.f;
  }
  float* out = dmixp + row0 * p.R;
#pragma unroll
  for (int m = 0; m < PER; ++m) {
    const int e = tid + m * kThreads;
    if (e < D * D) out[e] = acc[m];
  }
  if (tid < D) out[D * D + tid] = zacc;
  else if (tid < 2 * D) out[D * D + tid] = vacc;
  if (lane == 0) {
    sdg[warp] = dacc;
    sdg[kWarps + warp] = nacc;
  }
  __syncthreads();
  if (tid == 0) {
    float t = 0.f, n = 0.f;
    for (int x = 0; x < kWarps; ++x) {
      t += sdg[x];
      n += sdg[kWarps + x];
    }
    diag[(size_t)u * p.M + i] = t;
    dnp[row0] = n;
  }
}

// Shared memory: GS (D*D), Gz, Gv (D) | tiles of phi(q), phi(k), v, dnum,
// dv~ (TQ*D each) | E[j][t] = dnum_t . v_j + ds_t and P[j][t] = phi(q_t) .
// phi(k_j), t >= j (TQ*TQ each) | ds (TQ).
template <int D, typename T>
__global__ void __launch_bounds__(kThreads)
causal_bwd_rev_kernel(Plan p, const T* __restrict__ Q, const T* __restrict__ K, const T* __restrict__ V,
                      const T* __restrict__ dO, const float* __restrict__ mc, const float* __restrict__ tokbuf,
                      float* __restrict__ xk, float* __restrict__ xv) {
  constexpr int TQ = TileTokens<D>::value, LD = D + 1;
  constexpr int PER = (D * D + kThreads - 1) / kThreads;
  extern __shared__ float sm[];
  float* GS = sm;
  float* Gz = GS + D * LD;
  float* Gv = Gz + D;
  float* sq = Gv + D;
  float* sk = sq + TQ * LD;
  float* sx = sk + TQ * LD;
  float* sdn = sx + TQ * LD;
  float* sgv = sdn + TQ * LD;
  float* sE = sgv + TQ * LD;
  float* sPm = sE + TQ * TQ;
  float* sds = sPm + TQ * TQ;
  const int u = blockIdx.y, i = blockIdx.x, tid = threadIdx.x;
  const int jm = mc_index(p, u);
  const float w = mc[((size_t)jm * p.M + i) * p.M + i];
  const bool mala = p.norm == MHLA_NORM_MALA;
  for (int e = tid; e < D * LD + 2 * D; e += kThreads) sm[e] = 0.f;
  float acc[PER];
#pragma unroll
  for (int m = 0; m < PER; ++m) acc[m] = 0.f;

  for (int l0 = (p.nb - 1) / TQ * TQ; l0 >= 0; l0 -= TQ) {
    const int cnt = min(TQ, p.nb - l0);
    __syncthreads();
    for (int e = tid; e < TQ * D; e += kThreads) {
      const int tt = e / D, f = e % D;
      float qx = 0.f, kx = 0.f, vx = 0.f, dn = 0.f, gv = 0.f;
      if (tt < cnt) {
        const int tok = block_token(p, i, l0 + tt);
        const size_t off = tok_off(p, u, tok) + f;
        const float* tb = tokbuf + ((size_t)u * p.N + tok) * (D + 2);
        qx = phi_apply(to_f32(Q[off]), p.fmap);
        kx = phi_apply(to_f32(K[off]), p.fmap);
        vx = to_f32(V[off]);
        dn = tb[f];
        if (mala) gv = -tb[D + 1] * to_f32(dO[off]);
        if (f == 0) sds[tt] = tb[D];
      } else if (f == 0) {
        sds[tt] = 0.f;
      }
      sq[tt * LD + f] = qx;
      sk[tt * LD + f] = kx;
      sx[tt * LD + f] = vx;
      sdn[tt * LD + f] = dn;
      sgv[tt * LD + f] = gv;
    }
    __syncthreads();
    for (int e = tid; e < TQ * TQ; e += kThreads) {
      const int jj = e / TQ, tt = e % TQ;
      float a = 0.f, b = 0.f;
      if (tt >= jj && tt < cnt) {
        a = sds[tt];
        for (int f = 0; f < D; ++f) {
          a = fmaf(sdn[tt * LD + f], sx[jj * LD + f], a);
          b = fmaf(sq[tt * LD + f], sk[jj * LD + f], b);
        }
      }
      sE[e] = a;
      sPm[e] = b;
    }
    __syncthreads();
    // in-block parts for token j: w (GS v_j + Gz + sum_{t>=j} E[j][t] phi(q_t)) and
    // w (GS^T phi(k_j) + Gv + sum_{t>=j} (P[j][t] dnum_t + dv~_t))
    for (int e = tid; e < cnt * D; e += kThreads) {
      const int jj = e / D, f = e % D;
      float gk = Gz[f], gv = Gv[f];
      for (int c = 0; c < D; ++c) {
        gk = fmaf(GS[f * LD + c], sx[jj * LD + c], gk);
        gv = fmaf(GS[c * LD + f], sk[jj * LD + c], gv);
      }
      for (int tt = jj; tt < cnt; ++tt) {
        gk = fmaf(sE[jj * TQ + tt], sq[tt * LD + f], gk);
        gv = fmaf(sPm[jj * TQ + tt], sdn[tt * LD + f], gv) + sgv[tt * LD + f];
      }
      const size_t off = tok_off(p, u, block_token(p, i, l0 + jj)) + f;
      xk[off] = w * gk;
      xv[off] = w * gv;
    }
    __syncthreads();
    // the tile joins the suffix sums
#pragma unroll
    for (int m = 0; m < PER; ++m) {
      const int e = tid + m * kThreads;
      if (e < D * D) {
        float a = 0.f;
        for (int tt = 0; tt < cnt; ++tt) a = fmaf(sq[tt * LD + e / D], sdn[tt * LD + e % D], a);
        acc[m] = a;
      }
    }
    if (tid < D) {
      float a = 0.f;
      for (int tt = 0; tt < cnt; ++tt) a = fmaf(sds[tt], sq[tt * LD + tid], a);
      Gz[tid] += a;
    } else if (tid < 2 * D) {
      float a = 0.f;
      for (int tt = 0; tt < cnt; ++tt) a += sgv[tt * LD + tid - D];
      Gv[tid - D] += a;
    }
#pragma unroll
    for (int m = 0; m < PER; ++m) {
      const int e = tid + m * kThreads;
      if (e < D * D) GS[e / D * LD + e % D] += acc[m];
    }
  }
}

template <int D, typename T>
int run(const Plan& p, const CausalBwdBuffers& c, const void* q, const void* k, const void* v, const void* dout,
        void* dq, cudaStream_t s) {
  const size_t smf = sizeof(float) * fwd_smem_floats<D>();
  const size_t smr = sizeof(float) * rev_smem_floats<D>();
  auto kf = causal_bwd_fwd_kernel<D, T>;
  auto kr = causal_bwd_rev_kernel<D, T>;
  cudaError_t e = (cudaError_t)set_max_dynamic_smem((const void*)kf, (int)smf);
  if (e != cudaSuccess) return (int)e;
  if ((e = (cudaError_t)set_max_dynamic_smem((const void*)kr, (int)smr)) != cudaSuccess) return (int)e;
  kf<<<dim3(p.M, p.BH), kThreads, smf, s>>>(p, (const T*)q, (const T*)k, (const T*)v, (const T*)dout, c.mixed,
                                             c.rowsum_lower, c.mc, (T*)dq, c.dmixp, c.dnp, c.diag, c.tokbuf);
  if ((e = cudaGetLastError()) != cudaSuccess) return (int)e;
  kr<<<dim3(p.M, p.BH), kThreads, smr, s>>>(p, (const T*)q, (const T*)k, (const T*)v, (const T*)dout, c.mc,
                                             c.tokbuf, c.xk, c.xv);
  return (int)cudaGetLastError();
}

template <typename T>
int by_d(const Plan& p, const CausalBwdBuffers& c, const void* q, const void* k, const void* v, const void* dout,
         void* dq, cudaStream_t s) {
  switch (p.d) {
    case 16: return run<16, T>(p, c, q, k, v, dout, dq, s);
    case 32: return run<32, T>(p, c, q, k, v, dout, dq, s);
    case 64: return run<64, T>(p, c, q, k, v, dout, dq, s);
    case 128: return run<128, T>(p, c, q, k, v, dout, dq, s);
  }
  return (int)cudaErrorInvalidValue;
}

}  // namespace

int launch_bwd_causal_block(const Plan& p, const CausalBwdBuffers& c, const void* q, const void* k, const void* v,
                            const void* dout, void* dq, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (p.dtype == MHLA_DTYPE_F32) return by_d<float>(p, c, q, k, v, dout, dq, s);
  return by_d<__nv_bfloat16>(p, c, q, k, v, dout, dq, s);
}

}  // namespace mhla
