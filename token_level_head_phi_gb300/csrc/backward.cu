// Backward pass of the MHLA forward on the CUDA cores (float32 arithmetic,
// every head dimension, bf16 or float32 tensors): the gradients of
// sum(dO * o) with respect to Q, K, V and Mc.  The pages say Mc is learned
// end to end ("MHLA: Restoring Expressivity of Linear Attention via
// Token-Level Multi-Head", key design 3) but print no gradient; these are the
// chain rule of the forward steps taken in reverse (token t in query block
// i = b(t), token j in summary block b):
//
//   output:   dnum_t, ds_t from the norm (DIVISIVE dnum = dO/s,
//             ds = -(dO.o)/s; NONE dnum = dO; MALA below)
//             dphi(q_t) = S~_i dnum_t + z~_i ds_t
//             dS~_i = sum_t phi(q_t) dnum_t^T,  dz~_i = sum_t ds_t phi(q_t)
//   mixing:   dS_b = sum_i Mc[i,b] dS~_i (z, v likewise)
//             dMc[i,b] = sum over heads of <dS~_i, S_b> + <dz~_i, z_b>
//                        (+ <dv~_i, v_b> + dn~_i n_b for MALA)
//   summary:  dphi(k_j) = dS_b v_j + dz_b,  dv_j = dS_b^T phi(k_j) (+ dv_b)
//   map:      dq = dphi(q) * phi'(q),  dk = dphi(k) * phi'(k)
// MALA ("Rectifying Magnitude Neglect in Linear Attention", key designs,
// with the mixed sums): o = beta num - gamma v~_i, beta = 1 + 1/s,
// gamma = s / n~_i, so dnum = beta dO, ds = -(dO.num)/s^2 - (dO.v~_i)/n~_i,
// dv~_i = -sum_t gamma_t dO_t, dn~_i = sum_t (dO_t.v~_i) s_t / n~_i^2.
//
// Kernels, in launch order after the forward summaries and mixing are
// recomputed by the float32 forward kernels:
//   bwd_output   one CTA per (query block piece, head): dq and the piece's
//                partial dS~, dz~, dv~ (and dn~), kept per piece so the
//                accumulation order is fixed (no atomics)
//   bwd_mix      dS_b = sum over query pieces of Mc[i(piece), b] * partials
//   bwd_mc       dMc = sum over heads of partials-per-block . summaries-per-block
//   bwd_summary  one CTA per (summary block piece, head): dk, dv
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "backward.h"
#include "common.cuh"

namespace mhla {
namespace {

constexpr int kThreads = 256;
constexpr int kTile = 32;  // tokens per shared-memory tile
constexpr int kMcTile = 64;  // dMc entries per CTA side

__device__ __forceinline__ float phi_grad(float x, int fmap) { return phi_deriv(x, phi_apply(x, fmap), fmap); }

// One CTA per (query block piece, head).  Shared memory: S~_i [D][D], z~_i,
// v~_i, and per tile phi(q) [T][D], dO [T][D], dnum [T][D] and per-token
// scalars.  Thread e owns entries e, e + 256, ... of the partial dS~.
template <int D, typename T>
__global__ void __launch_bounds__(kThreads)
bwd_output_kernel(Plan p, const T* __restrict__ Q, const T* __restrict__ dO, const float* __restrict__ mixed,
                  const float* __restrict__ rowsum, T* __restrict__ dQ, float* __restrict__ dmixp,
                  float* __restrict__ dnp) {
  constexpr int PER = (D * D + kThreads - 1) / kThreads;
  constexpr int LD = D + 1;        // row stride: a column of consecutive rows spans 32 banks
  extern __shared__ float sm[];
  float* sS = sm;                  // D rows
  float* sz = sS + D * LD;         // D
  float* sv = sz + D;              // D
  float* sq = sv + D;              // kTile rows: phi(q)
  float* sg = sq + kTile * LD;     // kTile rows: dO
  float* sdn = sg + kTile * LD;    // kTile rows: dnum
  float* sds = sdn + kTile * LD;   // kTile: ds
  float* ssc = sds + kTile;        // kTile: s
  float* sgam = ssc + kTile;       // kTile: gamma (MALA)
  float* sdgam = sgam + kTile;     // kTile: dO . v~ (MALA)
  const int u = blockIdx.y;
  const int row = blockIdx.x;      // query piece: block i, piece row % splits
  const int i = row / p.splits;
  const int l0 = (row % p.splits) * p.split_len;
  const int l1 = min(p.nb, l0 + p.split_len);
  const int tid = threadIdx.x;
  const float* mrow = mixed + ((size_t)u * p.M + i) * p.R;
  for (int e = tid; e < D * D; e += kThreads) sS[e / D * LD + e % D] = mrow[e];
  for (int e = tid; e < 2 * D; e += kThreads) sz[e] = mrow[D * D + e];
  const float ntilde = (float)p.nb * rowsum[mc_index(p, u) * p.M + i];

  float acc[PER];
#pragma unroll
  for (int j = 0; j < PER; ++j) acc[j] = 0.f;
  float zacc = 0.f, vacc = 0.f, nacc = 0.f;

  for (int lt = l0; lt < l1; lt += kTile) {
    const int cnt = min(kTile, l1 - lt);
    __syncthreads();
    for (int e = tid; e < kTile * D; e += kThreads) {
      const int tt = e / D, f = e % D;
      float qx = 0.f, gx = 0.f;
      if (tt < cnt) {
        const size_t off = tok_off(p, u, block_token(p, i, lt + tt)) + f;
        qx = phi_apply(to_f32(Q[off]), p.fmap);
        gx = to_f32(dO[off]);
      }
      sq[tt * LD + f] = qx;
      sg[tt * LD + f] = gx;
    }
    __syncthreads();
    // per token: s = phi(q).z~ and the dO.v~ of MALA
    if (tid < kTile) {
      float s = 0.f, gv = 0.f;
      for (int k = 0; k < D; ++k) {
        s = fmaf(sq[tid * LD + k], sz[k], s);
        gv = fmaf(sg[tid * LD + k], sv[k], gv);
      }
      ssc[tid] = s;
      sdgam[tid] = gv;
    }
    __syncthreads();
    // dnum[t][c] and the per-token reduction dO.num for ds
    for (int e = tid; e < kTile * D; e += kThreads) {
      const int tt = e / D, c = e % D;
      float num = 0.f;
      for (int k = 0; k < D; ++k) num = fmaf(sq[tt * LD + k], sS[k * LD + c], num);
      const float g = sg[tt * LD + c];
      const float s = ssc[tt];
      float dn;
      if (p.norm == MHLA_NORM_DIVISIVE) dn = s != 0.f ? g / s : 0.f;   // s = 0: constant output
      else if (p.norm == MHLA_NORM_MALA) dn = s != 0.f ? (1.f + 1.f / s) * g : 0.f;
      else dn = g;
      sdn[tt * LD + c] = dn;
      // g * num replaces g: only the per-token sum dO . num is needed below
      sg[tt * LD + c] = g * num;
    }
    __syncthreads();
    if (tid < kTile) {
      float gnum = 0.f;
      for (int c = 0; c < D; ++c) gnum += sg[tid * LD + c];
      const float s = ssc[tid];
      float ds = 0.f;
      if (p.norm == MHLA_NORM_DIVISIVE) {
        ds = -gnum / (s * s);
      } else if (p.norm == MHLA_NORM_MALA) {
        const float dbeta = gnum, dgamma = -sdgam[tid];
        ds = -dbeta / (s * s) + dgamma / ntilde;
        sgam[tid] = s / ntilde;
      }
      if (tid >= cnt || (p.norm != MHLA_NORM_NONE && s == 0.f)) ds = 0.f;
      sds[tid] = ds;
    }
    __syncthreads();
    // dq[t][k] = (sum_c S~[k][c] dnum[t][c] + z~[k] ds[t]) * phi'(q)
    for (int e = tid; e < cnt * D; e += kThreads) {
      const int tt = e / D, k = e % D;
      float a = sz[k] * sds[tt];
      for (int c = 0; c < D; ++c) a = fmaf(sS[k * LD + c], sdn[tt * LD + c], a);
      const size_t off = tok_off(p, u, block_token(p, i, lt + tt)) + k;
      dQ[off] = from_f32<T>(a * phi_grad(to_f32(Q[off]), p.fmap));
    }
    // partial dS~ += phi(q) dnum^T, dz~ += ds phi(q); MALA: dv~, dn~
    for (int tt = 0; tt < cnt; ++tt) {
#pragma unroll
      for (int j = 0; j < PER; ++j) {
        const int e = tid + j * kThreads;
        if (e < D * D) acc[j] = fmaf(sq[tt * LD + e / D], sdn[tt * LD + e % D], acc[j]);
      }
      if (tid < D) {
        zacc = fmaf(sds[tt], sq[tt * LD + tid], zacc);
      } else if (tid < 2 * D && p.norm == MHLA_NORM_MALA) {
        // dv~ = -sum_t gamma_t dO_t (the tile's dO was overwritten above)
        const size_t off = tok_off(p, u, block_token(p, i, lt + tt)) + (tid - D);
        vacc = fmaf(-sgam[tt], to_f32(dO[off]), vacc);
      }
      if (tid == 0 && p.norm == MHLA_NORM_MALA)
        nacc += sdgam[tt] * ssc[tt] / (ntilde * ntilde);  // dn~ = -dgamma s / n~^2, dgamma = -dO.v~
    }
  }
  float* out = dmixp + ((size_t)u * p.M * p.splits + row) * p.R;
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int e = tid + j * kThreads;
    if (e < D * D) out[e] = acc[j];
  }
  if (tid < D) out[D * D + tid] = zacc;
  else if (tid < 2 * D) out[D * D + tid] = vacc;
  if (tid == 0) dnp[(size_t)u * p.M * p.splits + row] = nacc;
}

// dstack[u][b][r] = sum_q Mc[q / splits][b] * dmixp[u][q][r]: a tiled SGEMM
// with Mc transposed (32 summary blocks x 128 record columns per CTA).
__global__ void __launch_bounds__(kThreads)
bwd_mix_kernel(Plan p, const float* __restrict__ mc, const float* __restrict__ dmixp, float* __restrict__ dstack) {
  constexpr int TB = 32, TR = 128, TQ = 16;
  __shared__ float smc[TB][TQ + 1];
  __shared__ float sst[TQ][TR];
  const int u = blockIdx.z;
  const int b0 = blockIdx.y * TB;
  const int r0 = blockIdx.x * TR;
  const int tx = threadIdx.x % 32, ty = threadIdx.x / 32;
  const int rows = p.M * p.splits;
  const float* st = dmixp + (size_t)u * rows * p.R;
  mc += (size_t)mc_index(p, u) * p.M * p.M;
  float acc[4][4] = {};
  for (int q0 = 0; q0 < rows; q0 += TQ) {
    __syncthreads();
    for (int e = threadIdx.x; e < TB * TQ; e += kThreads) {
      const int bb = e / TQ, qq = e % TQ;
      const int b = b0 + bb, q = q0 + qq;
      smc[bb][qq] = (b < p.M && q < rows) ? mc[(size_t)(q / p.splits) * p.M + b] : 0.f;
    }
    for (int e = threadIdx.x; e < TQ * TR; e += kThreads) {
      const int qq = e / TR, rr = e % TR;
      const int q = q0 + qq, r = r0 + rr;
      sst[qq][rr] = (q < rows && r < p.R) ? st[(size_t)q * p.R + r] : 0.f;
    }
    __syncthreads();
#pragma unroll 4
    for (int qq = 0; qq < TQ; ++qq) {
      float a[4], bv[4];
#pragma unroll
      for (int m = 0; m < 4; ++m) a[m] = smc[ty * 4 + m][qq];
#pragma unroll
      for (int n = 0; n < 4; ++n) bv[n] = sst[qq][tx + 32 * n];
#pragma unroll
      for (int m = 0; m < 4; ++m)
#pragma unroll
        for (int n = 0; n < 4; ++n) acc[m][n] = fmaf(a[m], bv[n], acc[m][n]);
    }
  }
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const int b = b0 + ty * 4 + m;
    if (b >= p.M) continue;
    float* dst = dstack + ((size_t)u * p.M + b) * p.R;
#pragma unroll
    for (int n = 0; n < 4; ++n) {
      const int r = r0 + tx + 32 * n;
      if (r < p.R) dst[r] = acc[m][n];
    }
  }
}

// dMc[i][b] = sum_u sum_r dX~[u][i][r] X[u][b][r] (+ MALA: n_b sum_u dn~[u][i]),
// u over every unit (one shared Mc) or over the units of head blockIdx.z
// (one Mc per head),
// dX~ and X summed over pieces on the fly; one CTA per 16 x 16 tile of dMc,
// reduced over (u, r) in a fixed order.  The sum is blocked in three levels
// (32 record entries, one head, all heads): the terms of a DIVISIVE or MALA
// row cancel to a small fraction of their size, and one running float32
// sum over all d^2 + 2d entries of every head would carry a rounding error
// proportional to that count.
// Causal form (diag set): only b < i comes from the prefix partials; the
// diagonal is the sum of the in-block terms, and above it Mc does not enter
// the output (0).
// With groups > 1 the units of a head are split over blockIdx.z / mc_heads
// (group g takes every groups-th unit) into partial[g][h][M][M], which
// bwd_mc_reduce_kernel then sums in group order: a few tiles of dMc over
// many units would otherwise leave most of the GPU idle.
__device__ __forceinline__ float mc_assemble(const Plan& p, int h, int ustep, int i, int b, float acc,
                                             const float* __restrict__ dnp, const float* __restrict__ diag) {
  const int rows = p.M * p.splits;
  if (diag && b >= i) {
    float t = 0.f;
    if (b == i)
      for (int u = h; u < p.BH; u += ustep) t += diag[(size_t)u * p.M + i];
    return t;
  }
  if (p.norm == MHLA_NORM_MALA) {
    float dn = 0.f;
    for (int u = h; u < p.BH; u += ustep)
      for (int s = 0; s < p.splits; ++s) dn += dnp[(size_t)u * rows + (size_t)i * p.splits + s];
    acc = fmaf((float)p.nb, dn, acc);
  }
  return acc;
}

// 64 x 64 entries of dMc per CTA (4 x 4 per thread, rows ti + 16 a, columns
// tb + 16 c), the record dimension taken in chunks of 32 through shared
// memory; each unit's products are summed before they join the total.
__global__ void __launch_bounds__(kThreads)
bwd_mc_kernel(Plan p, const float* __restrict__ dmixp, const float* __restrict__ stack,
              const float* __restrict__ dnp, const float* __restrict__ diag, float* __restrict__ dmc, int groups,
              float* __restrict__ partial) {
  constexpr int TI = kMcTile, TK = 32;
  __shared__ float sa[TK][TI + 1];
  __shared__ float sb[TK][TI + 1];
  const int i0 = blockIdx.y * TI, b0 = blockIdx.x * TI;
  const int ti = threadIdx.x / 16, tb = threadIdx.x % 16;
  const int rows = p.M * p.splits;
  const int h = (int)blockIdx.z % p.mc_heads, g = (int)blockIdx.z / p.mc_heads;
  const int ustep = p.mc_heads == 1 ? 1 : p.H;
  float acc[4][4];
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[a][c] = 0.f;
  // causal form: a tile on or above the diagonal holds no product term
  const bool products = !(diag && b0 >= i0 + TI - 1);
  for (int u = h + g * ustep; products && u < p.BH; u += groups * ustep) {
    float acc_u[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc_u[a][c] = 0.f;
    const float* da = dmixp + (size_t)u * rows * p.R;
    const float* xa = stack + (size_t)u * rows * p.R;
    for (int r0 = 0; r0 < p.R; r0 += TK) {
      __syncthreads();
      for (int e = threadIdx.x; e < TI * TK; e += kThreads) {
        const int ii = e / TK, rr = e % TK;
        const int r = r0 + rr;
        float x = 0.f, y = 0.f;
        if (r < p.R) {
          if (i0 + ii < p.M)
            for (int s = 0; s < p.splits; ++s) x += da[((size_t)(i0 + ii) * p.splits + s) * p.R + r];
          if (b0 + ii < p.M)
            for (int s = 0; s < p.splits; ++s) y += xa[((size_t)(b0 + ii) * p.splits + s) * p.R + r];
        }
        sa[rr][ii] = x;
        sb[rr][ii] = y;
      }
      __syncthreads();
      // each chunk's 32 products are summed before they join the unit's sum
      float part[4][4];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int c = 0; c < 4; ++c) part[a][c] = 0.f;
#pragma unroll 8
      for (int rr = 0; rr < TK; ++rr) {
        float av[4], bv[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          av[a] = sa[rr][ti + 16 * a];
          bv[a] = sb[rr][tb + 16 * a];
        }
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int c = 0; c < 4; ++c) part[a][c] = fmaf(av[a], bv[c], part[a][c]);
      }
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc_u[a][c] += part[a][c];
    }
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[a][c] += acc_u[a][c];
  }
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int i = i0 + ti + 16 * a, b = b0 + tb + 16 * c;
      if (i >= p.M || b >= p.M) continue;
      if (groups > 1)
        partial[(((size_t)g * p.mc_heads + h) * p.M + i) * p.M + b] = acc[a][c];
      else
        dmc[((size_t)h * p.M + i) * p.M + b] = mc_assemble(p, h, ustep, i, b, acc[a][c], dnp, diag);
    }
}

// dMc[h][i][b] from the groups' partial sums, in group order.
__global__ void __launch_bounds__(kThreads)
bwd_mc_reduce_kernel(Plan p, const float* __restrict__ partial, int groups, const float* __restrict__ dnp,
                     const float* __restrict__ diag, float* __restrict__ dmc) {
  const size_t n = (size_t)p.mc_heads * p.M * p.M;
  const size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
  if (e >= n) return;
  const int h = (int)(e / ((size_t)p.M * p.M));
  const int i = (int)(e / p.M % p.M), b = (int)(e % p.M);
  float acc = 0.f;
  for (int g = 0; g < groups; ++g) acc += partial[(size_t)g * n + e];
  dmc[e] = mc_assemble(p, h, p.mc_heads == 1 ? 1 : p.H, i, b, acc, dnp, diag);
}

// One CTA per (summary block piece, head): dS_b, dz_b, dv_b in shared memory;
// dk_j = (dS_b v_j + dz_b) * phi'(k_j), dv_j = dS_b^T phi(k_j) + dv_b (the
// causal form adds the in-block parts xk, xv before phi').
template <int D, typename T>
__global__ void __launch_bounds__(kThreads)
bwd_summary_kernel(Plan p, const T* __restrict__ K, const T* __restrict__ V, const float* __restrict__ dstack,
                   const float* __restrict__ xk, const float* __restrict__ xv, T* __restrict__ dK,
                   T* __restrict__ dV) {
  // rows LD = D + 1 floats apart; thread (mg, nl) keeps tokens mg, mg + MG
  // and features nl + NL * b of the tile in registers
  constexpr int LD = D + 1, MG = kTile / 2, NL = kThreads / MG, RN = D / NL;
  static_assert(NL <= 32 && RN * NL == D, "tile split");
  extern __shared__ float sm[];
  float* sS = sm;                  // D rows: dS_b
  float* sz = sS + D * LD;         // D
  float* sv = sz + D;              // D
  float* sk = sv + D;              // kTile rows: phi(k)
  float* sx = sk + kTile * LD;     // kTile rows: v
  const int u = blockIdx.y;
  const int row = blockIdx.x;
  const int b = row / p.splits;
  const int l0 = (row % p.splits) * p.split_len;
  const int l1 = min(p.nb, l0 + p.split_len);
  const int tid = threadIdx.x, mg = tid / NL, nl = tid % NL;
  const float* drow = dstack + ((size_t)u * p.M + b) * p.R;
  for (int e = tid; e < D * D; e += kThreads) sS[e / D * LD + e % D] = drow[e];
  for (int e = tid; e < 2 * D; e += kThreads) sz[e] = drow[D * D + e];
  for (int lt = l0; lt < l1; lt += kTile) {
    const int cnt = min(kTile, l1 - lt);
    __syncthreads();
    for (int e = tid; e < kTile * D; e += kThreads) {
      const int tt = e / D, f = e % D;
      float kx = 0.f, vx = 0.f;
      if (tt < cnt) {
        const size_t off = tok_off(p, u, block_token(p, b, lt + tt)) + f;
        kx = phi_apply(to_f32(K[off]), p.fmap);
        vx = to_f32(V[off]);
      }
      sk[tt * LD + f] = kx;
      sx[tt * LD + f] = vx;
    }
    __syncthreads();
    float gk[2][RN], gv[2][RN];
#pragma unroll
    for (int c = 0; c < RN; ++c) {
      gk[0][c] = gk[1][c] = sz[nl + NL * c];
      gv[0][c] = gv[1][c] = sv[nl + NL * c];
    }
    for (int m = 0; m < D; ++m) {
      const float x0 = sx[mg * LD + m], x1 = sx[(mg + MG) * LD + m];
      const float k0 = sk[mg * LD + m], k1 = sk[(mg + MG) * LD + m];
#pragma unroll
      for (int c = 0; c < RN; ++c) {
        const int f = nl + NL * c;
        const float sf = sS[f * LD + m], sc = sS[m * LD + f];
        gk[0][c] = fmaf(sf, x0, gk[0][c]);   // (dS_b v_j)[f]
        gk[1][c] = fmaf(sf, x1, gk[1][c]);
        gv[0][c] = fmaf(sc, k0, gv[0][c]);   // (dS_b^T phi(k_j))[f]
        gv[1][c] = fmaf(sc, k1, gv[1][c]);
      }
    }
#pragma unroll
    for (int a = 0; a < 2; ++a) {
      const int tt = mg + MG * a;
      if (tt >= cnt) continue;
      const size_t base = tok_off(p, u, block_token(p, b, lt + tt));
#pragma unroll
      for (int c = 0; c < RN; ++c) {
        const size_t off = base + nl + NL * c;
        float k_ = gk[a][c], v_ = gv[a][c];
        if (xk) {
          k_ += xk[off];
          v_ += xv[off];
        }
        dK[off] = from_f32<T>(k_ * phi_grad(to_f32(K[off]), p.fmap));
        dV[off] = from_f32<T>(v_);
      }
    }
  }
}

template <int D, typename T>
int run_output(const Plan& p, const BwdBuffers& w, const void* q, const void* dout, void* dq, cudaStream_t s) {
  const size_t smo = sizeof(float) * (D * (D + 1) + 2 * D + 3 * kTile * (D + 1) + 4 * kTile);
  auto ko = bwd_output_kernel<D, T>;
  cudaError_t e = (cudaError_t)set_max_dynamic_smem((const void*)ko, (int)smo);
  if (e != cudaSuccess) return (int)e;
  ko<<<dim3(p.M * p.splits, p.BH), kThreads, smo, s>>>(p, (const T*)q, (const T*)dout, w.mixed, w.rowsum, (T*)dq,
                                                       w.dmixp, w.dnp);
  return (int)cudaGetLastError();
}

template <int D, typename T>
int run_summary(const Plan& p, const BwdBuffers& w, const void* k, const void* v, void* dk, void* dv,
                cudaStream_t s) {
  const size_t sms = sizeof(float) * (D * (D + 1) + 2 * D + 2 * kTile * (D + 1));
  auto ks = bwd_summary_kernel<D, T>;
  cudaError_t e = (cudaError_t)set_max_dynamic_smem((const void*)ks, (int)sms);
  if (e != cudaSuccess) return (int)e;
  ks<<<dim3(p.M * p.splits, p.BH), kThreads, sms, s>>>(p, (const T*)k, (const T*)v, w.dstack, w.xk, w.xv, (T*)dk,
                                                       (T*)dv);
  return (int)cudaGetLastError();
}

template <typename T>
int output_t(const Plan& p, const BwdBuffers& w, const void* q, const void* dout, void* dq, cudaStream_t s) {
  switch (p.d) {
    case 16: return run_output<16, T>(p, w, q, dout, dq, s);
    case 32: return run_output<32, T>(p, w, q, dout, dq, s);
    case 64: return run_output<64, T>(p, w, q, dout, dq, s);
    case 128: return run_output<128, T>(p, w, q, dout, dq, s);
  }
  return (int)cudaErrorInvalidValue;
}

template <typename T>
int summary_t(const Plan& p, const BwdBuffers& w, const void* k, const void* v, void* dk, void* dv, cudaStream_t s) {
  switch (p.d) {
    case 16: return run_summary<16, T>(p, w, k, v, dk, dv, s);
    case 32: return run_summary<32, T>(p, w, k, v, dk, dv, s);
    case 64: return run_summary<64, T>(p, w, k, v, dk, dv, s);
    case 128: return run_summary<128, T>(p, w, k, v, dk, dv, s);
  }
  return (int)cudaErrorInvalidValue;
}

}  // namespace

int launch_bwd_output(const Plan& p, const BwdBuffers& w, const void* q, const void* dout, void* dq, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (p.dtype == MHLA_DTYPE_F32) return output_t<float>(p, w, q, dout, dq, s);
  return output_t<__nv_bfloat16>(p, w, q, dout, dq, s);
}

int launch_bwd_mix(const Plan& p, const BwdBuffers& w, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  bwd_mix_kernel<<<dim3((p.R + 127) / 128, (p.M + 31) / 32, p.BH), kThreads, 0, s>>>(p, w.mc, w.dmixp, w.dstack);
  return (int)cudaGetLastError();
}

int bwd_mc_groups(const Plan& p) {
  // about four CTAs per SM of a 152-SM GPU, at most one group per unit of a
  // head and 64 groups
  const long long tiles = (long long)((p.M + kMcTile - 1) / kMcTile) * ((p.M + kMcTile - 1) / kMcTile) * p.mc_heads;
  const int units = p.mc_heads == 1 ? p.BH : p.BH / p.H;
  long long g = (608 + tiles - 1) / tiles;
  if (g > units) g = units;
  if (g > 64) g = 64;
  return g < 1 ? 1 : (int)g;
}

size_t bwd_mc_partial_bytes(const Plan& p) {
  const int g = bwd_mc_groups(p);
  return g > 1 ? sizeof(float) * (size_t)g * p.mc_heads * p.M * p.M : 0;
}

int launch_bwd_mc(const Plan& p, const BwdBuffers& w, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int groups = bwd_mc_groups(p);
  const unsigned nt = (unsigned)((p.M + kMcTile - 1) / kMcTile);
  bwd_mc_kernel<<<dim3(nt, nt, p.mc_heads * groups), kThreads, 0, s>>>(
      p, w.dmixp, w.stack, w.dnp, w.diag, w.dmc, groups, w.mc_partial);
  if (groups > 1) {
    const size_t n = (size_t)p.mc_heads * p.M * p.M;
    bwd_mc_reduce_kernel<<<(unsigned)((n + kThreads - 1) / kThreads), kThreads, 0, s>>>(p, w.mc_partial, groups,
                                                                                       w.dnp, w.diag, w.dmc);
  }
  return (int)cudaGetLastError();
}

int launch_bwd_summary(const Plan& p, const BwdBuffers& w, const void* k, const void* v, void* dk, void* dv,
                       void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (p.dtype == MHLA_DTYPE_F32) return summary_t<float>(p, w, k, v, dk, dv, s);
  return summary_t<__nv_bfloat16>(p, w, k, v, dk, dv, s);
}

}  // namespace mhla
