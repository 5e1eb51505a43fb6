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

// Tile geometry.  Each step of a kernel is a small product on shared
// memory, split over the CTA so that a thread keeps a register tile and a
// warp reads each operand value either as one broadcast or from 16-32
// different banks (rows of the D-wide arrays are LD = D + 1 floats apart):
//   token x feature  (TQ x D): 2 x RN per thread, rows t = mg + MG a,
//                    columns c = nl + NL b (NL threads per row group, all
//                    in one warp)
//   token x token    (TQ x TQ): 2 x 2 per thread, rows ti + TH a, columns ji + TH b
//   feature x feature (D x D): 4 x 4 per thread, rows fi + FQ a, columns ci + FQ b
template <int D>
struct Geo {
  static constexpr int TQ = D <= 64 ? 32 : 16;  // tokens per tile
  static constexpr int LD = D + 1;
  static constexpr int MG = TQ / 2;
  static constexpr int NL = kThreads / MG;
  static constexpr int RN = D / NL;
  static constexpr int TH = TQ / 2;
  static constexpr int FQ = D / 4;
  static constexpr int FT = (FQ * FQ + kThreads - 1) / kThreads;
  static_assert(NL <= 32 && 32 % NL == 0 && RN >= 1 && RN * NL == D, "token x feature split");
  static_assert(TH * TH <= kThreads && 2 * D <= kThreads, "tile split");
};

// Token rows of the per-token buffer the forward walk leaves for the reverse
// walk: dnum (D), ds, gamma and two floats of padding (16-byte rows).
template <int D>
struct TokRow {
  static constexpr int value = D + 4;
};

template <int D>
constexpr size_t fwd_smem_floats() {
  using G = Geo<D>;
  return 2 * D * G::LD + 4 * D + 5 * G::TQ * G::LD + G::TQ * G::TQ + 6 * G::TQ + 4 * kWarps;
}

// Bytes of the raw tiles in front of the float arrays: four token arrays
// (forward walk) or four token arrays and the per-token rows (reverse walk).
template <int D, typename T>
__host__ __device__ constexpr size_t fwd_raw_bytes() {
  return 4 * (size_t)Geo<D>::TQ * D * sizeof(T);
}
template <int D, typename T>
__host__ __device__ constexpr size_t rev_raw_bytes() {
  return 4 * (size_t)Geo<D>::TQ * D * sizeof(T) + (size_t)Geo<D>::TQ * TokRow<D>::value * sizeof(float);
}

template <int D>
constexpr size_t rev_smem_floats() {
  using G = Geo<D>;
  return D * G::LD + 2 * D + 5 * G::TQ * G::LD + 2 * G::TQ * G::TQ + G::TQ;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Sum over the NL threads of a row group (lanes aligned to NL in the warp).
template <int NL>
__device__ __forceinline__ float group_sum(float x) {
#pragma unroll
  for (int o = NL / 2; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

__device__ __forceinline__ float phi_grad(float x, int fmap) { return phi_deriv(x, phi_apply(x, fmap), fmap); }

// Asynchronous 16-byte copies global -> shared: the next tile's raw rows
// land while the current tile is worked on.
__device__ __forceinline__ void cpa16(void* dst, const void* src) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cpa_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cpa_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }

// Copies the raw rows of tile l0 (cnt tokens of block i, unit u) of the
// first n of the token arrays s0..s3 into raw[a][TQ][D] (rows at or past
// cnt are left as they are).
template <int D, int TQ, typename T>
__device__ __forceinline__ void prefetch_rows(const Plan& p, int u, int i, int l0, int cnt, const T* s0,
                                              const T* s1, const T* s2, const T* s3, int n, T* raw) {
  constexpr int CH = D * (int)sizeof(T) / 16;   // 16-byte pieces per row
  constexpr int EPC = 16 / (int)sizeof(T);      // elements per piece
  for (int e = threadIdx.x; e < n * TQ * CH; e += kThreads) {
    const int a = e / (TQ * CH), r = e % (TQ * CH), tt = r / CH, ch = r % CH;
    const T* src = a == 0 ? s0 : (a == 1 ? s1 : (a == 2 ? s2 : s3));
    if (tt < cnt)
      cpa16(raw + ((size_t)a * TQ + tt) * D + ch * EPC, src + tok_off(p, u, block_token(p, i, l0 + tt)) + ch * EPC);
  }
}

// Shared memory: C = Sp_i + w R and R (D rows each), zp, vp, rz, rv (D each)
// | tiles of phi(q), phi(k), v, dO, dnum (TQ rows each) | in-tile scores,
// later the in-tile dq weights E (TQ*TQ) | per token s, phi(q).rz, n, coef,
// ds, gamma (TQ each) | per-warp sums of the diagonal term and of dn~.
template <int D, typename T>
__global__ void __launch_bounds__(kThreads, D <= 64 ? 2 : 1)
causal_bwd_fwd_kernel(Plan p, const T* __restrict__ Q, const T* __restrict__ K, const T* __restrict__ V,
                      const T* __restrict__ dO, const float* __restrict__ mixed,
                      const float* __restrict__ rowsum_lower, const float* __restrict__ mc, T* __restrict__ dQ,
                      float* __restrict__ dmixp, float* __restrict__ dnp, float* __restrict__ diag,
                      float* __restrict__ tokbuf) {
  using G = Geo<D>;
  constexpr int TQ = G::TQ, LD = G::LD, MG = G::MG, NL = G::NL, RN = G::RN, TH = G::TH, FQ = G::FQ, FT = G::FT;
  extern __shared__ __align__(16) unsigned char smraw[];
  T* raw = reinterpret_cast<T*>(smraw);   // Q, K, V, dO rows of the next tile [4][TQ][D]
  float* sm = reinterpret_cast<float*>(smraw + fwd_raw_bytes<D, T>());
  float* sC = sm;               // Sp_i + w R
  float* sR = sC + D * LD;      // in-block state R (without w)
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
  float* ss = sa + TQ * TQ;     // s_t
  float* ssin = ss + TQ;        // phi(q_t) . rz_t
  float* snt = ssin + TQ;       // n_t
  float* scf = snt + TQ;        // dnum_t / dO_t
  float* sds = scf + TQ;        // ds
  float* sgm = sds + TQ;        // gamma
  double* sdg = reinterpret_cast<double*>(sgm + TQ);  // per-warp sums: diagonal term, dn~ [kWarps] each
  const int u = blockIdx.y, i = blockIdx.x;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int mg = tid / NL, nl = tid % NL;         // token x feature split
  const int jm = mc_index(p, u);
  const float w = mc[((size_t)jm * p.M + i) * p.M + i];
  const float* mrow = mixed + ((size_t)u * p.M + i) * p.R;
  for (int e = tid; e < D * D; e += kThreads) {
    sC[e / D * LD + e % D] = mrow[e];
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

  float acc[FT][4][4];          // dSp_i, feature x feature tiles
#pragma unroll
  for (int x = 0; x < FT; ++x)
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) acc[x][a][b] = 0.f;
  float zacc = 0.f, vacc = 0.f;
  // the diagonal term sums many cancelling per-token terms: formed and
  // summed in double
  double nacc = 0.0, dacc = 0.0;
  float rn = 0.f;  // tokens of the block before the tile

  prefetch_rows<D, TQ>(p, u, i, 0, min(TQ, p.nb), Q, K, V, dO, 4, raw);
  cpa_commit();
  for (int l0 = 0; l0 < p.nb; l0 += TQ) {
    const int cnt = min(TQ, p.nb - l0);
    cpa_wait_all();
    __syncthreads();
    for (int e = tid; e < TQ * D; e += kThreads) {
      const int tt = e / D, f = e % D;
      float qx = 0.f, kx = 0.f, vx = 0.f, gx = 0.f;
      if (tt < cnt) {
        qx = phi_apply(to_f32(raw[e]), p.fmap);
        kx = phi_apply(to_f32(raw[TQ * D + e]), p.fmap);
        vx = to_f32(raw[2 * TQ * D + e]);
        gx = to_f32(raw[3 * TQ * D + e]);
      }
      sq[tt * LD + f] = qx;
      sk[tt * LD + f] = kx;
      sx[tt * LD + f] = vx;
      sg[tt * LD + f] = gx;
    }
    __syncthreads();
    if (l0 + TQ < p.nb) prefetch_rows<D, TQ>(p, u, i, l0 + TQ, min(TQ, p.nb - l0 - TQ), Q, K, V, dO, 4, raw);
    cpa_commit();
    // masked in-tile scores a[t][j] = phi(q_t) . phi(k_j), j <= t
    if (tid < TH * TH) {
      const int ti = tid / TH, ji = tid % TH;
      float c2[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
      for (int f = 0; f < D; ++f) {
        const float q0 = sq[ti * LD + f], q1 = sq[(ti + TH) * LD + f];
        const float k0 = sk[ji * LD + f], k1 = sk[(ji + TH) * LD + f];
        c2[0][0] = fmaf(q0, k0, c2[0][0]);
        c2[0][1] = fmaf(q0, k1, c2[0][1]);
        c2[1][0] = fmaf(q1, k0, c2[1][0]);
        c2[1][1] = fmaf(q1, k1, c2[1][1]);
      }
#pragma unroll
      for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          const int tt = ti + TH * a, jj = ji + TH * b;
          sa[tt * TQ + jj] = (jj <= tt && tt < cnt) ? c2[a][b] : 0.f;
        }
    }
    // phi(q_t)^T C and phi(q_t)^T R, kept in registers for the norm step
    float ac[2][RN], ar[2][RN];
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
      for (int b = 0; b < RN; ++b) ac[a][b] = ar[a][b] = 0.f;
    for (int f = 0; f < D; ++f) {
      const float x0 = sq[mg * LD + f], x1 = sq[(mg + MG) * LD + f];
#pragma unroll
      for (int b = 0; b < RN; ++b) {
        const float cv = sC[f * LD + nl + NL * b], rv = sR[f * LD + nl + NL * b];
        ac[0][b] = fmaf(x0, cv, ac[0][b]);
        ac[1][b] = fmaf(x1, cv, ac[1][b]);
        ar[0][b] = fmaf(x0, rv, ar[0][b]);
        ar[1][b] = fmaf(x1, rv, ar[1][b]);
      }
    }
    __syncthreads();
    // per token: s_t, phi(q_t) . rz_t, n_t and dnum_t / dO_t
    for (int tt = warp; tt < TQ; tt += kWarps) {
      float sp = 0.f, sin = 0.f;
      for (int f = lane; f < D; f += 32) {
        sp = fmaf(sq[tt * LD + f], zP[f], sp);
        sin = fmaf(sq[tt * LD + f], zR[f], sin);
      }
      if (lane < TQ) sin += sa[tt * TQ + lane];
      sp = warp_sum(sp);
      sin = warp_sum(sin);
      if (lane == 0) {
        const float s = fmaf(w, sin, sp);
        const float nt = fmaf(w, rn + (float)(tt + 1), n_pre);
        const bool live = tt < cnt && (p.norm == MHLA_NORM_NONE || s != 0.f);
        ss[tt] = s;
        ssin[tt] = sin;
        snt[tt] = nt;
        scf[tt] = !live ? 0.f : (p.norm == MHLA_NORM_DIVISIVE ? 1.f / s : (mala ? 1.f + 1.f / s : 1.f));
      }
    }
    __syncthreads();
    // phi(q_t)^T R_t's in-tile part sum_{j<=t} a[t][j] v_j and rv_t's sum_{j<=t} v_j;
    // then the norm gradients of each token
    {
      float lo[2][RN], vl[2][RN];
#pragma unroll
      for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int b = 0; b < RN; ++b) lo[a][b] = vl[a][b] = 0.f;
      const int t0 = mg, t1 = mg + MG;
      for (int jj = 0; jj < cnt; ++jj) {
        const float a0 = sa[t0 * TQ + jj], a1 = sa[t1 * TQ + jj];
        const float m0 = jj <= t0 ? 1.f : 0.f, m1 = jj <= t1 ? 1.f : 0.f;
#pragma unroll
        for (int b = 0; b < RN; ++b) {
          const float xv = sx[jj * LD + nl + NL * b];
          lo[0][b] = fmaf(a0, xv, lo[0][b]);
          lo[1][b] = fmaf(a1, xv, lo[1][b]);
          vl[0][b] = fmaf(m0, xv, vl[0][b]);
          vl[1][b] = fmaf(m1, xv, vl[1][b]);
        }
      }
#pragma unroll
      for (int a = 0; a < 2; ++a) {
        const int tt = mg + MG * a;
        const float coef = scf[tt];
        float gnum = 0.f, gvt = 0.f, gain = 0.f, gvin = 0.f;
#pragma unroll
        for (int b = 0; b < RN; ++b) {
          const int c = nl + NL * b;
          const float ain = ar[a][b] + lo[a][b];      // phi(q_t)^T R_t, column c
          const float num = fmaf(w, lo[a][b], ac[a][b]);
          const float vin = vR[c] + vl[a][b];          // rv_t
          const float vt = fmaf(w, vin, vP[c]);
          const float g = sg[tt * LD + c];
          gnum = fmaf(g, num, gnum);
          gvt = fmaf(g, vt, gvt);
          gain = fmaf(g, ain, gain);
          gvin = fmaf(g, vin, gvin);
          sdn[tt * LD + c] = coef * g;
        }
        gnum = group_sum<NL>(gnum);
        gvt = group_sum<NL>(gvt);
        gain = group_sum<NL>(gain);
        gvin = group_sum<NL>(gvin);
        if (nl == 0) {
          const float s = ss[tt], sin = ssin[tt], nt = snt[tt];
          const float rnt = rn + (float)(tt + 1);
          const bool live = tt < cnt && (p.norm == MHLA_NORM_NONE || s != 0.f);
          float ds = 0.f, gamma = 0.f, dnt = 0.f;
          if (live && p.norm == MHLA_NORM_DIVISIVE) {
            ds = -gnum / (s * s);
          } else if (live && mala) {
            const float dgamma = -gvt;
            ds = -gnum / (s * s) + dgamma / nt;
            gamma = s / nt;
            dnt = -dgamma * s / (nt * nt);
          }
          sds[tt] = ds;
          sgm[tt] = gamma;
          if (tt < cnt) {
            // <dS~_t, R_t> + ds_t (phi(q_t) . rz_t) + <dv~_t, rv_t> + dn~_t rn_t
            dacc += (double)coef * gain + (double)ds * sin - (double)gamma * gvin + (double)dnt * rnt;
            nacc += dnt;
          }
        }
      }
    }
    __syncthreads();
    // in-tile dq weights E[t][j] = v_j . dnum_t + ds_t, j <= t
    if (tid < TH * TH) {
      const int ti = tid / TH, ji = tid % TH;
      float c2[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
      for (int c = 0; c < D; ++c) {
        const float d0 = sdn[ti * LD + c], d1 = sdn[(ti + TH) * LD + c];
        const float x0 = sx[ji * LD + c], x1 = sx[(ji + TH) * LD + c];
        c2[0][0] = fmaf(d0, x0, c2[0][0]);
        c2[0][1] = fmaf(d0, x1, c2[0][1]);
        c2[1][0] = fmaf(d1, x0, c2[1][0]);
        c2[1][1] = fmaf(d1, x1, c2[1][1]);
      }
#pragma unroll
      for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          const int tt = ti + TH * a, jj = ji + TH * b;
          sa[tt * TQ + jj] = (jj <= tt && tt < cnt) ? c2[a][b] + sds[tt] : 0.f;
        }
    }
    __syncthreads();
    // dq_t = (C dnum_t + (zp + w rz) ds_t + w sum_{j<=t} E[t][j] phi(k_j)) phi'(q_t)
    {
      float dqa[2][RN], lk[2][RN];
#pragma unroll
      for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int b = 0; b < RN; ++b) dqa[a][b] = lk[a][b] = 0.f;
      const int t0 = mg, t1 = mg + MG;
      for (int c = 0; c < D; ++c) {
        const float d0 = sdn[t0 * LD + c], d1 = sdn[t1 * LD + c];
#pragma unroll
        for (int b = 0; b < RN; ++b) {
          const float cv = sC[(nl + NL * b) * LD + c];
          dqa[0][b] = fmaf(d0, cv, dqa[0][b]);
          dqa[1][b] = fmaf(d1, cv, dqa[1][b]);
        }
      }
      for (int jj = 0; jj < cnt; ++jj) {
        const float e0 = sa[t0 * TQ + jj], e1 = sa[t1 * TQ + jj];
#pragma unroll
        for (int b = 0; b < RN; ++b) {
          const float kv = sk[jj * LD + nl + NL * b];
          lk[0][b] = fmaf(e0, kv, lk[0][b]);
          lk[1][b] = fmaf(e1, kv, lk[1][b]);
        }
      }
#pragma unroll
      for (int a = 0; a < 2; ++a) {
        const int tt = mg + MG * a;
        if (tt >= cnt) continue;
        const size_t base = tok_off(p, u, block_token(p, i, l0 + tt));
#pragma unroll
        for (int b = 0; b < RN; ++b) {
          const int k = nl + NL * b;
          const float x = fmaf(w, lk[a][b], fmaf(fmaf(w, zR[k], zP[k]), sds[tt], dqa[a][b]));
          dQ[base + k] = from_f32<T>(x * phi_grad(to_f32(Q[base + k]), p.fmap));
        }
      }
    }
    __syncthreads();
    // dSp += phi(q_t) dnum_t^T and the in-block state R += phi(k_j) v_j^T (C by w times it)
#pragma unroll
    for (int x = 0; x < FT; ++x) {
      const int qd = tid + kThreads * x;
      if (qd >= FQ * FQ) break;
      const int fi = qd / FQ, ci = qd % FQ;
      float st[4][4];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) st[a][b] = 0.f;
      for (int tt = 0; tt < cnt; ++tt) {
        float qa[4], ka[4], db[4], xb[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          qa[a] = sq[tt * LD + fi + FQ * a];
          ka[a] = sk[tt * LD + fi + FQ * a];
          db[a] = sdn[tt * LD + ci + FQ * a];
          xb[a] = sx[tt * LD + ci + FQ * a];
        }
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            acc[x][a][b] = fmaf(qa[a], db[b], acc[x][a][b]);
            st[a][b] = fmaf(ka[a], xb[b], st[a][b]);
          }
      }
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const int e = (fi + FQ * a) * LD + ci + FQ * b;
          sR[e] += st[a][b];
          sC[e] = fmaf(w, st[a][b], sC[e]);
        }
    }
    // dzp += ds_t phi(q_t), dvp += -gamma_t dO_t; rz, rv advance by the tile
    if (tid < D) {
      float z = 0.f;
      for (int tt = 0; tt < cnt; ++tt) {
        zacc = fmaf(sds[tt], sq[tt * LD + tid], zacc);
        z += sk[tt * LD + tid];
      }
      zR[tid] += z;
    } else if (tid < 2 * D) {
      const int c = tid - D;
      float z = 0.f;
      for (int tt = 0; tt < cnt; ++tt) {
        if (mala) vacc = fmaf(-sgm[tt], sg[tt * LD + c], vacc);
        z += sx[tt * LD + c];
      }
      vR[c] += z;
    }
    // per token for the reverse walk: dnum (D), ds, gamma
    for (int e = tid; e < cnt * (D + 2); e += kThreads) {
      const int tt = e / (D + 2), c = e % (D + 2);
      const float x = c < D ? sdn[tt * LD + c] : (c == D ? sds[tt] : sgm[tt]);
      tokbuf[((size_t)u * p.N + block_token(p, i, l0 + tt)) * TokRow<D>::value + c] = x;
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
  for (int x = 0; x < FT; ++x) {
    const int qd = tid + kThreads * x;
    if (qd >= FQ * FQ) break;
    const int fi = qd / FQ, ci = qd % FQ;
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) out[(fi + FQ * a) * D + ci + FQ * b] = acc[x][a][b];
  }
  if (tid < D) out[D * D + tid] = zacc;
  else if (tid < 2 * D) out[D * D + tid] = vacc;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    dacc += __shfl_xor_sync(0xffffffffu, dacc, o);
    nacc += __shfl_xor_sync(0xffffffffu, nacc, o);
  }
  if (lane == 0) {
    sdg[warp] = dacc;
    sdg[kWarps + warp] = nacc;
  }
  __syncthreads();
  if (tid == 0) {
    double t = 0.0, n = 0.0;
    for (int x = 0; x < kWarps; ++x) {
      t += sdg[x];
      n += sdg[kWarps + x];
    }
    diag[(size_t)u * p.M + i] = (float)t;
    dnp[row0] = (float)n;
  }
}

// Shared memory: GS (D rows), Gz, Gv (D) | tiles of phi(q), phi(k), v,
// dnum, dv~ (TQ rows each) | E[j][t] = dnum_t . v_j + ds_t and P[j][t] =
// phi(q_t) . phi(k_j), t >= j (TQ*TQ each) | ds (TQ).
template <int D, typename T>
__global__ void __launch_bounds__(kThreads, D <= 64 ? 2 : 1)
causal_bwd_rev_kernel(Plan p, const T* __restrict__ Q, const T* __restrict__ K, const T* __restrict__ V,
                      const T* __restrict__ dO, const float* __restrict__ mc, const float* __restrict__ tokbuf,
                      float* __restrict__ xk, float* __restrict__ xv) {
  using G = Geo<D>;
  constexpr int TQ = G::TQ, LD = G::LD, MG = G::MG, NL = G::NL, RN = G::RN, TH = G::TH, FQ = G::FQ, FT = G::FT;
  extern __shared__ __align__(16) unsigned char smraw[];
  T* raw = reinterpret_cast<T*>(smraw);   // Q, K, V, dO rows of the next tile [4][TQ][D]
  float* rtok = reinterpret_cast<float*>(smraw + 4 * (size_t)TQ * D * sizeof(T));  // [TQ][TokRow]
  float* sm = reinterpret_cast<float*>(smraw + rev_raw_bytes<D, T>());
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
  const int mg = tid / NL, nl = tid % NL;
  const int jm = mc_index(p, u);
  const float w = mc[((size_t)jm * p.M + i) * p.M + i];
  const bool mala = p.norm == MHLA_NORM_MALA;
  for (int e = tid; e < D * LD + 2 * D; e += kThreads) sm[e] = 0.f;

  constexpr int TR = TokRow<D>::value;
  const int narr = mala ? 4 : 3;
  // raw rows of tile l0: the token arrays and the forward walk's per-token rows
  auto prefetch = [&](int l0n) {
    const int cntn = min(TQ, p.nb - l0n);
    prefetch_rows<D, TQ>(p, u, i, l0n, cntn, Q, K, V, dO, narr, raw);
    for (int e = tid; e < TQ * (TR / 4); e += kThreads) {
      const int tt = e / (TR / 4), ch = e % (TR / 4);
      if (tt < cntn)
        cpa16(rtok + tt * TR + 4 * ch, tokbuf + ((size_t)u * p.N + block_token(p, i, l0n + tt)) * TR + 4 * ch);
    }
    cpa_commit();
  };
  prefetch((p.nb - 1) / TQ * TQ);
  for (int l0 = (p.nb - 1) / TQ * TQ; l0 >= 0; l0 -= TQ) {
    const int cnt = min(TQ, p.nb - l0);
    cpa_wait_all();
    __syncthreads();
    for (int e = tid; e < TQ * D; e += kThreads) {
      const int tt = e / D, f = e % D;
      float qx = 0.f, kx = 0.f, vx = 0.f, dn = 0.f, gv = 0.f;
      if (tt < cnt) {
        const float* tb = rtok + tt * TR;
        qx = phi_apply(to_f32(raw[e]), p.fmap);
        kx = phi_apply(to_f32(raw[TQ * D + e]), p.fmap);
        vx = to_f32(raw[2 * TQ * D + e]);
        dn = tb[f];
        if (mala) gv = -tb[D + 1] * to_f32(raw[3 * TQ * D + e]);
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
    if (l0 >= TQ) prefetch(l0 - TQ);
    // E[j][t] and P[j][t] for t >= j
    if (tid < TH * TH) {
      const int ji = tid / TH, ti = tid % TH;
      float e2[2][2] = {{0.f, 0.f}, {0.f, 0.f}}, p2[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
      for (int f = 0; f < D; ++f) {
        const float x0 = sx[ji * LD + f], x1 = sx[(ji + TH) * LD + f];
        const float k0 = sk[ji * LD + f], k1 = sk[(ji + TH) * LD + f];
        const float d0 = sdn[ti * LD + f], d1 = sdn[(ti + TH) * LD + f];
        const float q0 = sq[ti * LD + f], q1 = sq[(ti + TH) * LD + f];
        e2[0][0] = fmaf(x0, d0, e2[0][0]);
        e2[0][1] = fmaf(x0, d1, e2[0][1]);
        e2[1][0] = fmaf(x1, d0, e2[1][0]);
        e2[1][1] = fmaf(x1, d1, e2[1][1]);
        p2[0][0] = fmaf(k0, q0, p2[0][0]);
        p2[0][1] = fmaf(k0, q1, p2[0][1]);
        p2[1][0] = fmaf(k1, q0, p2[1][0]);
        p2[1][1] = fmaf(k1, q1, p2[1][1]);
      }
#pragma unroll
      for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          const int jj = ji + TH * a, tt = ti + TH * b;
          const bool on = tt >= jj && tt < cnt;
          sE[jj * TQ + tt] = on ? e2[a][b] + sds[tt] : 0.f;
          sPm[jj * TQ + tt] = on ? p2[a][b] : 0.f;
        }
    }
    __syncthreads();
    // in-block parts for token j: w (GS v_j + Gz + sum_{t>=j} E[j][t] phi(q_t)) and
    // w (GS^T phi(k_j) + Gv + sum_{t>=j} (P[j][t] dnum_t + dv~_t))
    {
      float gk[2][RN], gv[2][RN];
      const int j0 = mg, j1 = mg + MG;
#pragma unroll
      for (int b = 0; b < RN; ++b) {
        gk[0][b] = gk[1][b] = Gz[nl + NL * b];
        gv[0][b] = gv[1][b] = Gv[nl + NL * b];
      }
      for (int c = 0; c < D; ++c) {
        const float x0 = sx[j0 * LD + c], x1 = sx[j1 * LD + c];
        const float k0 = sk[j0 * LD + c], k1 = sk[j1 * LD + c];
#pragma unroll
        for (int b = 0; b < RN; ++b) {
          const int f = nl + NL * b;
          const float gf = GS[f * LD + c], gc = GS[c * LD + f];
          gk[0][b] = fmaf(gf, x0, gk[0][b]);
          gk[1][b] = fmaf(gf, x1, gk[1][b]);
          gv[0][b] = fmaf(gc, k0, gv[0][b]);
          gv[1][b] = fmaf(gc, k1, gv[1][b]);
        }
      }
      for (int tt = 0; tt < cnt; ++tt) {
        const float e0 = sE[j0 * TQ + tt], e1 = sE[j1 * TQ + tt];
        const float p0 = sPm[j0 * TQ + tt], p1 = sPm[j1 * TQ + tt];
        const float m0 = tt >= j0 ? 1.f : 0.f, m1 = tt >= j1 ? 1.f : 0.f;
#pragma unroll
        for (int b = 0; b < RN; ++b) {
          const int f = nl + NL * b;
          const float qv = sq[tt * LD + f], dv = sdn[tt * LD + f], gt = sgv[tt * LD + f];
          gk[0][b] = fmaf(e0, qv, gk[0][b]);
          gk[1][b] = fmaf(e1, qv, gk[1][b]);
          gv[0][b] = fmaf(m0, gt, fmaf(p0, dv, gv[0][b]));
          gv[1][b] = fmaf(m1, gt, fmaf(p1, dv, gv[1][b]));
        }
      }
#pragma unroll
      for (int a = 0; a < 2; ++a) {
        const int jj = mg + MG * a;
        if (jj >= cnt) continue;
        const size_t base = tok_off(p, u, block_token(p, i, l0 + jj));
#pragma unroll
        for (int b = 0; b < RN; ++b) {
          xk[base + nl + NL * b] = w * gk[a][b];
          xv[base + nl + NL * b] = w * gv[a][b];
        }
      }
    }
    __syncthreads();
    // the tile joins the suffix sums
#pragma unroll
    for (int x = 0; x < FT; ++x) {
      const int qd = tid + kThreads * x;
      if (qd >= FQ * FQ) break;
      const int fi = qd / FQ, ci = qd % FQ;
      float st[4][4];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) st[a][b] = 0.f;
      for (int tt = 0; tt < cnt; ++tt) {
        float qa[4], db[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          qa[a] = sq[tt * LD + fi + FQ * a];
          db[a] = sdn[tt * LD + ci + FQ * a];
        }
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int b = 0; b < 4; ++b) st[a][b] = fmaf(qa[a], db[b], st[a][b]);
      }
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) GS[(fi + FQ * a) * LD + ci + FQ * b] += st[a][b];
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
  }
}

template <int D, typename T>
int run(const Plan& p, const CausalBwdBuffers& c, const void* q, const void* k, const void* v, const void* dout,
        void* dq, cudaStream_t s) {
  const size_t smf = fwd_raw_bytes<D, T>() + sizeof(float) * fwd_smem_floats<D>();
  const size_t smr = rev_raw_bytes<D, T>() + sizeof(float) * rev_smem_floats<D>();
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
