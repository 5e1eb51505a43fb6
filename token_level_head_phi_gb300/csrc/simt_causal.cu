// Block-ordered causal MHLA output on the CUDA cores (float32 arithmetic).
//
// Tokens are ordered by (block, position inside the block); query t of block
// i sees the earlier blocks through the strict lower triangle of Mc and the
// tokens of its own block up to itself through Mc[i, i]:
//     S~_t = S<_i + Mc[i,i] sum_{j in i, j <= t} phi(k_j) v_j^T
//     S<_i = sum_{b < i} Mc[i, b] S_b                 (z, v, n likewise)
// ("MHLA: Restoring Expressivity of Linear Attention via Token-Level
// Multi-Head", key design 2 with its chunkwise, streaming remarks; the pages
// define no causal form, this is the block-ordered reading).  The mixing
// kernel forms S<_i with the masked copy of Mc that launch_mc_strict_lower
// writes.  One CTA per (block, head) walks the block in 32-token tiles (16 at
// d = 128): the tile's own causal part is a masked score matrix, the part
// before it is the running state S<_i + Mc[i,i] (sum of the earlier tiles),
// kept in shared memory and advanced after each tile; the next tile's rows
// arrive by asynchronous copies while the current one is worked on.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace mhla {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

// mcl = Mc with its diagonal and upper triangle zeroed, for `heads` matrices.
__global__ void strict_lower_kernel(int heads, int M, const float* __restrict__ mc, float* __restrict__ mcl) {
  const size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
  if (idx >= (size_t)heads * M * M) return;
  const int r = (int)(idx / M), b = (int)(idx % M), i = r % M;
  mcl[idx] = b < i ? mc[idx] : 0.f;
}

// Tile geometry: every step is a small product on shared-memory tiles whose
// rows are LD = D + 4 floats apart (16-byte rows, so a thread reads up to
// four consecutive values as one vector; 8 consecutive rows start in 8
// different 16-byte bank groups), split so that a thread keeps a register
// tile:
//   token x feature   (TQ x D): 2 x RN, rows mg + MG a, columns RN nl + b
//   token x token     (TQ x TQ): 2 x 2, rows ti + TH a, columns ji + TH b
//                     (the feature sum taken four features at a time)
//   feature x feature (D x D): 4 x 4, rows 4 fi + a, columns 4 ci + b
template <int D>
struct Geo {
  static constexpr int TQ = D <= 64 ? 32 : 16;
  static constexpr int LD = D + 4;
  static constexpr int MG = TQ / 2;
  static constexpr int NL = kThreads / MG;
  static constexpr int RN = D / NL;
  static constexpr int TH = TQ / 2;
  static constexpr int FQ = D / 4;
  static constexpr int FT = (FQ * FQ + kThreads - 1) / kThreads;
  static_assert(NL <= 32 && 32 % NL == 0 && RN >= 1 && RN * NL == D, "token x feature split");
  static_assert(TH * TH <= kThreads && 2 * D <= kThreads, "tile split");
};

template <int D, typename T>
__host__ __device__ constexpr size_t raw_bytes() {
  return 3 * (size_t)Geo<D>::TQ * D * sizeof(T);
}

template <int D>
constexpr size_t smem_floats() {
  using G = Geo<D>;
  return D * G::LD + 2 * D + 3 * G::TQ * G::LD + G::TQ * G::TQ + G::TQ;
}

// RT consecutive floats of shared memory as one vector (RT = 4, 2 or 1).
template <int RT>
__device__ __forceinline__ void lds_vec(const float* src, float (&x)[RT]) {
  if constexpr (RT == 4) {
    const float4 t = *reinterpret_cast<const float4*>(src);
    x[0] = t.x; x[1] = t.y; x[2] = t.z; x[3] = t.w;
  } else if constexpr (RT == 2) {
    const float2 t = *reinterpret_cast<const float2*>(src);
    x[0] = t.x; x[1] = t.y;
  } else {
    x[0] = src[0];
  }
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Asynchronous 16-byte copies global -> shared (the next tile's raw rows).
__device__ __forceinline__ void cpa16(void* dst, const void* src) {
  const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(d), "l"(src) : "memory");
}
__device__ __forceinline__ void cpa_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cpa_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }

// Raw Q, K, V rows of tile l0 (cnt tokens of block i, unit u) into raw[3][TQ][D].
template <int D, int TQ, typename T>
__device__ __forceinline__ void prefetch_rows(const Plan& p, int u, int i, int l0, int cnt, const T* q, const T* k,
                                              const T* v, T* raw) {
  constexpr int CH = D * (int)sizeof(T) / 16;
  constexpr int EPC = 16 / (int)sizeof(T);
  for (int e = threadIdx.x; e < 3 * TQ * CH; e += kThreads) {
    const int a = e / (TQ * CH), r = e % (TQ * CH), tt = r / CH, ch = r % CH;
    const T* src = a == 0 ? q : (a == 1 ? k : v);
    if (tt < cnt)
      cpa16(raw + ((size_t)a * TQ + tt) * D + ch * EPC, src + tok_off(p, u, block_token(p, i, l0 + tt)) + ch * EPC);
  }
  cpa_commit();
}

// Shared memory: raw Q, K, V rows of the next tile | state S (D rows), z, v
// (D each) | phi(q), phi(k), v tiles (TQ rows each) | scores (TQ*TQ) |
// per-token s (TQ).
template <int D, typename T>
__global__ void __launch_bounds__(kThreads, D <= 64 ? 3 : 1)
causal_output_kernel(Plan p, const T* __restrict__ Q, const T* __restrict__ K, const T* __restrict__ V,
                     const float* __restrict__ mixed, const float* __restrict__ rowsum_lower,
                     const float* __restrict__ mc, T* __restrict__ out) {
  using G = Geo<D>;
  constexpr int TQ = G::TQ, LD = G::LD, MG = G::MG, NL = G::NL, RN = G::RN, TH = G::TH, FQ = G::FQ, FT = G::FT;
  extern __shared__ __align__(16) unsigned char smraw[];
  T* raw = reinterpret_cast<T*>(smraw);
  float* sm = reinterpret_cast<float*>(smraw + raw_bytes<D, T>());
  float* sS = sm;                   // D rows
  float* sz = sS + D * LD;          // D
  float* sv = sz + D;               // D
  float* sq = sv + D;               // TQ rows
  float* sk = sq + TQ * LD;         // TQ rows
  float* sx = sk + TQ * LD;         // TQ rows (values)
  float* sa = sx + TQ * LD;         // TQ*TQ
  float* ss = sa + TQ * TQ;         // TQ
  const int u = blockIdx.y;
  const int i = blockIdx.x;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int mg = tid / NL, nl = tid % NL;
  const int jm = mc_index(p, u);
  const float w = mc[((size_t)jm * p.M + i) * p.M + i];
  prefetch_rows<D, TQ>(p, u, i, 0, min(TQ, p.nb), Q, K, V, raw);
  const float* mrow = mixed + ((size_t)u * p.M + i) * p.R;
  for (int e = tid; e < D * D; e += kThreads) sS[e / D * LD + e % D] = mrow[e];
  for (int e = tid; e < 2 * D; e += kThreads) sz[e] = mrow[D * D + e];
  float n_state = (float)p.nb * rowsum_lower[jm * p.M + i];   // n<_i

  for (int l0 = 0; l0 < p.nb; l0 += TQ) {
    const int cnt = min(TQ, p.nb - l0);
    cpa_wait_all();
    __syncthreads();
    for (int e = tid; e < TQ * D; e += kThreads) {
      const int tt = e / D, f = e % D;
      float qx = 0.f, kx = 0.f, vx = 0.f;
      if (tt < cnt) {
        qx = phi_apply(to_f32(raw[e]), p.fmap);
        kx = phi_apply(to_f32(raw[TQ * D + e]), p.fmap);
        vx = to_f32(raw[2 * TQ * D + e]);
      }
      sq[tt * LD + f] = qx;
      sk[tt * LD + f] = kx;
      sx[tt * LD + f] = vx;
    }
    __syncthreads();
    if (l0 + TQ < p.nb) prefetch_rows<D, TQ>(p, u, i, l0 + TQ, min(TQ, p.nb - l0 - TQ), Q, K, V, raw);
    // masked in-tile scores a[t][j] = phi(q_t) . phi(k_j), j <= t
    if (tid < TH * TH) {
      const int ti = tid / TH, ji = tid % TH;
      float c2[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
      for (int f = 0; f < D; f += 4) {
        float q0[4], q1[4], k0[4], k1[4];
        lds_vec<4>(sq + ti * LD + f, q0);
        lds_vec<4>(sq + (ti + TH) * LD + f, q1);
        lds_vec<4>(sk + ji * LD + f, k0);
        lds_vec<4>(sk + (ji + TH) * LD + f, k1);
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          c2[0][0] = fmaf(q0[x], k0[x], c2[0][0]);
          c2[0][1] = fmaf(q0[x], k1[x], c2[0][1]);
          c2[1][0] = fmaf(q1[x], k0[x], c2[1][0]);
          c2[1][1] = fmaf(q1[x], k1[x], c2[1][1]);
        }
      }
#pragma unroll
      for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          const int tt = ti + TH * a, jj = ji + TH * b;
          sa[tt * TQ + jj] = (jj <= tt && tt < cnt) ? c2[a][b] : 0.f;
        }
    }
    // phi(q_t)^T S_state, kept in registers
    float num[2][RN];
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
      for (int b = 0; b < RN; ++b) num[a][b] = 0.f;
    for (int f = 0; f < D; ++f) {
      const float x0 = sq[mg * LD + f], x1 = sq[(mg + MG) * LD + f];
      float cv[RN];
      lds_vec<RN>(sS + f * LD + RN * nl, cv);
#pragma unroll
      for (int b = 0; b < RN; ++b) {
        num[0][b] = fmaf(x0, cv[b], num[0][b]);
        num[1][b] = fmaf(x1, cv[b], num[1][b]);
      }
    }
    __syncthreads();
    // denominators s_t = phi(q_t) . z_state + w sum_{j <= t} a[t][j]
    for (int tt = warp; tt < TQ; tt += kWarps) {
      float s = 0.f;
      for (int f = lane; f < D; f += 32) s = fmaf(sq[tt * LD + f], sz[f], s);
      const float r = warp_sum(lane < TQ ? sa[tt * TQ + lane] : 0.f);
      s = warp_sum(s);
      if (lane == 0) ss[tt] = fmaf(w, r, s);
    }
    __syncthreads();
    // in-tile part sum_{j<=t} a[t][j] v_j (and sum_{j<=t} v_j), then the norm
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
        float xv[RN];
        lds_vec<RN>(sx + jj * LD + RN * nl, xv);
#pragma unroll
        for (int b = 0; b < RN; ++b) {
          lo[0][b] = fmaf(a0, xv[b], lo[0][b]);
          lo[1][b] = fmaf(a1, xv[b], lo[1][b]);
          vl[0][b] = fmaf(m0, xv[b], vl[0][b]);
          vl[1][b] = fmaf(m1, xv[b], vl[1][b]);
        }
      }
#pragma unroll
      for (int a = 0; a < 2; ++a) {
        const int tt = mg + MG * a;
        if (tt >= cnt) continue;
        const float s = ss[tt];
        const size_t base = tok_off(p, u, block_token(p, i, l0 + tt));
#pragma unroll
        for (int b = 0; b < RN; ++b) {
          const int c = RN * nl + b;
          const float nm = fmaf(w, lo[a][b], num[a][b]);
          float o = nm;
          if (p.norm == MHLA_NORM_DIVISIVE) {
            o = s != 0.f ? nm / s : 0.f;
          } else if (p.norm == MHLA_NORM_MALA) {
            const float ntil = n_state + w * (float)(tt + 1);
            const float vt = sv[c] + w * vl[a][b];
            o = s != 0.f ? (1.f + 1.f / s) * nm - (s / ntil) * vt : 0.f;
          }
          out[base + c] = from_f32<T>(o);
        }
      }
    }
    __syncthreads();
    // advance the state by the whole tile: S += w sum_j phi(k_j) v_j^T (z, v, n)
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
      for (int jj = 0; jj < cnt; ++jj) {
        float ka[4], xb[4];
        lds_vec<4>(sk + jj * LD + 4 * fi, ka);
        lds_vec<4>(sx + jj * LD + 4 * ci, xb);
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int b = 0; b < 4; ++b) st[a][b] = fmaf(ka[a], xb[b], st[a][b]);
      }
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const int e = (4 * fi + a) * LD + 4 * ci + b;
          sS[e] = fmaf(w, st[a][b], sS[e]);
        }
    }
    if (tid < D) {
      float a = 0.f;
      for (int jj = 0; jj < cnt; ++jj) a += sk[jj * LD + tid];
      sz[tid] = fmaf(w, a, sz[tid]);
    } else if (tid < 2 * D) {
      float a = 0.f;
      for (int jj = 0; jj < cnt; ++jj) a += sx[jj * LD + tid - D];
      sv[tid - D] = fmaf(w, a, sv[tid - D]);
    }
    n_state = fmaf(w, (float)cnt, n_state);
  }
}

template <int D, typename T>
int run(const Plan& p, const void* q, const void* k, const void* v, const float* mixed, const float* rl,
        const float* mc, void* out, cudaStream_t s) {
  const size_t smem = raw_bytes<D, T>() + sizeof(float) * smem_floats<D>();
  auto kern = causal_output_kernel<D, T>;
  cudaError_t e = (cudaError_t)set_max_dynamic_smem((const void*)kern, (int)smem);
  if (e != cudaSuccess) return (int)e;
  kern<<<dim3(p.M, p.BH), kThreads, smem, s>>>(p, (const T*)q, (const T*)k, (const T*)v, mixed, rl, mc, (T*)out);
  return (int)cudaGetLastError();
}

template <typename T>
int by_d(const Plan& p, const void* q, const void* k, const void* v, const float* mixed, const float* rl,
         const float* mc, void* out, cudaStream_t s) {
  switch (p.d) {
    case 16: return run<16, T>(p, q, k, v, mixed, rl, mc, out, s);
    case 32: return run<32, T>(p, q, k, v, mixed, rl, mc, out, s);
    case 64: return run<64, T>(p, q, k, v, mixed, rl, mc, out, s);
    case 128: return run<128, T>(p, q, k, v, mixed, rl, mc, out, s);
  }
  return (int)cudaErrorInvalidValue;
}

}  // namespace

int launch_mc_strict_lower(const Plan& p, const float* mc, float* mcl, void* stream) {
  const size_t n = (size_t)p.mc_heads * p.M * p.M;
  strict_lower_kernel<<<(unsigned)((n + 255) / 256), 256, 0, (cudaStream_t)stream>>>(p.mc_heads, p.M, mc, mcl);
  return (int)cudaGetLastError();
}

int launch_simt_causal_output(const Plan& p, const void* q, const void* k, const void* v, const float* mixed,
                              const float* rowsum_lower, const float* mc, void* out, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (p.dtype == MHLA_DTYPE_F32) return by_d<float>(p, q, k, v, mixed, rowsum_lower, mc, out, s);
  return by_d<__nv_bfloat16>(p, q, k, v, mixed, rowsum_lower, mc, out, s);
}

}  // namespace mhla
