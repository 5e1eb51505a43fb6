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
// writes.  One CTA per (block, head) walks the block in 32-token tiles: the
// tile's own causal part is a masked 32 x 32 score matrix, the part before it
// is the running state S<_i + Mc[i,i] (sum of the earlier tiles), kept in
// shared memory and advanced after each tile.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace mhla {
namespace {

constexpr int kThreads = 256;
constexpr int kTQ = 32;

// mcl = Mc with its diagonal and upper triangle zeroed, for `heads` matrices.
__global__ void strict_lower_kernel(int heads, int M, const float* __restrict__ mc, float* __restrict__ mcl) {
  const size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
  if (idx >= (size_t)heads * M * M) return;
  const int r = (int)(idx / M), b = (int)(idx % M), i = r % M;
  mcl[idx] = b < i ? mc[idx] : 0.f;
}

// Shared memory: state S (D*D), z (D), v (D) | phi(q), phi(k), v tiles
// (kTQ*D each) | scores (kTQ*kTQ) | per-token s (kTQ).
template <int D, typename T>
__global__ void __launch_bounds__(kThreads)
causal_output_kernel(Plan p, const T* __restrict__ Q, const T* __restrict__ K, const T* __restrict__ V,
                     const float* __restrict__ mixed, const float* __restrict__ rowsum_lower,
                     const float* __restrict__ mc, T* __restrict__ out) {
  extern __shared__ float sm[];
  float* sS = sm;                   // D*D
  float* sz = sS + D * D;           // D
  float* sv = sz + D;               // D
  float* sq = sv + D;               // kTQ*D
  float* sk = sq + kTQ * D;         // kTQ*D
  float* sx = sk + kTQ * D;         // kTQ*D (values)
  float* sa = sx + kTQ * D;         // kTQ*kTQ
  float* ss = sa + kTQ * kTQ;       // kTQ
  const int u = blockIdx.y;
  const int i = blockIdx.x;
  const int tid = threadIdx.x;
  const int j = mc_index(p, u);
  const float w = mc[((size_t)j * p.M + i) * p.M + i];
  const float* mrow = mixed + ((size_t)u * p.M + i) * p.R;
  for (int e = tid; e < D * D + 2 * D; e += kThreads) sm[e] = mrow[e];
  float n_state = (float)p.nb * rowsum_lower[j * p.M + i];   // n<_i

  for (int l0 = 0; l0 < p.nb; l0 += kTQ) {
    const int cnt = min(kTQ, p.nb - l0);
    __syncthreads();
    for (int e = tid; e < kTQ * D; e += kThreads) {
      const int tt = e / D, f = e % D;
      float qx = 0.f, kx = 0.f, vx = 0.f;
      if (tt < cnt) {
        const size_t off = tok_off(p, u, block_token(p, i, l0 + tt)) + f;
        qx = phi_apply(to_f32(Q[off]), p.fmap);
        kx = phi_apply(to_f32(K[off]), p.fmap);
        vx = to_f32(V[off]);
      }
      sq[e] = qx;
      sk[e] = kx;
      sx[e] = vx;
    }
    __syncthreads();
    // masked in-tile scores a[t][j] = phi(q_t) . phi(k_j), j <= t
    for (int e = tid; e < kTQ * kTQ; e += kThreads) {
      const int tt = e / kTQ, j = e % kTQ;
      float a = 0.f;
      if (j <= tt && tt < cnt) {
        for (int f = 0; f < D; ++f) a = fmaf(sq[tt * D + f], sk[j * D + f], a);
      }
      sa[e] = a;
    }
    __syncthreads();
    // denominators s_t = phi(q_t) . z_state + w sum_{j <= t} a[t][j]
    if (tid < kTQ) {
      float s = 0.f, r = 0.f;
      for (int f = 0; f < D; ++f) s = fmaf(sq[tid * D + f], sz[f], s);
      for (int j = 0; j <= tid; ++j) r += sa[tid * kTQ + j];
      ss[tid] = fmaf(w, r, s);
    }
    __syncthreads();
    for (int e = tid; e < cnt * D; e += kThreads) {
      const int tt = e / D, c = e % D;
      float num = 0.f, loc = 0.f, vloc = 0.f;
      for (int f = 0; f < D; ++f) num = fmaf(sq[tt * D + f], sS[f * D + c], num);
      for (int j = 0; j <= tt; ++j) {
        loc = fmaf(sa[tt * kTQ + j], sx[j * D + c], loc);
        vloc += sx[j * D + c];
      }
      num = fmaf(w, loc, num);
      const float s = ss[tt];
      float o = num;
      if (p.norm == MHLA_NORM_DIVISIVE) {
        o = s != 0.f ? num / s : 0.f;
      } else if (p.norm == MHLA_NORM_MALA) {
        const float ntil = n_state + w * (float)(tt + 1);
        const float vt = sv[c] + w * vloc;
        o = s != 0.f ? (1.f + 1.f / s) * num - (s / ntil) * vt : 0.f;
      }
      out[tok_off(p, u, block_token(p, i, l0 + tt)) + c] = from_f32<T>(o);
    }
    __syncthreads();
    // advance the state by the whole tile: S += w sum_j phi(k_j) v_j^T (z, v, n)
    for (int e = tid; e < D * D; e += kThreads) {
      const int f = e / D, c = e % D;
      float acc = 0.f;
      for (int j = 0; j < cnt; ++j) acc = fmaf(sk[j * D + f], sx[j * D + c], acc);
      sS[e] = fmaf(w, acc, sS[e]);
    }
    if (tid < D) {
      float a = 0.f;
      for (int j = 0; j < cnt; ++j) a += sk[j * D + tid];
      sz[tid] = fmaf(w, a, sz[tid]);
    } else if (tid < 2 * D) {
      float a = 0.f;
      for (int j = 0; j < cnt; ++j) a += sx[j * D + tid - D];
      sv[tid - D] = fmaf(w, a, sv[tid - D]);
    }
    n_state = fmaf(w, (float)cnt, n_state);
  }
}

template <int D, typename T>
int run(const Plan& p, const void* q, const void* k, const void* v, const float* mixed, const float* rl,
        const float* mc, void* out, cudaStream_t s) {
  const size_t smem = sizeof(float) * (D * D + 2 * D + 3 * kTQ * D + kTQ * kTQ + kTQ);
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
