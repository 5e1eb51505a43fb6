// CUDA-core (SIMT) path of the MHLA forward: float32 arithmetic for every
// supported head dimension and both dtypes.  It is the path of the float32
// mode (tolerance 1e-5 against the float64 oracle, which rules out tf32 and
// bf16 tensor-core operands) and the cross-check of the tensor-core path.
//
// Three steps, one kernel each ("MHLA: Restoring Expressivity of Linear
// Attention via Token-Level Multi-Head", overall framework and key design 2):
//   summary: S_b = sum_{j in b} phi(K_j) V_j^T, z_b = sum phi(K_j), v_b = sum V_j
//   mix:     S~_i = sum_b Mc[i, b] S_b (and z~, v~) -- one GEMM over the stack
//   output:  o = phi(q)^T S~_i / phi(q)^T z~_i, or the NONE / MALA forms
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "plan.h"

namespace mhla {
namespace {

constexpr int kThreads = 256;

// RT consecutive floats of shared memory (16- or 8-byte aligned for RT = 4, 2).
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

// One CTA per (stack row = block piece, head unit).  A thread keeps RT x RT
// entries of the d x d summary, rows RT fi + a and columns RT ci + b, and
// reads each token's RT phi(k) and RT v values as one vector; the next tile's
// K and V values are loaded into registers while the current tile is
// multiplied.  z_b and v_b: each thread sums its own feature (tid % D) over
// its tokens, and the threads of a feature are summed at the end.
template <int D, typename Tin>
__global__ void __launch_bounds__(kThreads)
simt_summary_kernel(Plan p, const Tin* __restrict__ K, const Tin* __restrict__ V,
                    float* __restrict__ stack) {
  constexpr int TT = 32;
  constexpr int RT = D * D >= 16 * kThreads ? 4 : (D * D >= 4 * kThreads ? 2 : 1);
  constexpr int FQ = D / RT;
  constexpr int FT = (FQ * FQ + kThreads - 1) / kThreads;
  constexpr int PT = TT * D / kThreads;   // values of each array a thread loads per tile
  static_assert(kThreads % D == 0 && PT >= 1, "token split");
  __shared__ __align__(16) float sk[TT * D];
  __shared__ __align__(16) float sv[TT * D];
  const int u = blockIdx.y;
  const int row = blockIdx.x;
  const int b = row / p.splits;
  const int l0 = (row % p.splits) * p.split_len;
  const int l1 = min(p.nb, l0 + p.split_len);
  const int tid = threadIdx.x;

  float acc[FT][RT][RT];
#pragma unroll
  for (int x = 0; x < FT; ++x)
#pragma unroll
    for (int a = 0; a < RT; ++a)
#pragma unroll
      for (int c = 0; c < RT; ++c) acc[x][a][c] = 0.f;
  float zp = 0.f, vp = 0.f;   // feature tid % D, over this thread's tokens
  Tin rk[PT], rv[PT];
  auto fetch = [&](int lt) {
    const int cnt = min(TT, l1 - lt);
#pragma unroll
    for (int m = 0; m < PT; ++m) {
      const int e = tid + m * kThreads, tt = e / D;
      if (tt < cnt) {
        const size_t off = tok_off(p, u, block_token(p, b, lt + tt)) + e % D;
        rk[m] = K[off];
        rv[m] = V[off];
      }
    }
  };
  if (l0 < l1) fetch(l0);
  for (int lt = l0; lt < l1; lt += TT) {
    const int cnt = min(TT, l1 - lt);
    __syncthreads();
#pragma unroll
    for (int m = 0; m < PT; ++m) {
      const int e = tid + m * kThreads;
      const bool in = e / D < cnt;
      const float kx = in ? phi_apply(to_f32(rk[m]), p.fmap) : 0.f;
      const float vx = in ? to_f32(rv[m]) : 0.f;
      sk[e] = kx;
      sv[e] = vx;
      zp += kx;
      vp += vx;
    }
    __syncthreads();
    if (lt + TT < l1) fetch(lt + TT);
#pragma unroll
    for (int x = 0; x < FT; ++x) {
      const int qd = tid + kThreads * x;
      if (qd >= FQ * FQ) break;
      const int fi = qd / FQ, ci = qd % FQ;
      for (int tt = 0; tt < cnt; ++tt) {
        float ka[RT], vb[RT];
        lds_vec<RT>(sk + tt * D + RT * fi, ka);
        lds_vec<RT>(sv + tt * D + RT * ci, vb);
#pragma unroll
        for (int a = 0; a < RT; ++a)
#pragma unroll
          for (int c = 0; c < RT; ++c) acc[x][a][c] = fmaf(ka[a], vb[c], acc[x][a][c]);
      }
    }
  }
  float* out = stack + ((size_t)u * p.M * p.splits + row) * p.R;
#pragma unroll
  for (int x = 0; x < FT; ++x) {
    const int qd = tid + kThreads * x;
    if (qd >= FQ * FQ) break;
    const int fi = qd / FQ, ci = qd % FQ;
#pragma unroll
    for (int a = 0; a < RT; ++a)
#pragma unroll
      for (int c = 0; c < RT; ++c) out[(RT * fi + a) * D + RT * ci + c] = acc[x][a][c];
  }
  __syncthreads();
  sk[tid] = zp;
  sv[tid] = vp;
  __syncthreads();
  if (tid < D) {
    float z = 0.f, v = 0.f;
    for (int g = 0; g < kThreads / D; ++g) {
      z += sk[tid + D * g];
      v += sv[tid + D * g];
    }
    out[D * D + tid] = z;
    out[D * D + D + tid] = v;
  }
}

// mixed[u][i][r] = sum_row Mc[i][row / splits] * stack[u][row][r]: a plain
// tiled SGEMM, 32 query blocks x 128 stack columns per CTA.
__global__ void __launch_bounds__(kThreads)
simt_mix_kernel(Plan p, const float* __restrict__ mc, const float* __restrict__ stack,
                float* __restrict__ mixed) {
  constexpr int TI = 32, TR = 128, TQ = 16;
  __shared__ float smc[TI][TQ + 1];
  __shared__ float sst[TQ][TR];
  const int u = blockIdx.z;
  const int i0 = blockIdx.y * TI;
  const int r0 = blockIdx.x * TR;
  const int tx = threadIdx.x % 32, ty = threadIdx.x / 32;
  const int rows = p.M * p.splits;
  const float* st = stack + (size_t)u * rows * p.R;
  mc += (size_t)mc_index(p, u) * p.M * p.M;
  float acc[4][4] = {};
  for (int q0 = 0; q0 < rows; q0 += TQ) {
    __syncthreads();
    for (int e = threadIdx.x; e < TI * TQ; e += kThreads) {
      const int ii = e / TQ, qq = e % TQ;
      const int i = i0 + ii, q = q0 + qq;
      smc[ii][qq] = (i < p.M && q < rows) ? mc[(size_t)i * p.M + q / p.splits] : 0.f;
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
    const int i = i0 + ty * 4 + m;
    if (i >= p.M) continue;
    float* dst = mixed + ((size_t)u * p.M + i) * p.R;
#pragma unroll
    for (int n = 0; n < 4; ++n) {
      const int r = r0 + tx + 32 * n;
      if (r < p.R) dst[r] = acc[m][n];
    }
  }
}

// One CTA per (64-token tile of query block i, head unit).  The mixed
// summary S~_i sits in shared memory; each thread computes outputs
// (token, c) with the denominator of its token precomputed once.
template <int D, typename Tin>
__global__ void __launch_bounds__(kThreads)
simt_output_kernel(Plan p, const Tin* __restrict__ Q, const float* __restrict__ mixed,
                   const float* __restrict__ rowsum, Tin* __restrict__ out) {
  constexpr int TQ = 64;
  extern __shared__ float sm[];
  float* sS = sm;              // D*D
  float* sz = sS + D * D;      // D
  float* sv = sz + D;          // D
  float* sq = sv + D;          // TQ*D
  float* ss = sq + TQ * D;     // TQ
  const int tiles = (p.nb + TQ - 1) / TQ;
  const int u = blockIdx.y;
  const int i = blockIdx.x / tiles;
  const int l0 = (blockIdx.x % tiles) * TQ;
  const int cnt = min(TQ, p.nb - l0);
  const int tid = threadIdx.x;
  const float* mrow = mixed + ((size_t)u * p.M + i) * p.R;
  for (int e = tid; e < D * D + 2 * D; e += kThreads) sm[e] = mrow[e];
  for (int e = tid; e < TQ * D; e += kThreads) {
    const int tt = e / D, f = e % D;
    float x = 0.f;
    if (tt < cnt) x = phi_apply(to_f32(Q[tok_off(p, u, block_token(p, i, l0 + tt)) + f]), p.fmap);
    sq[e] = x;
  }
  __syncthreads();
  if (tid < cnt) {
    float s = 0.f;
#pragma unroll 8
    for (int k = 0; k < D; ++k) s = fmaf(sq[tid * D + k], sz[k], s);
    ss[tid] = s;
  }
  __syncthreads();
  const float n_mixed = (float)p.nb * rowsum[mc_index(p, u) * p.M + i];
  for (int e = tid; e < cnt * D; e += kThreads) {
    const int tt = e / D, c = e % D;
    float a = 0.f;
#pragma unroll 8
    for (int k = 0; k < D; ++k) a = fmaf(sq[tt * D + k], sS[k * D + c], a);
    float o;
    const float s = ss[tt];
    if (p.norm == MHLA_NORM_DIVISIVE) {
      o = s != 0.f ? a / s : 0.f;          // s = 0: no key mass, output 0
    } else if (p.norm == MHLA_NORM_MALA) {
      const float beta = 1.f + 1.f / s;
      const float gamma = s / n_mixed;
      o = s != 0.f ? beta * a - gamma * sv[c] : 0.f;
    } else {
      o = a;
    }
    out[tok_off(p, u, block_token(p, i, l0 + tt)) + c] = from_f32<Tin>(o);
  }
}

// Row sums of `rows` rows of length M (every row of every mixing matrix).
__global__ void mc_rowsum_kernel(int rows, int M, const float* __restrict__ mc, float* __restrict__ rowsum) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) / 32;
  const int lane = threadIdx.x % 32;
  if (warp >= rows) return;
  float s = 0.f;
  for (int b = lane; b < M; b += 32) s += mc[(size_t)warp * M + b];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) rowsum[warp] = s;
}

template <int D, typename Tin>
int summary_dispatch(const Plan& p, const void* k, const void* v, float* stack, cudaStream_t s) {
  dim3 grid(p.M * p.splits, p.BH);
  simt_summary_kernel<D, Tin><<<grid, kThreads, 0, s>>>(p, (const Tin*)k, (const Tin*)v, stack);
  return (int)cudaGetLastError();
}

template <int D, typename Tin>
int output_dispatch(const Plan& p, const void* q, const float* mixed, const float* rowsum, void* out,
                    cudaStream_t s) {
  const size_t smem = sizeof(float) * (D * D + 2 * D + 64 * D + 64);
  auto kern = simt_output_kernel<D, Tin>;
  if (smem > 48 * 1024) {
    cudaError_t e = (cudaError_t)set_max_dynamic_smem((const void*)kern, (int)smem);
    if (e != cudaSuccess) return (int)e;
  }
  const int tiles = (p.nb + 63) / 64;
  dim3 grid(p.M * tiles, p.BH);
  kern<<<grid, kThreads, smem, s>>>(p, (const Tin*)q, mixed, rowsum, (Tin*)out);
  return (int)cudaGetLastError();
}

template <typename Tin>
int summary_by_d(const Plan& p, const void* k, const void* v, float* stack, cudaStream_t s) {
  switch (p.d) {
    case 16: return summary_dispatch<16, Tin>(p, k, v, stack, s);
    case 32: return summary_dispatch<32, Tin>(p, k, v, stack, s);
    case 64: return summary_dispatch<64, Tin>(p, k, v, stack, s);
    case 128: return summary_dispatch<128, Tin>(p, k, v, stack, s);
  }
  return (int)cudaErrorInvalidValue;
}

template <typename Tin>
int output_by_d(const Plan& p, const void* q, const float* mixed, const float* rowsum, void* out,
                cudaStream_t s) {
  switch (p.d) {
    case 16: return output_dispatch<16, Tin>(p, q, mixed, rowsum, out, s);
    case 32: return output_dispatch<32, Tin>(p, q, mixed, rowsum, out, s);
    case 64: return output_dispatch<64, Tin>(p, q, mixed, rowsum, out, s);
    case 128: return output_dispatch<128, Tin>(p, q, mixed, rowsum, out, s);
  }
  return (int)cudaErrorInvalidValue;
}

}  // namespace

int launch_mc_rowsum(const Plan& p, const float* mc, float* rowsum, void* stream) {
  const int threads = 256;
  const int rows = p.M * p.mc_heads;
  const int blocks = (rows * 32 + threads - 1) / threads;
  mc_rowsum_kernel<<<blocks, threads, 0, (cudaStream_t)stream>>>(rows, p.M, mc, rowsum);
  return (int)cudaGetLastError();
}

int launch_simt_summary(const Plan& p, const void* k, const void* v, float* stack, void* stream) {
  if (p.dtype == MHLA_DTYPE_F32) return summary_by_d<float>(p, k, v, stack, (cudaStream_t)stream);
  return summary_by_d<__nv_bfloat16>(p, k, v, stack, (cudaStream_t)stream);
}

int launch_simt_mix(const Plan& p, const float* mc, const float* stack, float* mixed, void* stream) {
  dim3 grid((p.R + 127) / 128, (p.M + 31) / 32, p.BH);
  simt_mix_kernel<<<grid, kThreads, 0, (cudaStream_t)stream>>>(p, mc, stack, mixed);
  return (int)cudaGetLastError();
}

int launch_simt_output(const Plan& p, const void* q, const float* mixed, const float* rowsum,
                       void* out, void* stream) {
  if (p.dtype == MHLA_DTYPE_F32)
    return output_by_d<float>(p, q, mixed, rowsum, out, (cudaStream_t)stream);
  return output_by_d<__nv_bfloat16>(p, q, mixed, rowsum, out, (cudaStream_t)stream);
}

}  // namespace mhla
