// Multi-Head Mixing for few blocks ("MHLA: Restoring Expressivity of Linear
// Attention via Token-Level Multi-Head", key design 2) on the CUDA cores,
// between the tensor-core summary and output kernels.
//
// With M <= kSmallMixMaxM query blocks the mixing S~_i = sum_b Mc[i,b] S_b is
// a contraction over a handful of records per head: a tensor-core tile of 128
// query blocks and 64 records would be almost all padding.  Here every thread
// owns two consecutive entries r of the record, reads them once from each of
// the head's Q records and accumulates all M mixed values in registers, in
// float32:
//   fp16 records:  X[q][r] 2^eS[q] (2^eZ[q] for the z and v rows) -- the
//                  record's own power of two, so the sums carry the true
//                  scale, which bf16 (float32's range) holds;
//   split records: X_hi[q][r] + X_lo[q][r].
// The mixed summaries are written as the tensor-core mixing writes them (bf16
// high parts, low residuals where the output step reads them); for fp16
// records the output scales are 1 (sinfo), so the output step applies
// nothing more.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "tc_common.cuh"
#include "tc_host.h"

namespace mhla {
namespace {

using namespace tc;

constexpr int kThreads = 256;  // two record entries per thread: 512 per CTA

template <bool kF16>
__global__ void __launch_bounds__(kThreads) tc_mixs_kernel(const Plan p, int Q, const float* __restrict__ mc,
                                                           const void* __restrict__ stack,
                                                           const __nv_bfloat16* __restrict__ stack_lo,
                                                           const int2* __restrict__ rexp,
                                                           __nv_bfloat16* __restrict__ mixed_hi,
                                                           __nv_bfloat16* __restrict__ mixed_lo,
                                                           float4* __restrict__ sinfo, int write_lo) {
  __shared__ float w_s[kSmallMixMaxQ * kSmallMixMaxM];  // [q][i] = Mc[i][q / splits]
  __shared__ float2 sc_s[kSmallMixMaxQ];                // {2^eS[q], 2^eZ[q]} (fp16 records)
  // the records come from the summary kernel
  pdl_wait();
  pdl_launch_dependents();
  const int M = p.M, R = p.R;
  const int u = blockIdx.y;
  const float* mrow = mc + (size_t)mc_index(p, u) * M * M;
  for (int t = threadIdx.x; t < Q * M; t += kThreads) {
    const int q = t / M, i = t - q * M;
    w_s[t] = mrow[(size_t)i * M + q / p.splits];
  }
  if (kF16) {
    for (int t = threadIdx.x; t < Q; t += kThreads) {
      const int2 e = rexp[(size_t)u * Q + t];
      sc_s[t] = make_float2(exp2f((float)e.x), exp2f((float)e.y));
    }
    if (blockIdx.x == 0)
      for (int i = threadIdx.x; i < M; i += kThreads) sinfo[(size_t)u * M + i] = make_float4(1.f, 0.f, 0.f, 0.f);
  }
  __syncthreads();
  const int r = 2 * (blockIdx.x * kThreads + threadIdx.x);
  if (r >= R) return;
  const bool zpart = r >= p.d * p.d;  // rows of z_b and v_b
  float a0[kSmallMixMaxM], a1[kSmallMixMaxM];
#pragma unroll
  for (int i = 0; i < kSmallMixMaxM; ++i) a0[i] = a1[i] = 0.f;
  // unrolled so that the loads of several records are in flight together
#pragma unroll 8
  for (int q = 0; q < Q; ++q) {
    const size_t off = ((size_t)u * Q + q) * R + r;
    float x0, x1;
    if (kF16) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(static_cast<const __half*>(stack) + off));
      const float s = zpart ? sc_s[q].y : sc_s[q].x;
      x0 = f.x * s;
      x1 = f.y * s;
    } else {
      const float2 h = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(
          static_cast<const __nv_bfloat16*>(stack) + off));
      const float2 l = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(stack_lo + off));
      x0 = h.x + l.x;
      x1 = h.y + l.y;
    }
    const float* w = w_s + q * M;
#pragma unroll
    for (int i = 0; i < kSmallMixMaxM; ++i) {
      if (i < M) {
        a0[i] = fmaf(w[i], x0, a0[i]);
        a1[i] = fmaf(w[i], x1, a1[i]);
      }
    }
  }
  const bool lo = write_lo || zpart;
#pragma unroll
  for (int i = 0; i < kSmallMixMaxM; ++i) {
    if (i < M) {
      const size_t off = ((size_t)u * M + i) * R + r;
      const __nv_bfloat162 h = __floats2bfloat162_rn(a0[i], a1[i]);
      *reinterpret_cast<__nv_bfloat162*>(mixed_hi + off) = h;
      if (lo) {
        const float2 hf = __bfloat1622float2(h);
        *reinterpret_cast<__nv_bfloat162*>(mixed_lo + off) = __floats2bfloat162_rn(a0[i] - hf.x, a1[i] - hf.y);
      }
    }
  }
}

}  // namespace

bool small_mix_supported(const Plan& p) { return p.M <= kSmallMixMaxM && p.M * p.splits <= kSmallMixMaxQ; }

int launch_tc_mix_small(const Plan& p, const float* mc, const TcBuffers& b, cudaStream_t s) {
  const int Q = p.M * p.splits;
  const dim3 grid((unsigned)((p.R + 2 * kThreads - 1) / (2 * kThreads)), (unsigned)b.slots);
  const int write_lo = tc_out_lo(p) ? 1 : 0;
  if (b.f16)
    return launch_pdl(tc_mixs_kernel<true>, grid, dim3(kThreads), 0, s, p, Q, mc, (const void*)b.stack,
                      (const __nv_bfloat16*)b.stack_lo, (const int2*)b.rexp, b.mixed_hi, b.mixed_lo, b.sinfo,
                      write_lo);
  return launch_pdl(tc_mixs_kernel<false>, grid, dim3(kThreads), 0, s, p, Q, mc, (const void*)b.stack,
                    (const __nv_bfloat16*)b.stack_lo, (const int2*)b.rexp, b.mixed_hi, b.mixed_lo, b.sinfo,
                    write_lo);
}

}  // namespace mhla
