// Per-head mixing operands of the fp16 path (DIVISIVE and NONE).
//
// The mixing ("MHLA: Restoring Expressivity of Linear Attention via
// Token-Level Multi-Head", key design 2) forms S~_i = sum_b Mc[i,b] S_b and
// z~_i = sum_b Mc[i,b] z_b.  The summary kernel stores record q of a head as
// fp16 S_q 2^-eS[q] and z_q 2^-eZ[q], each exponent taken from the record
// part's own largest entry, so a record keeps full fp16 precision whatever
// the scale of K and V.  This kernel folds those exponents into the other
// operand, one fp16 copy of Mc per head and part:
//     McS[i][q] = Mc[i][b(q)] 2^(eS[q] - ES[i]),  McZ likewise with eZ, EZ,
// where the row exponent ES[i] = max over q with Mc[i][b(q)] != 0 of
// (eS[q] + exponent of Mc[i][b(q)]) makes the row's largest entry fall in
// [0.5, 1): the mixing GEMM then yields S~_i 2^-ES[i] and z~_i 2^-EZ[i], and
// no fp16 operand or float32 accumulator leaves its range.  An entry far
// below its row's largest (more than 2^24 smaller) rounds to a subnormal or
// to zero: its term is below the fp16 rounding of the row's largest term.
// The output step multiplies back: DIVISIVE o = (phi(q)^T S~') /
// (phi(q)^T z~') 2^(ES - EZ), NONE o = (phi(q)^T S~') 2^ES; both factors go
// into the per-(head, block) record sinfo.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <climits>

#include "tc_common.cuh"
#include "tc_host.h"

namespace mhla {
namespace {

using namespace tc;

constexpr int kRowsPerCta = 8;  // one warp per query block

// Exponent x of a float m != 0 with |m| = f 2^x, f in [0.5, 1) (read from
// the exponent field; a subnormal m counts as 2^-126, an over-estimate that
// only makes its row's entries smaller).
__device__ __forceinline__ int frexp_exponent(float m) {
  return (int)((__float_as_uint(m) >> 23) & 0xFFu) - 126;
}

// Grid (ceil(M / kRowsPerCta), slots); warp w of CTA (x, u) builds row
// i = x * kRowsPerCta + w of head u's two Mc copies and its output scale.
__global__ void __launch_bounds__(32 * kRowsPerCta) tc_scale_kernel(const Plan p, int Q, int Qp, int splits,
                                                                    const float* __restrict__ mc,
                                                                    const int2* __restrict__ rexp,
                                                                    __half* __restrict__ mcx,
                                                                    float4* __restrict__ sinfo) {
  // the record exponents come from the summary kernel
  pdl_wait();
  pdl_launch_dependents();
  const int lane = threadIdx.x % 32;
  const int u = blockIdx.y;
  const int i = blockIdx.x * kRowsPerCta + threadIdx.x / 32;
  if (i >= p.M) return;
  const float* row = mc + ((size_t)mc_index(p, u) * p.M + i) * p.M;
  const int2* ex = rexp + (size_t)u * Q;
  int es = INT_MIN, ez = INT_MIN;
  for (int q = lane; q < Q; q += 32) {
    const float m = row[splits == 1 ? q : q / splits];
    if (m != 0.f) {
      const int xm = frexp_exponent(m);
      const int2 e = ex[q];
      es = max(es, e.x + xm);
      ez = max(ez, e.y + xm);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    es = max(es, __shfl_xor_sync(0xffffffffu, es, o));
    ez = max(ez, __shfl_xor_sync(0xffffffffu, ez, o));
  }
  // an all-zero row mixes nothing: any exponent (its entries stay zero)
  if (es == INT_MIN) es = 0;
  if (ez == INT_MIN) ez = 0;
  __half2* ds = reinterpret_cast<__half2*>(mcx + (((size_t)u * 2 + 0) * p.M + i) * Qp);
  __half2* dz = reinterpret_cast<__half2*>(mcx + (((size_t)u * 2 + 1) * p.M + i) * Qp);
  for (int q2 = lane; 2 * q2 < Qp; q2 += 32) {
    float s[2] = {0.f, 0.f}, z[2] = {0.f, 0.f};
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const int q = 2 * q2 + t;
      if (q < Q) {
        const float m = row[splits == 1 ? q : q / splits];
        const int2 e = ex[q];
        s[t] = ldexpf(m, e.x - es);
        z[t] = ldexpf(m, e.y - ez);
      }
    }
    ds[q2] = __floats2half2_rn(s[0], s[1]);
    dz[q2] = __floats2half2_rn(z[0], z[1]);
  }
  if (lane == 0) {
    const float scale = p.norm == MHLA_NORM_DIVISIVE ? exp2f((float)(es - ez)) : exp2f((float)es);
    sinfo[(size_t)u * p.M + i] = make_float4(scale, 0.f, 0.f, 0.f);
  }
}

}  // namespace

int launch_tc_scale(const Plan& p, const float* mc, const TcBuffers& b, cudaStream_t s) {
  const dim3 grid((unsigned)((p.M + kRowsPerCta - 1) / kRowsPerCta), (unsigned)b.slots);
  return launch_pdl(tc_scale_kernel, grid, dim3(32 * kRowsPerCta), 0, s, p, p.M * p.splits, b.Qp, p.splits, mc,
                    (const int2*)b.rexp, b.mcx, b.sinfo);
}

}  // namespace mhla
