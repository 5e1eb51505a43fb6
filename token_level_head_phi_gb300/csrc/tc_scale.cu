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

constexpr int kWarps = 8;      // one query block (row) per warp
constexpr int kQChunk = 4096;  // record exponents staged in shared memory at a time (at most 16 KB)
// Exponents travel as unsigned 16-bit lanes with a bias: record exponents
// e + kBias, Mc exponents x + kBias (mc_word in tc_mix.cu; the word 0 is a
// zero entry).  Every sum below then stays in [0, 2^16) per lane, so plain
// 32-bit adds and masks act on both lanes (S part low, z part high) at once.
constexpr int kBias = 8192;

// fp16 bits of mantissa 2^(x + e - E - 1) for Mc word w (one part): the
// mantissa's bits under a new exponent while the result is a normal fp16
// number; below that, the subnormal with the mantissa shifted right and
// rounded to nearest even (2^-24 steps; a result that rounds up to 2^-14
// lands on the smallest normal number, as the encoding continues there).
__device__ __forceinline__ uint32_t place(uint32_t w, int e, int E) {
  if (w == 0u) return 0u;
  const int x = (int)(w >> 16) - kBias;
  const uint32_t h = w & 0xFFFFu, sign = h & 0x8000u;
  const int biased = x + e - E + 14;
  if (biased >= 1) return sign | ((uint32_t)biased << 10) | (h & 0x3FFu);
  const int sh = 1 - biased;
  if (sh > 11) return sign;
  const uint32_t m11 = (h & 0x3FFu) | 0x400u;
  uint32_t q = m11 >> sh;
  const uint32_t rem = m11 & ((1u << sh) - 1u), half = 1u << (sh - 1);
  q += (rem > half || (rem == half && (q & 1u))) ? 1u : 0u;
  return sign | q;
}

// Both parts of one entry: fp16 bits for the S copy (low half) and the z
// copy (high half).  e2 = {eS, eZ} + kBias per lane, c2 = {14 - ES, 14 - EZ}
// + 256 per lane (non-negative), so t = e2 + x + kBias + c2 holds the biased
// fp16 exponents x + e - E + 14 (at most 14) plus 2 kBias + 256 = 16640, a
// multiple of 64.  While both lie in [1, 14] the result is the mantissa bits
// with t's low six bits shifted above them; otherwise each part takes the
// exact path (a zero entry included).
__device__ __forceinline__ uint32_t place2(uint32_t w, uint32_t e2, uint32_t c2, int es, int ez) {
  const uint32_t t = e2 + __byte_perm(w, 0u, 0x3232) + c2;
  if (((t - 0x41014101u) & 0xFFF0FFF0u) == 0u)
    return (__byte_perm(w, 0u, 0x1010) & 0x83FF83FFu) | ((t << 10) & 0xFC00FC00u);
  return place(w, (int)(e2 & 0xFFFFu) - kBias, es) | (place(w, (int)(e2 >> 16) - kBias, ez) << 16);
}

// Grid (ceil(M / kWarps), slots): warp w of CTA (x, u) builds row
// i = x * kWarps + w of head u's two Mc copies and its output scale.  The
// head's record exponents pass through shared memory in chunks of kQChunk,
// packed {eS, eZ} + kBias as 16-bit lanes; each lane reads four consecutive
// Mc words and four packed exponents (16 bytes each) at a time.  For rows of
// at most kCacheQ records (kCached) a lane loads its Mc words once, while
// the exponents are being staged, and keeps them in registers for both
// passes.
constexpr int kCacheQ = 512;

template <bool kCached>
__global__ void __launch_bounds__(32 * kWarps) tc_scale_kernel(const Plan p, int Q, int Qp,
                                                               const uint32_t* __restrict__ mcw,
                                                               const int2* __restrict__ rexp,
                                                               __half* __restrict__ mcx,
                                                               float4* __restrict__ sinfo) {
  constexpr int kIters = kCached ? kCacheQ / 128 : 1;
  extern __shared__ __align__(16) uint32_t ex_s[];  // min(Qp, kQChunk) words
  // the record exponents come from the summary kernel
  pdl_wait();
  pdl_launch_dependents();
  const int lane = threadIdx.x % 32;
  const int u = blockIdx.y;
  const int i = blockIdx.x * kWarps + threadIdx.x / 32;
  const bool live = i < p.M;
  const uint4* row = reinterpret_cast<const uint4*>(mcw + ((size_t)mc_index(p, u) * p.M + (live ? i : 0)) * Qp);
  const int2* ex = rexp + (size_t)u * Q;
  auto stage = [&](int c0, int n) {
    for (int t = threadIdx.x; t < n; t += blockDim.x) {
      const int2 e = c0 + t < Q ? ex[c0 + t] : make_int2(0, 0);
      ex_s[t] = (uint32_t)(e.x + kBias) | ((uint32_t)(e.y + kBias) << 16);
    }
  };
  auto amax = [](uint32_t mx, const uint4& w4, const uint4& e4) {
    mx = __viaddmax_u16x2(e4.x, __byte_perm(w4.x, 0u, 0x3232), mx);
    mx = __viaddmax_u16x2(e4.y, __byte_perm(w4.y, 0u, 0x3232), mx);
    mx = __viaddmax_u16x2(e4.z, __byte_perm(w4.z, 0u, 0x3232), mx);
    return __viaddmax_u16x2(e4.w, __byte_perm(w4.w, 0u, 0x3232), mx);
  };
  // row exponents: the largest eS[q] + x(Mc[i][b(q)]) (and eZ) over nonzero
  // weights, as biased lanes (a zero weight adds only the record's e + kBias,
  // below every real sum)
  uint32_t mx = 0u;
  uint4 wc[kIters];
  if (kCached) {
#pragma unroll
    for (int k = 0; k < kIters; ++k)
      if (live && 4 * lane + 128 * k < Qp) wc[k] = __ldg(row + lane + 32 * k);
    stage(0, Qp);
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kIters; ++k)
      if (live && 4 * lane + 128 * k < Qp)
        mx = amax(mx, wc[k], *reinterpret_cast<const uint4*>(ex_s + 4 * lane + 128 * k));
  } else {
    for (int c0 = 0; c0 < Qp; c0 += kQChunk) {
      const int n = min(kQChunk, Qp - c0);
      __syncthreads();
      stage(c0, n);
      __syncthreads();
      if (live) {
#pragma unroll 4
        for (int q = 4 * lane; q < n; q += 128)
          mx = amax(mx, __ldg(row + (c0 + q) / 4), *reinterpret_cast<const uint4*>(ex_s + q));
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = __vimax3_u16x2(mx, __shfl_xor_sync(0xffffffffu, mx, o), 0u);
  int es = (int)(mx & 0xFFFFu) - 2 * kBias, ez = (int)(mx >> 16) - 2 * kBias;
  // an all-zero row mixes nothing: any exponent (its entries stay zero)
  if (es < -kBias / 2) es = 0;
  if (ez < -kBias / 2) ez = 0;
  const uint32_t c2 = (uint32_t)(14 - es + 256) | ((uint32_t)(14 - ez + 256) << 16);
  uint2* ds = reinterpret_cast<uint2*>(mcx + (((size_t)u * 2 + 0) * p.M + i) * Qp);
  uint2* dz = reinterpret_cast<uint2*>(mcx + (((size_t)u * 2 + 1) * p.M + i) * Qp);
  auto emit = [&](int q, const uint4& w4, const uint4& e4) {
    const uint32_t r0 = place2(w4.x, e4.x, c2, es, ez), r1 = place2(w4.y, e4.y, c2, es, ez);
    const uint32_t r2 = place2(w4.z, e4.z, c2, es, ez), r3 = place2(w4.w, e4.w, c2, es, ez);
    ds[q / 4] = make_uint2(__byte_perm(r0, r1, 0x5410), __byte_perm(r2, r3, 0x5410));
    dz[q / 4] = make_uint2(__byte_perm(r0, r1, 0x7632), __byte_perm(r2, r3, 0x7632));
  };
  if (kCached) {
#pragma unroll
    for (int k = 0; k < kIters; ++k) {
      const int q = 4 * lane + 128 * k;
      if (live && q < Qp) emit(q, wc[k], *reinterpret_cast<const uint4*>(ex_s + q));
    }
  } else {
    for (int c0 = 0; c0 < Qp; c0 += kQChunk) {
      const int n = min(kQChunk, Qp - c0);
      if (c0 > 0) {
        __syncthreads();
        stage(c0, n);
      }
      __syncthreads();
      if (live) {
#pragma unroll 4
        for (int q = 4 * lane; q < n; q += 128)
          emit(c0 + q, __ldg(row + (c0 + q) / 4), *reinterpret_cast<const uint4*>(ex_s + q));
      }
    }
  }
  if (live && lane == 0) {
    const float scale = p.norm == MHLA_NORM_DIVISIVE ? exp2f((float)(es - ez)) : exp2f((float)es);
    sinfo[(size_t)u * p.M + i] = make_float4(scale, 0.f, 0.f, 0.f);
  }
}

}  // namespace

int launch_tc_scale(const Plan& p, const TcBuffers& b, cudaStream_t s) {
  const dim3 grid((unsigned)((p.M + kWarps - 1) / kWarps), (unsigned)b.slots);
  const size_t smem = 4 * (size_t)(b.Qp < kQChunk ? b.Qp : kQChunk);
  auto kern = b.Qp <= kCacheQ ? tc_scale_kernel<true> : tc_scale_kernel<false>;
  return launch_pdl(kern, grid, dim3(32 * kWarps), smem, s, p, p.M * p.splits, b.Qp, (const uint32_t*)b.mcw,
                    (const int2*)b.rexp, b.mcx, b.sinfo);
}

}  // namespace mhla
