// Standalone launches of the mixing kernel (body in tc_mix.cuh) and of the
// small preparation kernel that builds the Mc copies.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstring>

#include "tc_mix.cuh"
#include "tc_mixt.cuh"

namespace mhla {
namespace {

using namespace tc;
using mx::MixArgs;
using mx::kAtom;
using mx::kATile;
using mx::kMaxStages;
using mx::kSmemBytes;
using mx::kStageArea;
using mx::kThreads;

// One entry of Mc as the fp16 path's exponent-folding kernel reads it: the
// fp16 bits of the mantissa 2f in [1, 2) of |m| = f 2^x, f in [0.5, 1), with
// m's sign (a mantissa that rounds up to 2 becomes 1 with x + 1), and above
// them x + 8192 as an unsigned 16-bit field, so that m = mantissa 2^(x - 1)
// up to the fp16 rounding of the mantissa; a zero entry is the word 0.  (The
// bias keeps every exponent sum the folding kernel forms positive and inside
// its 16-bit lane.)
__device__ __forceinline__ uint32_t mc_word(float m) {
  if (m == 0.f) return 0u;
  int x = 0;
  const float f = frexpf(fabsf(m), &x);
  uint32_t h = __half_as_ushort(__float2half_rn(2.f * f));
  if (h == 0x4000u) {  // 2.0
    h = 0x3C00u;       // 1.0
    ++x;
  }
  if (m < 0.f) h |= 0x8000u;
  return h | ((uint32_t)(x + 8192) << 16);
}

// Also zeroes the progress counters of a fused launch.
// One warp per row i of Mc.  Split path: the bf16 high and low parts (and an
// fp16 copy scaled by 2^-e_i, largest entry of the row in [0.5, 1]), the row
// scale 2^e_i, the row sum of hi + lo in float32 and the block record
// {1, n~_i} of the output step.  fp16 path: the mantissa-and-exponent words
// mcw instead of the copies.  Columns are expanded over pieces.  `rows` rows
// of length M: every row of every mixing matrix (one per head when each head
// has its own).
__global__ void tc_prep_kernel(int rows, int M, int splits, int Q, int Qp, const float* __restrict__ mc,
                               __half* __restrict__ mc_f16, float* __restrict__ mc_scale,
                               __nv_bfloat16* __restrict__ mc_hi, __nv_bfloat16* __restrict__ mc_lo,
                               uint32_t* __restrict__ mcw, float* __restrict__ rowsum,
                               float4* __restrict__ blkinfo, float nb, unsigned int* __restrict__ flow, int nflow) {
  // the previous call's kernels may still read what this one writes
  pdl_wait();
  pdl_launch_dependents();
  // the progress counters of a fused launch start at zero
  for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < nflow; t += gridDim.x * blockDim.x) flow[t] = 0u;
  const int i = (blockIdx.x * blockDim.x + threadIdx.x) / 32;
  const int lane = threadIdx.x % 32;
  if (i >= rows) return;
  const float* row = mc + (size_t)i * M;
  float s = 0.f, amax = 0.f;
  for (int b = lane; b < M; b += 32) {
    const __nv_bfloat16 h = __float2bfloat16_rn(row[b]);
    s += __bfloat162float(h) + __bfloat162float(__float2bfloat16_rn(row[b] - __bfloat162float(h)));
    amax = fmaxf(amax, fabsf(row[b]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    s += __shfl_xor_sync(0xffffffffu, s, o);
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  }
  int ex = 0;
  if (amax > 0.f && amax <= 3.0e38f) frexpf(amax, &ex);  // amax = f * 2^ex, f in [0.5, 1)
  const float down = ldexpf(1.f, -ex);
  for (int q = lane; q < Qp; q += 32) {
    const float x = q < Q ? row[q / splits] : 0.f;
    if (mcw) {
      mcw[(size_t)i * Qp + q] = mc_word(x);
      continue;
    }
    const __nv_bfloat16 h = __float2bfloat16_rn(x);
    mc_hi[(size_t)i * Qp + q] = h;
    mc_lo[(size_t)i * Qp + q] = __float2bfloat16_rn(x - __bfloat162float(h));
    mc_f16[(size_t)i * Qp + q] = __float2half_rn(x * down);
  }
  if (lane == 0) {
    rowsum[i] = s;
    mc_scale[i] = ldexpf(1.f, ex);
    blkinfo[i] = make_float4(1.f, nb * s, 0.f, 0.f);
  }
}

template <bool kF16>
__global__ void __launch_bounds__(mx::kThreads, 1) tc_mix_kernel(const __grid_constant__ mx::MixArgs a, const Plan p) {
  FlowCtl f = {};
  f.cta = blockIdx.x;
  f.ncta = gridDim.x;
  mx::mix_body<kF16>(a, p, f);
}

template <bool kF16>
int launch_variant(const MixArgs& a, const Plan& p, cudaStream_t s) {
  cudaError_t ce = (cudaError_t)set_max_dynamic_smem((const void*)tc_mix_kernel<kF16>, (int)kSmemBytes);
  if (ce != cudaSuccess) return (int)ce;
  const int grid = a.units < num_sms() ? a.units : num_sms();
  return launch_pdl(tc_mix_kernel<kF16>, dim3(grid), dim3(kThreads), kSmemBytes, s, a, p);
}

__global__ void __launch_bounds__(mt::kThreads, 1) tc_mixt_kernel(const __grid_constant__ mt::MixTArgs a, const Plan p) {
  mt::mixt_body(a, p);
}

int launch_mixt(const mt::MixTArgs& a, const Plan& p, cudaStream_t s) {
  auto kern = tc_mixt_kernel;
  cudaError_t ce = (cudaError_t)set_max_dynamic_smem((const void*)kern, (int)mt::kSmemBytes);
  if (ce != cudaSuccess) return (int)ce;
  int grid = a.itiles * a.items;
  if (grid > num_sms()) grid = num_sms();
  return launch_pdl(kern, dim3(grid), dim3(mt::kThreads), mt::kSmemBytes, s, a, p);
}

}  // namespace

bool mixt_supported(const Plan& p, const TcBuffers& b) {
  const int Q = p.M * p.splits;
  const int kchunks = (Q + 63) / 64;
  // The head's two fp16 Mc copies plus two 128-column accumulators fit the
  // 512 TMEM columns.  Taken for one query-block tile (M <= 128): then every
  // stack tile is read once, as in the streaming kernel, and Mc stays off
  // shared memory (measured: 1D 32k 29 -> 23 us, 14x14 x 192 heads 60 -> 40
  // us).  With more tiles each stack tile would be read once per 128 query
  // blocks instead of once per 256 (video: 66 -> 89 us); the split precision
  // of MALA measured the same in both kernels and stays on the streaming one.
  return b.f16 && p.R % 128 == 0 && 2 * kchunks * 32 <= 256 && p.M <= 128;
}

int build_mixt_args(const Plan& p, const TcBuffers& b, mt::MixTArgs* out) {
  mt::MixTArgs& a = *out;
  memset(&a, 0, sizeof(a));
  const int Q = p.M * p.splits;
  const int W = p.R;
  const uint64_t dimsX[4] = {64, (uint64_t)Q, (uint64_t)(W / 64), (uint64_t)b.slots};
  const uint64_t strX[3] = {2ull * W, 128, 2ull * W * Q};
  const uint32_t boxX[4] = {64, 64, 2, 1};
  int e;
  if ((e = encode_tmap(&a.tmX, b.stack, 4, dimsX, strX, boxX, true)) != 0) return e;
  const uint64_t dimsO[3] = {(uint64_t)p.R, (uint64_t)p.M, (uint64_t)b.slots};
  const uint64_t strO[2] = {2ull * p.R, 2ull * p.R * p.M};
  const uint32_t boxO[3] = {64, 128, 1};
  if ((e = encode_tmap_bf16(&a.tmO, b.mixed_hi, 3, dimsO, strO, boxO)) != 0) return e;
  if ((e = encode_tmap_bf16(&a.tmO_lo, b.mixed_lo, 3, dimsO, strO, boxO)) != 0) return e;
  a.mcx = b.mcx;
  a.Q = Q;
  a.Qp = b.Qp;
  a.kchunks = (Q + 63) / 64;
  a.itiles = (p.M + 127) / 128;
  a.rtiles = W / 128;
  a.items = b.slots * a.rtiles;
  a.stage_bytes = mt::kBTile;
  a.stages = (int)(mt::kStageArea / a.stage_bytes);
  if (a.stages > mt::kMaxStages) a.stages = mt::kMaxStages;
  a.err = p.err;
  return 0;
}

int launch_tc_prep(const Plan& p, const float* mc, const TcBuffers& b, cudaStream_t s) {
  const int threads = 256;
  const int rows = p.M * p.mc_heads;
  const int blocks = (rows * 32 + threads - 1) / threads;
  return launch_pdl(tc_prep_kernel, dim3(blocks), dim3(threads), 0, s, rows, p.M, p.splits, p.M * p.splits, b.Qp, mc,
                    b.mc_f16, b.mc_scale, b.mc_hi, b.mc_lo, b.f16 ? b.mcw : nullptr, b.rowsum, b.blkinfo,
                    (float)p.nb, b.flow, b.flow ? 3 * p.BH : 0);
}

int build_mix_args(const Plan& p, const TcBuffers& b, int slots, mx::MixArgs* out) {
  MixArgs& a = *out;
  memset(&a, 0, sizeof(a));
  const int Q = p.M * p.splits;
  const bool f16 = b.f16;
  const int W = p.R;
  const void* src = b.stack;
  const void* src_lo = b.stack_lo;
  // A tile of the stack: 64 pieces (q) x 128 record entries (r) as two
  // 64-wide atoms, one box: dimensions (r within atom, q, atom, slot), so
  // the box lands as [atom][q][64 r]
  const uint64_t dimsA[4] = {64, (uint64_t)Q, (uint64_t)(W / 64), (uint64_t)slots};
  const uint64_t strA[3] = {2ull * W, 128, 2ull * W * Q};
  const uint32_t boxA[4] = {64, 64, 2, 1};
  int e;
  if ((e = encode_tmap(&a.tmA, src, 4, dimsA, strA, boxA, f16)) != 0) return e;
  if ((e = encode_tmap_bf16(&a.tmA_lo, src_lo ? src_lo : src, 4, dimsA, strA, boxA)) != 0) return e;
  // query-block tile: a multiple of 64 so that each epilogue group stores
  // whole 32-row boxes that never reach into the next tile
  const int nt_max = f16 ? 256 : 128;
  int NT = (p.M + 63) / 64 * 64;
  if (NT > nt_max) NT = nt_max;
  const uint64_t dimsB[2] = {(uint64_t)Q, (uint64_t)p.M * (f16 ? 2 * slots : p.mc_heads)};
  const uint64_t strB[1] = {2ull * b.Qp};
  const uint32_t boxB[2] = {64, (uint32_t)NT};
  if (f16) {
    // the per-head copies with the record exponents folded in
    if ((e = encode_tmap(&a.tmB, b.mcx, 2, dimsB, strB, boxB, true)) != 0) return e;
    a.tmB_lo = a.tmB;
    a.b_per_slot = 1;
  } else {
    if ((e = encode_tmap_bf16(&a.tmB, b.mc_hi, 2, dimsB, strB, boxB)) != 0) return e;
    if ((e = encode_tmap_bf16(&a.tmB_lo, b.mc_lo, 2, dimsB, strB, boxB)) != 0) return e;
  }
  const uint64_t dimsO[3] = {(uint64_t)p.R, (uint64_t)p.M, (uint64_t)slots};
  const uint64_t strO[2] = {2ull * p.R, 2ull * p.R * p.M};
  const uint32_t boxO[3] = {128, 32, 1};
  if ((e = encode_tmap_plain(&a.tmO, b.mixed_hi, 3, dimsO, strO, boxO)) != 0) return e;
  if ((e = encode_tmap_plain(&a.tmO_lo, b.mixed_lo, 3, dimsO, strO, boxO)) != 0) return e;
  a.Q = Q;
  a.NT = NT;
  a.itiles = (p.M + NT - 1) / NT;
  a.rtiles = W / 128;
  a.kchunks = (Q + 63) / 64;
  a.units = p.BH * a.rtiles * a.itiles;
  a.r_off = 0;
  a.write_lo = tc_out_lo(p);
  const uint32_t btile = (uint32_t)NT * 128u;
  if (f16) {
    a.off_b = kATile;
    a.stage_bytes = (kATile + btile + 1023u) / 1024u * 1024u;
  } else {
    a.off_alo = kATile;
    a.off_b = 2 * kATile;
    a.off_blo = a.off_b + btile;
    a.stage_bytes = (a.off_blo + btile + 1023u) / 1024u * 1024u;
  }
  a.stages = (int)(kStageArea / a.stage_bytes);
  if (a.stages > kMaxStages) a.stages = kMaxStages;
  a.err = p.err;
  return 0;
}

int launch_tc_mix(const Plan& p, const TcBuffers& b, cudaStream_t s) {
  if (mixt_supported(p, b)) {
    mt::MixTArgs t;
    int e = build_mixt_args(p, b, &t);
    if (e != 0) return e;
    return launch_mixt(t, p, s);
  }
  MixArgs a;
  int e = build_mix_args(p, b, b.slots, &a);
  if (e != 0) return e;
  return b.f16 ? launch_variant<true>(a, p, s) : launch_variant<false>(a, p, s);
}

}  // namespace mhla
