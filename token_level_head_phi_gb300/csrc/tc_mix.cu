// Multi-Head Mixing on the tensor cores ("MHLA: Restoring Expressivity of
// Linear Attention via Token-Level Multi-Head", key design 2: the mixing is a
// single product of Mc with the stack of block summaries).
//
// Per head, with a stack X [Q][W] (one row per block piece) and
// McExp [M][Q] (McExp[i][q] = Mc[i][q / splits]):
//     Mixed[i][r0 + r] = sum_q McExp[i][q] X[q][r]
// computed transposed so that the long r axis fills the 128-row MMA:
//     D[r][i] = sum_q X^T[r][q] McExp^T[q][i]
//   A = X^T  : MN-major (r contiguous), two 64-wide atoms per 128-row tile
//   B = McExp: K-major (q contiguous), N = up to 256 query blocks per tile
// Two precisions:
//   kF16  (DIVISIVE/NONE): X = fp16(x * 2^-s), B = fp16(Mc * 2^-e_i); one MMA
//         per K step; Mixed keeps the factor 2^-(s + e_i), which the output
//         step multiplies back.
//   split (MALA): X and Mc as bf16 high + low parts, D = Xh Mh + Xh Ml + Xl Mh.
// The epilogue writes Mixed as bf16 (plus the low residual where the output
// step needs it): 32 query blocks x 128 r at a time, transposed through a
// shared-memory tile and stored by TMA.  In the fp16 case Mixed holds
// S~_i / 2^(s + e_i); the output step multiplies the scale back.
//
// Also here: the small preparation kernel that builds the Mc copies.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstring>

#include "common.cuh"
#include "tc_common.cuh"
#include "tc_host.h"

namespace mhla {
namespace {

using namespace tc;

constexpr int kMaxStages = 4;
constexpr int kThreads = 384;                       // 4 control warps + 8 epilogue warps
constexpr int kEpiGroups = 2;                       // epilogue groups (column halves)
constexpr uint32_t kAtom = 64 * 128;                // 64 q-rows x 64 r (8 KB)
constexpr uint32_t kATile = 2 * kAtom;              // 128 r
constexpr uint32_t kStageArea = 192 * 1024;         // shared memory for the stages
constexpr uint32_t kStagingBytes = 2 * 32 * 256;    // per group: [32 i][128 r] bf16, hi and lo
constexpr uint32_t kStaging = kStageArea;
constexpr uint32_t kBars = kStaging + kEpiGroups * kStagingBytes;
constexpr uint32_t kSmemBytes = kBars + 256 + 1024;
constexpr uint32_t kTmemCols = 512;                 // two accumulators of up to 256 columns

struct MixArgs {
  CUtensorMap tmA, tmA_lo;     // 3D (W, Q, BH), box (64, 64, 1)
  CUtensorMap tmB, tmB_lo;     // 2D (Q, M),     box (64, NT)
  CUtensorMap tmO, tmO_lo;     // 3D (R, M, BH) view of Mixed, box (128, 32, 1), no swizzle
  int Q, NT, itiles, rtiles, kchunks, units;
  int r_off;                   // column of Mixed where this part starts
  int write_lo;                // write the low residual of every value
  int stages;
  uint32_t stage_bytes, off_alo, off_b, off_blo;
  unsigned int* err;
};

template <bool kF16>
__global__ void __launch_bounds__(kThreads, 1) tc_mix_kernel(const __grid_constant__ MixArgs a, const Plan p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gb = smem_raw + (base - raw);
  const uint32_t bars = base + kBars;
  const int kStages = a.stages;
  auto full = [&](int s) { return bars + 8u * s; };
  auto empty = [&](int s) { return bars + 8u * (kMaxStages + s); };
  auto accfull = [&](int x) { return bars + 8u * (2 * kMaxStages + x); };
  auto accempty = [&](int x) { return bars + 8u * (2 * kMaxStages + 2 + x); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gb + kBars + 8 * (2 * kMaxStages + 4));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gb + kBars + 8 * (2 * kMaxStages + 4) + 8);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(accfull(x), 1);
      mbar_init(accempty(x), 128 * kEpiGroups);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&a.tmA);
    tma_prefetch_desc(&a.tmB);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int per_head = a.rtiles * a.itiles;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------- producer
      const uint64_t pol_a = policy_evict_first();
      const uint64_t pol_b = policy_evict_last();
      const uint32_t bytes = kF16 ? kATile + (uint32_t)a.NT * 128u : 2u * kATile + 2u * (uint32_t)a.NT * 128u;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int w = blockIdx.x; w < a.units && ok; w += gridDim.x) {
        const int u = w / per_head;
        const int rem = w % per_head;
        const int r0 = (rem / a.itiles) * 128;
        const int i0 = (rem % a.itiles) * a.NT;
        for (int kc = 0; kc < a.kchunks; ++kc) {
          if (!(ok = mbar_wait(empty(stage), phase ^ 1u, a.err, 0x201, abort_flag))) break;
          const uint32_t st = base + (uint32_t)stage * a.stage_bytes;
          mbar_arrive_expect_tx(full(stage), bytes);
          tma_load_3d(st, &a.tmA, full(stage), r0, kc * 64, u, pol_a);
          tma_load_3d(st + kAtom, &a.tmA, full(stage), r0 + 64, kc * 64, u, pol_a);
          tma_load_2d(st + a.off_b, &a.tmB, full(stage), kc * 64, i0, pol_b);
          if (!kF16) {
            tma_load_3d(st + a.off_alo, &a.tmA_lo, full(stage), r0, kc * 64, u, pol_a);
            tma_load_3d(st + a.off_alo + kAtom, &a.tmA_lo, full(stage), r0 + 64, kc * 64, u, pol_a);
            tma_load_2d(st + a.off_blo, &a.tmB_lo, full(stage), kc * 64, i0, pol_b);
          }
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // --------------------------------------------------------------- MMA
      const uint32_t idesc = kF16 ? idesc_f16_f32(128, a.NT, true, false) : idesc_bf16_f32(128, a.NT, true, false);
      int stage = 0, acc = 0;
      uint32_t phase = 0, accph = 0;
      bool ok = true;
      for (int w = blockIdx.x; w < a.units && ok; w += gridDim.x) {
        if (!(ok = mbar_wait(accempty(acc), accph ^ 1u, a.err, 0x202, abort_flag))) break;
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)acc * 256u;
        for (int kc = 0; kc < a.kchunks; ++kc) {
          if (!(ok = mbar_wait(full(stage), phase, a.err, 0x203, abort_flag))) break;
          tc_fence_after();
          const uint32_t st = base + (uint32_t)stage * a.stage_bytes;
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const uint64_t ahi = sdesc_sw128(st + (uint32_t)ks * 2048u, kAtom, 1024u);
            const uint64_t bhi = sdesc_sw128(st + a.off_b + (uint32_t)ks * 32u, 0u, 1024u);
            umma_bf16(d, ahi, bhi, idesc, (kc > 0 || ks > 0) ? 1u : 0u);
            if (!kF16) {
              const uint64_t alo = sdesc_sw128(st + a.off_alo + (uint32_t)ks * 2048u, kAtom, 1024u);
              const uint64_t blo = sdesc_sw128(st + a.off_blo + (uint32_t)ks * 32u, 0u, 1024u);
              umma_bf16(d, ahi, blo, idesc, 1u);
              umma_bf16(d, alo, bhi, idesc, 1u);
            }
          }
          umma_commit(empty(stage));
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(accfull(acc));
        if (++acc == 2) {
          acc = 0;
          accph ^= 1u;
        }
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ epilogue
    // warp 4 + 4g + q: TMEM lane quarter q, query-block columns of half g.
    // Each 32-column slice goes through a [32 i][128 r] staging tile and
    // one TMA store (rows of Mixed are contiguous in r).
    const int q4 = warp & 3;
    const int g = (warp - 4) >> 2;
    const int gt = threadIdx.x - 128 - 128 * g;  // 0..127 within the group
    const int rl = 32 * q4 + lane;               // row of the 128-row tile
    uint8_t* stg = gb + kStaging + g * kStagingBytes;
    const uint32_t stg_addr = base + kStaging + g * kStagingBytes;
    const int half_nt = a.NT / 2;
    int acc = 0;
    uint32_t accph = 0;
    bool ok = true;
    for (int w = blockIdx.x; w < a.units && ok; w += gridDim.x) {
      const int u = w / per_head;
      const int rem = w % per_head;
      const int r0 = a.r_off + (rem / a.itiles) * 128;
      const int i0 = (rem % a.itiles) * a.NT;
      const bool lo = a.write_lo || r0 >= p.d * p.d;  // z~, v~ always carry their low residual
      ok = mbar_wait(accfull(acc), accph, a.err, 0x204, abort_flag);
      if (!(ok = named_all(1 + g, 128, ok))) break;
      tc_fence_after();
      const uint32_t taddr = tmem + (uint32_t)acc * 256u + ((uint32_t)(32 * q4) << 16);
      for (int c0 = g * half_nt; c0 < (g + 1) * half_nt; c0 += 32) {
        float v[32];
        tmem_ld32(taddr + (uint32_t)c0, v);
        tmem_wait_ld();
        // the previous slice's store has finished reading the staging tile
        if (gt == 0) bulk_wait_read<0>();
        named_sync(1 + g, 128);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const __nv_bfloat16 h = __float2bfloat16_rn(v[j]);
          reinterpret_cast<__nv_bfloat16*>(stg)[j * 128 + rl] = h;
          if (lo)
            reinterpret_cast<__nv_bfloat16*>(stg + 8192)[j * 128 + rl] = __float2bfloat16_rn(v[j] - __bfloat162float(h));
        }
        fence_proxy_async();
        named_sync(1 + g, 128);
        if (gt == 0) {
          tma_store_3d(&a.tmO, stg_addr, r0, i0 + c0, u);
          if (lo) tma_store_3d(&a.tmO_lo, stg_addr + 8192, r0, i0 + c0, u);
          bulk_commit();
        }
      }
      tc_fence_before();
      mbar_arrive(accempty(acc));
      if (++acc == 2) {
        acc = 0;
        accph ^= 1u;
      }
    }
    if (gt == 0) bulk_wait<0>();
  }
  __syncwarp();

  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// One warp per row i of Mc: the fp16 copy scaled by 2^-e_i (largest entry of
// the row in [0.5, 1]), the bf16 high and low parts, the row scale 2^e_i and
// the row sum of hi + lo in float32.  Columns are expanded over pieces.
__global__ void tc_prep_kernel(int M, int splits, int Q, int Qp, const float* __restrict__ mc,
                               __half* __restrict__ mc_f16, float* __restrict__ mc_scale,
                               __nv_bfloat16* __restrict__ mc_hi, __nv_bfloat16* __restrict__ mc_lo,
                               float* __restrict__ rowsum, float4* __restrict__ blkinfo, int f16,
                               float inv_stack_scale, float nb) {
  const int i = (blockIdx.x * blockDim.x + threadIdx.x) / 32;
  const int lane = threadIdx.x % 32;
  if (i >= M) return;
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
    const __nv_bfloat16 h = __float2bfloat16_rn(x);
    mc_hi[(size_t)i * Qp + q] = h;
    mc_lo[(size_t)i * Qp + q] = __float2bfloat16_rn(x - __bfloat162float(h));
    mc_f16[(size_t)i * Qp + q] = __float2half_rn(x * down);
  }
  if (lane == 0) {
    rowsum[i] = s;
    mc_scale[i] = ldexpf(1.f, ex);
    // the fp16 mixing leaves S~_i divided by 2^ex 2^s; the output step
    // multiplies it back
    blkinfo[i] = make_float4(f16 ? ldexpf(inv_stack_scale, ex) : 1.f, nb * s, 0.f, 0.f);
  }
}

template <bool kF16>
int launch_variant(const MixArgs& a, const Plan& p, cudaStream_t s) {
  cudaError_t ce = cudaFuncSetAttribute(tc_mix_kernel<kF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (ce != cudaSuccess) return (int)ce;
  const int grid = a.units < num_sms() ? a.units : num_sms();
  tc_mix_kernel<kF16><<<grid, kThreads, kSmemBytes, s>>>(a, p);
  return (int)cudaGetLastError();
}

}  // namespace

int launch_tc_prep(const Plan& p, const float* mc, const TcBuffers& b, cudaStream_t s) {
  const int threads = 256;
  const int blocks = (p.M * 32 + threads - 1) / threads;
  tc_prep_kernel<<<blocks, threads, 0, s>>>(p.M, p.splits, p.M * p.splits, b.Qp, mc, b.mc_f16, b.mc_scale, b.mc_hi,
                                             b.mc_lo, b.rowsum, b.blkinfo, b.f16 ? 1 : 0, 1.f / b.stack_scale,
                                             (float)p.nb);
  return (int)cudaGetLastError();
}

int launch_tc_mix(const Plan& p, const TcBuffers& b, cudaStream_t s) {
  MixArgs a;
  memset(&a, 0, sizeof(a));
  const int Q = p.M * p.splits;
  const bool f16 = b.f16;
  const int W = p.R;
  const void* src = b.stack;
  const void* src_lo = b.stack_lo;
  const uint64_t dimsA[3] = {(uint64_t)W, (uint64_t)Q, (uint64_t)p.BH};
  const uint64_t strA[2] = {2ull * W, 2ull * W * Q};
  const uint32_t boxA[3] = {64, 64, 1};
  int e;
  if ((e = encode_tmap(&a.tmA, src, 3, dimsA, strA, boxA, f16)) != 0) return e;
  if ((e = encode_tmap_bf16(&a.tmA_lo, src_lo ? src_lo : src, 3, dimsA, strA, boxA)) != 0) return e;
  // query-block tile: a multiple of 64 so that each epilogue group stores
  // whole 32-row boxes that never reach into the next tile
  const int nt_max = f16 ? 256 : 128;
  int NT = (p.M + 63) / 64 * 64;
  if (NT > nt_max) NT = nt_max;
  const uint64_t dimsB[2] = {(uint64_t)Q, (uint64_t)p.M};
  const uint64_t strB[1] = {2ull * b.Qp};
  const uint32_t boxB[2] = {64, (uint32_t)NT};
  if (f16) {
    if ((e = encode_tmap(&a.tmB, b.mc_f16, 2, dimsB, strB, boxB, true)) != 0) return e;
    a.tmB_lo = a.tmB;
  } else {
    if ((e = encode_tmap_bf16(&a.tmB, b.mc_hi, 2, dimsB, strB, boxB)) != 0) return e;
    if ((e = encode_tmap_bf16(&a.tmB_lo, b.mc_lo, 2, dimsB, strB, boxB)) != 0) return e;
  }
  const uint64_t dimsO[3] = {(uint64_t)p.R, (uint64_t)p.M, (uint64_t)p.BH};
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
  a.write_lo = p.norm == MHLA_NORM_MALA;
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
  return f16 ? launch_variant<true>(a, p, s) : launch_variant<false>(a, p, s);
}

}  // namespace mhla
