// Multi-Head Mixing on the tensor cores ("MHLA: Restoring Expressivity of
// Linear Attention via Token-Level Multi-Head", key design 2: the mixing is a
// single product of Mc with the stack of block summaries).
//
// Per head, with the stack X [Q][R] (one row of R = d*d + 2d values per block
// piece: S_b, z_b, v_b) and McExp [M][Q] (McExp[i][q] = Mc[i][q / splits]):
//     Mixed[i][r] = sum_q McExp[i][q] X[q][r]
// computed transposed so that the long R axis fills the 128-row MMA:
//     D[r][i] = sum_q X^T[r][q] McExp^T[q][i]
//   A = X^T  : MN-major (r contiguous), two 64-wide atoms per 128-row tile
//   B = McExp: K-major (q contiguous), N = up to 256 query blocks per tile
// so every Mc element is read once per (head, 128-row tile) and the epilogue
// writes Mixed with each warp storing 32 consecutive r of one query block.
// The MALA norm adds the low bf16 residual of X as a second A operand.
//
// Also here: the small preparation kernel that rounds Mc to bf16, expands it
// over summary pieces and sums its rows (n~_i = n_b * sum_b bf16(Mc[i,b])).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstring>

#include "common.cuh"
#include "tc_common.cuh"
#include "tc_host.h"

namespace mhla {
namespace {

using namespace tc;

constexpr int kMaxStages = 4;
constexpr int kThreads = 256;
constexpr uint32_t kAtom = 64 * 128;                // 64 q-rows x 64 r (8 KB)
constexpr uint32_t kATile = 2 * kAtom;              // 128 r
constexpr uint32_t kStageArea = 200 * 1024;         // shared memory for the stages
constexpr uint32_t kBars = kStageArea;
constexpr uint32_t kSmemBytes = kBars + 256 + 1024;
constexpr uint32_t kTmemCols = 512;                 // two accumulators of up to 256 columns

struct MixArgs {
  CUtensorMap tmA_hi, tmA_lo;  // 3D (R, Q, BH), box (64, 64, 1)
  CUtensorMap tmB_hi, tmB_lo;  // 2D (Q, M),     box (64, NT)
  __nv_bfloat16* mixed_hi;
  __nv_bfloat16* mixed_lo;
  int Q, NT, itiles, rtiles, kchunks, units;
  int use_lo_in;   // extra MMA with the low residual of the stack (MALA)
  int write_lo_s;  // write the low residual of S~ (aux rows always get one)
  int stages;      // pipeline depth (<= kMaxStages)
  uint32_t stage_bytes, off_alo, off_bhi, off_blo;
  unsigned int* err;
};

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
      mbar_init(accempty(x), 128);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&a.tmA_hi);
    tma_prefetch_desc(&a.tmB_hi);
    tma_prefetch_desc(&a.tmB_lo);
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
      const uint32_t bytes = kATile * (a.use_lo_in ? 2u : 1u) + 2u * (uint32_t)a.NT * 128u;
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
          tma_load_3d(st, &a.tmA_hi, full(stage), r0, kc * 64, u, pol_a);
          tma_load_3d(st + kAtom, &a.tmA_hi, full(stage), r0 + 64, kc * 64, u, pol_a);
          if (a.use_lo_in) {
            tma_load_3d(st + a.off_alo, &a.tmA_lo, full(stage), r0, kc * 64, u, pol_a);
            tma_load_3d(st + a.off_alo + kAtom, &a.tmA_lo, full(stage), r0 + 64, kc * 64, u, pol_a);
          }
          tma_load_2d(st + a.off_bhi, &a.tmB_hi, full(stage), kc * 64, i0, pol_b);
          tma_load_2d(st + a.off_blo, &a.tmB_lo, full(stage), kc * 64, i0, pol_b);
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
      const uint32_t idesc = idesc_bf16_f32(128, a.NT, true, false);
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
            // X_hi Mc_hi + X_hi Mc_lo (+ X_lo Mc_hi): Mc carries its low bf16
            // residual in every norm, the stack only for MALA
            const uint64_t ahi = sdesc_sw128(st + (uint32_t)ks * 2048u, kAtom, 1024u);
            const uint64_t bhi = sdesc_sw128(st + a.off_bhi + (uint32_t)ks * 32u, 0u, 1024u);
            const uint64_t blo = sdesc_sw128(st + a.off_blo + (uint32_t)ks * 32u, 0u, 1024u);
            umma_bf16(d, ahi, bhi, idesc, (kc > 0 || ks > 0) ? 1u : 0u);
            umma_bf16(d, ahi, blo, idesc, 1u);
            if (a.use_lo_in)
              umma_bf16(d, sdesc_sw128(st + a.off_alo + (uint32_t)ks * 2048u, kAtom, 1024u), bhi, idesc, 1u);
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
    const int e = warp - 4;
    int acc = 0;
    uint32_t accph = 0;
    bool ok = true;
    for (int w = blockIdx.x; w < a.units && ok; w += gridDim.x) {
      const int u = w / per_head;
      const int rem = w % per_head;
      const int r = (rem / a.itiles) * 128 + 32 * e + lane;
      const int i0 = (rem % a.itiles) * a.NT;
      const bool aux = r >= p.d * p.d;
      const bool lo = a.write_lo_s || aux;
      ok = mbar_wait(accfull(acc), accph, a.err, 0x204, abort_flag);
      if (!(ok = named_all(1, 128, ok))) break;
      tc_fence_after();
      const uint32_t taddr = tmem + (uint32_t)acc * 256u + ((uint32_t)(32 * e) << 16);
      __nv_bfloat16* dst_hi = a.mixed_hi + ((size_t)u * p.M + i0) * p.R + r;
      __nv_bfloat16* dst_lo = a.mixed_lo + ((size_t)u * p.M + i0) * p.R + r;
      for (int c0 = 0; c0 < a.NT; c0 += 32) {
        float v[32];
        tmem_ld32(taddr + (uint32_t)c0, v);
        tmem_wait_ld();
        if (r < p.R) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (i0 + c0 + j < p.M) {
              const __nv_bfloat16 h = __float2bfloat16_rn(v[j]);
              const size_t off = (size_t)(c0 + j) * p.R;
              dst_hi[off] = h;
              if (lo) dst_lo[off] = __float2bfloat16_rn(v[j] - __bfloat162float(h));
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(accempty(acc));
      if (++acc == 2) {
        acc = 0;
        accph ^= 1u;
      }
    }
  }
  __syncwarp();

  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// One warp per row i of Mc: high and low bf16 parts, expanded over pieces,
// and the row sum of hi + lo in float32.
__global__ void tc_prep_kernel(int M, int splits, int Q, int Qp, const float* __restrict__ mc,
                               __nv_bfloat16* __restrict__ mc_hi, __nv_bfloat16* __restrict__ mc_lo,
                               float* __restrict__ rowsum) {
  const int i = (blockIdx.x * blockDim.x + threadIdx.x) / 32;
  const int lane = threadIdx.x % 32;
  if (i >= M) return;
  const float* row = mc + (size_t)i * M;
  for (int q = lane; q < Qp; q += 32) {
    const float x = q < Q ? row[q / splits] : 0.f;
    const __nv_bfloat16 h = __float2bfloat16_rn(x);
    mc_hi[(size_t)i * Qp + q] = h;
    mc_lo[(size_t)i * Qp + q] = __float2bfloat16_rn(x - __bfloat162float(h));
  }
  float s = 0.f;
  for (int b = lane; b < M; b += 32) {
    const __nv_bfloat16 h = __float2bfloat16_rn(row[b]);
    s += __bfloat162float(h) + __bfloat162float(__float2bfloat16_rn(row[b] - __bfloat162float(h)));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) rowsum[i] = s;
}

}  // namespace

int launch_tc_prep(const Plan& p, const float* mc, const TcBuffers& b, cudaStream_t s) {
  const int threads = 256;
  const int blocks = (p.M * 32 + threads - 1) / threads;
  tc_prep_kernel<<<blocks, threads, 0, s>>>(p.M, p.splits, p.M * p.splits, b.Qp, mc, b.mc_exp, b.mc_exp_lo,
                                             b.rowsum);
  return (int)cudaGetLastError();
}

int launch_tc_mix(const Plan& p, const TcBuffers& b, cudaStream_t s) {
  MixArgs a;
  memset(&a, 0, sizeof(a));
  const int Q = p.M * p.splits;
  const uint64_t dimsA[3] = {(uint64_t)p.R, (uint64_t)Q, (uint64_t)p.BH};
  const uint64_t strA[2] = {2ull * p.R, 2ull * p.R * Q};
  const uint32_t boxA[3] = {64, 64, 1};
  int e;
  if ((e = encode_tmap_bf16(&a.tmA_hi, b.stack_hi, 3, dimsA, strA, boxA)) != 0) return e;
  a.use_lo_in = b.stack_lo != nullptr;
  if ((e = encode_tmap_bf16(&a.tmA_lo, a.use_lo_in ? b.stack_lo : b.stack_hi, 3, dimsA, strA, boxA)) != 0) return e;
  int NT = (p.M + 15) / 16 * 16;
  if (NT > 256) NT = 256;
  const uint64_t dimsB[2] = {(uint64_t)Q, (uint64_t)p.M};
  const uint64_t strB[1] = {2ull * b.Qp};
  const uint32_t boxB[2] = {64, (uint32_t)NT};
  if ((e = encode_tmap_bf16(&a.tmB_hi, b.mc_exp, 2, dimsB, strB, boxB)) != 0) return e;
  if ((e = encode_tmap_bf16(&a.tmB_lo, b.mc_exp_lo, 2, dimsB, strB, boxB)) != 0) return e;
  a.mixed_hi = b.mixed_hi;
  a.mixed_lo = b.mixed_lo;
  a.Q = Q;
  a.NT = NT;
  a.itiles = (p.M + NT - 1) / NT;
  a.rtiles = (p.R + 127) / 128;
  a.kchunks = (Q + 63) / 64;
  a.units = p.BH * a.rtiles * a.itiles;
  a.write_lo_s = p.norm == MHLA_NORM_MALA;
  const uint32_t btile = (uint32_t)NT * 128u;
  a.off_alo = kATile;
  a.off_bhi = kATile * (a.use_lo_in ? 2u : 1u);
  a.off_blo = a.off_bhi + btile;
  a.stage_bytes = (a.off_blo + btile + 1023u) / 1024u * 1024u;
  a.stages = (int)(kStageArea / a.stage_bytes);
  if (a.stages > kMaxStages) a.stages = kMaxStages;
  a.err = p.err;
  cudaError_t ce = cudaFuncSetAttribute(tc_mix_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (ce != cudaSuccess) return (int)ce;
  const int grid = a.units < num_sms() ? a.units : num_sms();
  tc_mix_kernel<<<grid, kThreads, kSmemBytes, s>>>(a, p);
  return (int)cudaGetLastError();
}

}  // namespace mhla
