// Output-step gradients on the tensor cores (head dimension 64, bf16).
//
// For query block i ("MHLA: Restoring Expressivity of Linear Attention via
// Token-Level Multi-Head", flowchart output node; "Rectifying Magnitude
// Neglect in Linear Attention", key designs, for MALA), with P = phi(Q) and
// dO the gradient of the loss with respect to the output:
//     num_t = P_t S~_i,  s_t = P_t . z~_i
//     DIVISIVE dnum = dO / s,        ds = -(dO . num) / s^2
//     NONE     dnum = dO,            ds = 0
//     MALA     dnum = beta dO,       ds = -(dO . num) / s^2 - (dO . v~_i) / n~_i
//              (beta = 1 + 1/s, gamma = s / n~_i)
//     dq_t   = (S~_i dnum_t + z~_i ds_t) * phi'(q_t)
//     dS~_i  = sum_t P_t^T dnum_t,  dz~_i = sum_t ds_t P_t
//     MALA:  dv~_i = -sum_t gamma_t dO_t,  dn~_i = sum_t (dO_t . v~_i) s_t / n~_i^2
// Per token tile (up to 128 tokens of block i, one TMA box from the grid):
//   MMA1  D1 = P [S~_i | Z]          M = 128 tokens, N = 80, K = 64
//         (Z holds z~_i as columns (hi, hi, lo): s = D1[64] + D1[66])
//   MMA2  D2 += [P | W]^T [G | G2]   M = 128 (rows 0..63 features of P,
//         rows 64.. the MALA weights W), N = 80, K = tokens; accumulated over
//         the tiles of a block piece
//   MMA3  D3 = [G | G2] [S~_i | Z]^T  M = 128 tokens, N = 64 (k), K = 64 + 16
// where G = dnum and G2 = (ds hi, ds lo, ds hi, e hi, e lo) per token with
// e_t = (dO_t . v~_i) s_t / n~_i^2, and W = (gamma/beta hi, lo, 1) per token
// (zero outside MALA): D2 rows 0..63 are dS~_i (columns 0..63) and dz~_i
// (columns 64 + 65), rows 64 + 65 give sum_t gamma_t dO_t (as
// sum_t (gamma_t / beta_t) dnum_t), D2[66][67] + D2[66][68] = sum_t e_t.
// Every operand is split into bf16 high + low parts and contracted with three
// MMAs (hi hi + hi lo + lo hi), so the records carry about 16 significant
// bits: dMc contracts them against the forward records.
// The piece's D2 becomes one gradient record (hi and lo planes, the layout
// of the forward stack: dS~ rows, then dz~, dv~), stored by TMA.
// Persistent, warp-specialised CTA (512 threads): warp 0 Q/dO producer,
// warp 1 TMEM + MMA, warp 2 block-operand producer, warp 3 Z and v~_i, warps
// 4-11 phi(Q) (two threads per row), warps 12-15 epilogues (one thread per
// token row = TMEM lane): G, G2, W from D1; dq from D3; the record from D2.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstring>

#include "common.cuh"
#include "tc_bwd.h"
#include "tc_common.cuh"

namespace mhla {
namespace {

using namespace tc;

constexpr int kThreads = 512;
constexpr int kXfThreads = 128;                 // warps 4..7
constexpr int kEpiThreads = 128;                // warps 8..11 (E1), 12..15 (dq, record)
constexpr uint32_t kTile = 128 * 128;           // 128 token rows x 64 bf16
constexpr uint32_t kBTile = 64 * 128;           // 64 rows x 64 bf16
constexpr int kStages = 2;
constexpr int kBStages = 2;
// token stage: Q -> P hi -> dq | dO -> G hi | P lo
constexpr uint32_t kStageBytes = 3 * kTile;
constexpr uint32_t kOffGlo = kStages * kStageBytes;
constexpr uint32_t kOffG2 = kOffGlo + kTile;
constexpr uint32_t kOffW = kOffG2 + kTile;
constexpr uint32_t kOffZero = kOffW + kTile;    // 16 rows of zeros
// block-operand stage: S~ hi | S~ lo | Z | misc (v~ floats, aux rows, info)
constexpr uint32_t kOffSlo = kBTile;
constexpr uint32_t kOffZ = 2 * kBTile;
constexpr uint32_t kOffMisc = 3 * kBTile;
constexpr uint32_t kOffV = kOffMisc;            // 64 floats
constexpr uint32_t kOffAux = kOffMisc + 256;    // z~, v~ rows: hi (256 B), lo (256 B)
constexpr uint32_t kOffInfo = kOffMisc + 768;   // float4 {., n~_i, ., .}
constexpr uint32_t kBStageBytes = 3 * kBTile + 1024;
constexpr uint32_t kBBase = kOffZero + 2048;
// record staging: S rows hi | S rows lo | zv rows hi | zv rows lo
constexpr uint32_t kStaging = kBBase + kBStages * kBStageBytes;
constexpr uint32_t kStagingBytes = 2 * kBTile + 2048;
constexpr uint32_t kScratch = kStaging + kStagingBytes;  // 64 floats (MALA row exchange)
constexpr uint32_t kBars = kScratch + 1024;
constexpr int kNumBars = 4 * kStages + 3 * kBStages + 6 + 4;
constexpr uint32_t kSmemBytes = kBars + 8 * kNumBars + 16 + 1024;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColD1 = 0, kColD3 = 128, kColD2 = 256;  // D2 double-buffered at 256, 384
static_assert(kSmemBytes <= 232448, "shared memory");
static_assert(kBStageBytes % 1024 == 0 && kBBase % 1024 == 0 && kStaging % 1024 == 0, "alignment");

struct BoArgs {
  CUtensorMap tmQ, tmG, tmDQ;          // 5D (64, Wg, Hg, T, BH), box (64, cw, ch, ct, 1)
  CUtensorMap tmB_hi, tmB_lo;          // 3D (64, R/64, BH*M) over the mixed planes, box (64, 64, 1)
  CUtensorMap tmS_hi, tmS_lo;          // 2D (64, BH*Q*66) over the gradient planes, box (64, 64)
  CUtensorMap tmZV_hi, tmZV_lo;        // same, box (64, 2)
  const __nv_bfloat16* mixed_hi;
  const __nv_bfloat16* mixed_lo;
  const float4* blkinfo;
  float* dnp;                          // [BH][Q] dn~ per piece (MALA)
  int R, units, splits, cpp;
  ChunkShape c;
  FastDiv f_head, f_splits;
  unsigned int* err;
};

__device__ __forceinline__ void bo_unit(const Plan& p, const BoArgs& a, int w, int& u, int& i, int& c0, int& c1) {
  const uint32_t uu = fdiv((uint32_t)w, a.f_head);
  const uint32_t rem = (uint32_t)w - uu * (uint32_t)(p.M * a.splits);
  const uint32_t ii = fdiv(rem, a.f_splits);
  const int piece = (int)(rem - ii * (uint32_t)a.splits);
  u = (int)uu;
  i = (int)ii;
  c0 = piece * a.cpp;
  c1 = min(a.c.per_block, c0 + a.cpp);
}

__device__ __forceinline__ uint32_t bf16_bits(float x) {
  return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x));
}

// hi and lo bf16 parts of x
__device__ __forceinline__ void split1(float x, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat16 h = __float2bfloat16_rn(x);
  hi = (uint32_t)__bfloat16_as_ushort(h);
  lo = bf16_bits(x - __bfloat162float(h));
}

__global__ void __launch_bounds__(kThreads, 1) tc_bwd_output_kernel(const __grid_constant__ BoArgs a, const Plan p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gb = smem_raw + (base - raw);
  const uint32_t bars = base + kBars;
  auto tfull = [&](int s) { return bars + 8u * s; };
  auto pready = [&](int s) { return bars + 8u * (kStages + s); };
  auto tempty = [&](int s) { return bars + 8u * (2 * kStages + s); };
  auto bfull = [&](int x) { return bars + 8u * (4 * kStages + x); };
  auto bready = [&](int x) { return bars + 8u * (4 * kStages + kBStages + x); };
  auto bempty = [&](int x) { return bars + 8u * (4 * kStages + 2 * kBStages + x); };
  const uint32_t b0 = bars + 8u * (4 * kStages + 3 * kBStages);
  const uint32_t d1full = b0, d1empty = b0 + 8, gready = b0 + 16, gfree = b0 + 24, d3full = b0 + 32,
                 d3empty = b0 + 40;
  auto d2full = [&](int x) { return b0 + 48 + 8u * x; };
  auto d2empty = [&](int x) { return b0 + 64 + 8u * x; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gb + kBars + 8 * kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gb + kBars + 8 * kNumBars + 8);
  auto tst = [&](int s) { return base + (uint32_t)s * kStageBytes; };
  auto bst = [&](int x) { return base + kBBase + (uint32_t)x * kBStageBytes; };

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int rows = a.c.rows;
  const int rows_pad = a.c.rows_pad;
  const bool mala = p.norm == MHLA_NORM_MALA;

  // zero: G lo, G2, W, the zero rows, every token stage (rows past a tile
  // stay finite), the Z tiles
  for (uint32_t off = threadIdx.x * 16u; off < kOffZero + 2048u; off += kThreads * 16u)
    *reinterpret_cast<uint4*>(gb + off) = make_uint4(0u, 0u, 0u, 0u);
  for (int x = 0; x < kBStages; ++x)
    for (uint32_t off = threadIdx.x * 16u; off < kBTile; off += kThreads * 16u)
      *reinterpret_cast<uint4*>(gb + kBBase + x * kBStageBytes + kOffZ + off) = make_uint4(0u, 0u, 0u, 0u);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(tfull(s), 1);
      mbar_init(pready(s), kXfThreads / 32);
      mbar_init(tempty(s), 1);
    }
    for (int x = 0; x < kBStages; ++x) {
      mbar_init(bfull(x), 1);
      mbar_init(bready(x), 1);
      mbar_init(bempty(x), 1);
    }
    mbar_init(d1full, 1);
    mbar_init(d1empty, kEpiThreads / 32);
    mbar_init(gready, kEpiThreads / 32);
    mbar_init(gfree, 1);
    mbar_init(d3full, 1);
    mbar_init(d3empty, kEpiThreads / 32);
    for (int x = 0; x < 2; ++x) {
      mbar_init(d2full(x), 1);
      mbar_init(d2empty(x), 1);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&a.tmQ);
    tma_prefetch_desc(&a.tmG);
    tma_prefetch_desc(&a.tmDQ);
  }
  if (warp == 2 && lane == 0) {
    tma_prefetch_desc(&a.tmB_hi);
    tma_prefetch_desc(&a.tmB_lo);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------- Q, dO producer
      const uint64_t pol = policy_evict_first();
      const uint32_t bytes = (uint32_t)rows * 128u;
      int s = 0;
      uint32_t ph = 0;
      long long issued = 0;
      bool ok = true;
      for (int w = blockIdx.x; w < a.units && ok; w += gridDim.x) {
        int u, i, c0, c1;
        bo_unit(p, a, w, u, i, c0, c1);
        for (int c = c0; c < c1; ++c) {
          if (!(ok = mbar_wait(tempty(s), ph ^ 1u, a.err, 0x801, abort_flag))) break;
          int x0, y0, t0;
          chunk_origin(p, a.c, (uint32_t)i, (uint32_t)c, x0, y0, t0);
          mbar_arrive_expect_tx(tfull(s), 2 * bytes);
          tma_load_5d(tst(s), &a.tmQ, tfull(s), 0, x0, y0, t0, u, pol);
          tma_load_5d(tst(s) + kTile, &a.tmG, tfull(s), 0, x0, y0, t0, u, pol);
          ++issued;
          if (++s == kStages) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      drain_loads(tfull(0), kStages, issued, a.err, 0x802);
    }
  } else if (warp == 2) {
    // ----------------------------------------- block-operand producer
    const uint64_t pol = policy_evict_last();
    int x = 0;
    uint32_t ph = 0;
    long long issued = 0;
    for (int w = blockIdx.x; w < a.units; w += gridDim.x) {
      int u, i, c0, c1;
      bo_unit(p, a, w, u, i, c0, c1);
      bool ok = true;
      if (lane == 0) ok = mbar_wait(bempty(x), ph ^ 1u, a.err, 0x803, abort_flag);
      if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
      const uint32_t st = bst(x);
      const int rec = u * p.M + i;
      const __nv_bfloat16* src = (lane < 16 ? a.mixed_hi : a.mixed_lo) + (size_t)rec * a.R + 64 * 64 + (lane & 15) * 8;
      cp_async16(st + kOffAux + (lane < 16 ? 0u : 256u) + (lane & 15) * 16, src);
      if (lane == 0) cp_async16(st + kOffInfo, a.blkinfo + i);
      cp_async_arrive(bfull(x));
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_expect_tx(bfull(x), 2 * kBTile);
        tma_load_3d(st, &a.tmB_hi, bfull(x), 0, 0, rec, pol);
        tma_load_3d(st + kOffSlo, &a.tmB_lo, bfull(x), 0, 0, rec, pol);
      }
      ++issued;
      if (++x == kBStages) {
        x = 0;
        ph ^= 1u;
      }
    }
    if (lane == 0) drain_loads(bfull(0), kBStages, issued, a.err, 0x804);
  } else if (warp == 3) {
    // ------------------------------------- Z (z~ as hi, hi, lo) and v~
    int x = 0;
    uint32_t ph = 0;
    for (int w = blockIdx.x; w < a.units; w += gridDim.x) {
      const bool ok = mbar_wait(bfull(x), ph, a.err, 0x805, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) break;
      uint8_t* st = gb + kBBase + x * kBStageBytes;
      const __nv_bfloat16* aux = reinterpret_cast<const __nv_bfloat16*>(st + kOffAux);
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int k = lane + 32 * j;
        *reinterpret_cast<__nv_bfloat16*>(st + kOffZ + sw128_offset(k, 0)) = aux[k];
        *reinterpret_cast<__nv_bfloat16*>(st + kOffZ + sw128_offset(k, 1)) = aux[k];
        *reinterpret_cast<__nv_bfloat16*>(st + kOffZ + sw128_offset(k, 2)) = aux[128 + k];
        reinterpret_cast<float*>(st + kOffV)[k] = __bfloat162float(aux[64 + k]) + __bfloat162float(aux[192 + k]);
      }
      fence_proxy_async();
      mbar_arrive_warp(bready(x));
      if (++x == kBStages) {
        x = 0;
        ph ^= 1u;
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // --------------------------------------------------------------- MMA
      const uint32_t id1 = idesc_bf16_f32(128, 80, false, true);
      const uint32_t id1s = idesc_bf16_f32(128, 64, false, true);
      const uint32_t id2 = idesc_bf16_f32(128, 80, true, true);
      const uint32_t id3 = idesc_bf16_f32(128, 64, false, false);
      const uint32_t glo = base + kOffGlo, g2 = base + kOffG2, wt = base + kOffW, zero = base + kOffZero;
      const int ksteps2 = rows_pad / 16;
      int s = 0, x = 0;
      uint32_t ph = 0, bph = 0;
      long long n = 0, m = 0;   // chunks, units
      bool ok = true;
      for (int w = blockIdx.x; w < a.units && ok; w += gridDim.x) {
        int u, i, c0, c1;
        bo_unit(p, a, w, u, i, c0, c1);
        const int d2 = (int)(m & 1);
        if (!(ok = mbar_wait(bready(x), bph, a.err, 0x806, abort_flag))) break;
        if (!(ok = mbar_wait(d2empty(d2), (uint32_t)((m >> 1) & 1) ^ 1u, a.err, 0x807, abort_flag))) break;
        const uint32_t bs = bst(x);
        const uint32_t sh = bs, sl = bs + kOffSlo, zt = bs + kOffZ;
        const uint32_t D1 = tmem + kColD1, D3 = tmem + kColD3, D2 = tmem + kColD2 + 128u * (uint32_t)d2;
        for (int c = c0; c < c1; ++c) {
          const uint32_t np = (uint32_t)(n & 1);
          if (!(ok = mbar_wait(pready(s), ph, a.err, 0x808, abort_flag))) break;
          if (!(ok = mbar_wait(d1empty, np ^ 1u, a.err, 0x809, abort_flag))) break;
          tc_fence_after();
          const uint32_t phi = tst(s), gt = phi + kTile, plo = phi + 2 * kTile;
          // MMA1: D1 = P [S~ | Z], P = P hi + P lo, S~ = hi + lo
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const uint64_t ah = sdesc_sw128(phi + (uint32_t)ks * 32u, 0u, 1024u);
            const uint64_t al = sdesc_sw128(plo + (uint32_t)ks * 32u, 0u, 1024u);
            const uint64_t bh = sdesc_sw128(sh + (uint32_t)ks * 2048u, zt - sh, 1024u);
            umma_bf16(D1, ah, bh, id1, ks > 0 ? 1u : 0u);
            umma_bf16(D1, ah, sdesc_sw128(sl + (uint32_t)ks * 2048u, 0u, 1024u), id1s, 1u);
            umma_bf16(D1, al, bh, id1, 1u);
          }
          umma_commit(d1full);
          if (!(ok = mbar_wait(gready, np, a.err, 0x80a, abort_flag))) break;
          if (!(ok = mbar_wait(d3empty, np ^ 1u, a.err, 0x80b, abort_flag))) break;
          tc_fence_after();
          // MMA2: D2 += [P | W]^T [G | G2] over the tile's tokens
          for (int kt = 0; kt < ksteps2; ++kt) {
            const uint32_t o = (uint32_t)kt * 2048u;
            const uint64_t aw = sdesc_sw128(phi + o, wt - phi, 1024u);         // P hi | W
            const uint64_t az = sdesc_sw128(plo + o, zero - (plo + o), 1024u); // P lo | 0
            const uint64_t bg = sdesc_sw128(gt + o, g2 - gt, 1024u);           // G hi | G2
            const uint64_t bz = sdesc_sw128(glo + o, zero - (glo + o), 1024u); // G lo | 0
            umma_bf16(D2, aw, bg, id2, (c > c0 || kt > 0) ? 1u : 0u);
            umma_bf16(D2, aw, bz, id2, 1u);
            umma_bf16(D2, az, bg, id2, 1u);
          }
          // MMA3: D3 = [G | G2] [S~ | Z]^T
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const uint32_t o = (uint32_t)ks * 32u;
            const uint64_t ah = sdesc_sw128(gt + o, 0u, 1024u), al = sdesc_sw128(glo + o, 0u, 1024u);
            const uint64_t bh = sdesc_sw128(sh + o, 0u, 1024u);
            umma_bf16(D3, ah, bh, id3, ks > 0 ? 1u : 0u);
            umma_bf16(D3, ah, sdesc_sw128(sl + o, 0u, 1024u), id3, 1u);
            umma_bf16(D3, al, bh, id3, 1u);
          }
          umma_bf16(D3, sdesc_sw128(g2, 0u, 1024u), sdesc_sw128(zt, 0u, 1024u), id3, 1u);
          umma_commit(gfree);
          umma_commit(d3full);
          ++n;
          if (++s == kStages) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(d2full(d2));
        umma_commit(bempty(x));
        ++m;
        if (++x == kBStages) {
          x = 0;
          bph ^= 1u;
        }
      }
    }
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------ phi(Q): P hi in place, P lo aside
    const int row = threadIdx.x - 128;
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int w = blockIdx.x; w < a.units && ok; w += gridDim.x) {
      int u, i, c0, c1;
      bo_unit(p, a, w, u, i, c0, c1);
      for (int c = c0; c < c1; ++c) {
        ok = mbar_wait(tfull(s), ph, a.err, 0x80c, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        uint8_t* rp = gb + s * kStageBytes + row * 128;
        if (row < rows) {
#pragma unroll 2
          for (int j = 0; j < 8; ++j) {
            const uint32_t off = ((j + row) & 7) << 4;
            uint4 xv = *reinterpret_cast<const uint4*>(rp + off), lo;
            uint32_t* xp = &xv.x;
            uint32_t* lp = &lo.x;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float2 f = bf16x2_to_float2(xp[q]);
              const float f0 = phi_map(f.x, p.fmap), f1 = phi_map(f.y, p.fmap);
              xp[q] = pack_bf16x2(f0, f1);
              const float2 g = bf16x2_to_float2(xp[q]);
              lp[q] = pack_bf16x2(f0 - g.x, f1 - g.y);
            }
            *reinterpret_cast<uint4*>(rp + off) = xv;
            *reinterpret_cast<uint4*>(rp + 2 * kTile + off) = lo;
          }
        } else if (row < rows_pad) {
          // padding rows of the token contraction: zero
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            *reinterpret_cast<uint4*>(rp + (j << 4)) = make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4*>(rp + 2 * kTile + (j << 4)) = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        fence_proxy_async();
        mbar_arrive_warp(pready(s));
        if (++s == kStages) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
  } else if (warp >= 8 && warp < 12) {
    // ------------------------------------------------ E1: D1 -> G, G2, W
    const int q4 = warp & 3;
    const int t = 32 * q4 + lane;       // token row = TMEM lane
    uint8_t* g2row = gb + kOffG2 + t * 128 + ((t & 7) << 4);   // logical chunk 0 of row t
    uint8_t* wrow = gb + kOffW + t * 128 + ((t & 7) << 4);
    uint8_t* glo_row = gb + kOffGlo + t * 128;
    int s = 0, x = 0;
    uint32_t ph = 0, bph = 0;
    long long n = 0;
    bool ok = true;
    for (int w = blockIdx.x; w < a.units && ok; w += gridDim.x) {
      int u, i, c0, c1;
      bo_unit(p, a, w, u, i, c0, c1);
      ok = mbar_wait(bready(x), bph, a.err, 0x80d, abort_flag);
      if (!named_all(5, kEpiThreads, ok)) {
        ok = false;
        break;
      }
      const uint8_t* bp = gb + kBBase + x * kBStageBytes;
      const float* vt = reinterpret_cast<const float*>(bp + kOffV);
      const float ntil = reinterpret_cast<const float4*>(bp + kOffInfo)->y;
      for (int c = c0; c < c1; ++c) {
        const uint32_t np = (uint32_t)(n & 1);
        uint8_t* grow = gb + s * kStageBytes + kTile + t * 128;   // dO -> G hi
        // ------------------------------------------ E1: D1 -> G, G2, W
        ok = mbar_wait(d1full, np, a.err, 0x80e, abort_flag);
        if (!named_all(5, kEpiThreads, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t ta = tmem + ((uint32_t)(32 * q4) << 16);
        float dot = 0.f, dgv = 0.f, sden;
        {
          float nm[32], zc[16];
#pragma unroll 1
          for (int h = 0; h < 2; ++h) {
            tmem_ld32(ta + kColD1 + 32u * h, nm);
            tmem_wait_ld();
            if (t < rows) {
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const uint4 gv = *reinterpret_cast<const uint4*>(grow + ((((4 * h + j) ^ t) & 7) << 4));
                const uint32_t* gp = &gv.x;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                  const float2 g = bf16x2_to_float2(gp[q]);
                  const int cc = 8 * j + 2 * q;
                  dot = fmaf(g.x, nm[cc], fmaf(g.y, nm[cc + 1], dot));
                  dgv = fmaf(g.x, vt[32 * h + cc], fmaf(g.y, vt[32 * h + cc + 1], dgv));
                }
              }
            }
          }
          tmem_ld16(ta + kColD1 + 64u, zc);
          tmem_wait_ld();
          sden = zc[0] + zc[2];
        }
        tc_fence_before();
        mbar_arrive_warp(d1empty);
        float scale = 1.f, ds = 0.f, wgt = 0.f, e = 0.f;
        if (p.norm == MHLA_NORM_DIVISIVE) {
          scale = 1.f / sden;
          ds = -dot * scale * scale;
        } else if (mala) {
          const float inv = 1.f / sden;
          scale = 1.f + inv;                       // beta
          const float gamma = sden / ntil;
          ds = -dot * inv * inv - dgv / ntil;
          wgt = gamma / scale;
          e = dgv * sden / (ntil * ntil);
        }
        // G lo, G2 and W are free once the previous tile's MMAs are done
        ok = mbar_wait(gfree, np ^ 1u, a.err, 0x80f, abort_flag);
        if (!named_all(5, kEpiThreads, ok)) {
          ok = false;
          break;
        }
        if (t < rows) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint32_t off = (uint32_t)(((j ^ t) & 7) << 4);
            uint4 gv = *reinterpret_cast<const uint4*>(grow + off), lv;
            uint32_t* gp = &gv.x;
            uint32_t* lp = &lv.x;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float2 g = bf16x2_to_float2(gp[q]);
              const float y0 = g.x * scale, y1 = g.y * scale;
              gp[q] = pack_bf16x2(y0, y1);
              const float2 hgt = bf16x2_to_float2(gp[q]);
              lp[q] = pack_bf16x2(y0 - hgt.x, y1 - hgt.y);
            }
            *reinterpret_cast<uint4*>(grow + off) = gv;
            *reinterpret_cast<uint4*>(glo_row + off) = lv;
          }
          uint32_t dh, dl, eh, el, wh, wl;
          split1(ds, dh, dl);
          split1(e, eh, el);
          split1(wgt, wh, wl);
          *reinterpret_cast<uint4*>(g2row) = make_uint4(dh | (dl << 16), dh | (eh << 16), el, 0u);
          if (mala) *reinterpret_cast<uint4*>(wrow) = make_uint4(wh | (wl << 16), 0x3F80u, 0u, 0u);
        } else if (t < rows_pad) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            *reinterpret_cast<uint4*>(grow + (j << 4)) = make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4*>(glo_row + (j << 4)) = make_uint4(0u, 0u, 0u, 0u);
          }
          *reinterpret_cast<uint4*>(g2row) = make_uint4(0u, 0u, 0u, 0u);
          *reinterpret_cast<uint4*>(wrow) = make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async();
        mbar_arrive_warp(gready);

        ++n;
        if (++s == kStages) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (++x == kBStages) {
        x = 0;
        bph ^= 1u;
      }
    }
  } else if (warp >= 12) {
    // ------------------------------------- dq from D3, records from D2
    const int q4 = warp & 3;
    const int t = 32 * q4 + lane;       // token row = TMEM lane
    const int et = threadIdx.x - 384;
    float* scratch = reinterpret_cast<float*>(gb + kScratch);
    int s = 0;
    uint32_t ph = 0;
    long long n = 0, m = 0;
    bool ok = true;
    for (int w = blockIdx.x; w < a.units && ok; w += gridDim.x) {
      int u, i, c0, c1;
      bo_unit(p, a, w, u, i, c0, c1);
      for (int c = c0; c < c1; ++c) {
        const uint32_t np = (uint32_t)(n & 1);
        uint8_t* qrow = gb + s * kStageBytes + t * 128;   // P hi -> dq
        const uint8_t* lrow = qrow + 2 * kTile;           // P lo
        const uint32_t ta = tmem + ((uint32_t)(32 * q4) << 16);
        // ------------------------------------------------- E2: D3 -> dq
        ok = mbar_wait(d3full, np, a.err, 0x810, abort_flag);
        if (!named_all(6, kEpiThreads, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
          float dq[32];
          tmem_ld32(ta + kColD3 + 32u * h, dq);
          tmem_wait_ld();
          if (t < rows) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint32_t off = (uint32_t)((((4 * h + j) ^ t) & 7) << 4);
              uint4 ph4 = *reinterpret_cast<const uint4*>(qrow + off);
              const uint4 pl4 = *reinterpret_cast<const uint4*>(lrow + off);
              uint32_t* hp = &ph4.x;
              const uint32_t* lp = &pl4.x;
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const int cc = 8 * j + 2 * q;
                float d0 = 1.f, d1 = 1.f;
                if (p.fmap == MHLA_FEATURE_ELU1) {
                  const float2 fh = bf16x2_to_float2(hp[q]), fl = bf16x2_to_float2(lp[q]);
                  d0 = fminf(fh.x + fl.x, 1.f);
                  d1 = fminf(fh.y + fl.y, 1.f);
                }
                hp[q] = pack_bf16x2(dq[cc] * d0, dq[cc + 1] * d1);
              }
              *reinterpret_cast<uint4*>(qrow + off) = ph4;
            }
          }
        }
        tc_fence_before();
        mbar_arrive_warp(d3empty);
        fence_proxy_async();
        named_sync(6, kEpiThreads);
        if (et == 0) {
          int x0, y0, t0;
          chunk_origin(p, a.c, (uint32_t)i, (uint32_t)c, x0, y0, t0);
          tma_store_5d(&a.tmDQ, tst(s), 0, x0, y0, t0, u);
          bulk_commit();
          bulk_wait_read<0>();
          mbar_arrive(tempty(s));
        }
        ++n;
        if (++s == kStages) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (!ok) break;
      // ------------------------------------- piece record from D2
      const int d2 = (int)(m & 1);
      ok = mbar_wait(d2full(d2), (uint32_t)((m >> 1) & 1), a.err, 0x811, abort_flag);
      if (!named_all(6, kEpiThreads, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint8_t* st_hi = gb + kStaging;
      uint8_t* st_lo = st_hi + kBTile;
      uint8_t* zv_hi = st_hi + 2 * kBTile;
      uint8_t* zv_lo = zv_hi + 1024;
      if (et == 0) bulk_wait_read<0>();   // the previous record's stores have read the staging
      named_sync(6, kEpiThreads);
      const uint32_t td = tmem + kColD2 + 128u * (uint32_t)d2 + ((uint32_t)(32 * q4) << 16);
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        float v[32];
        tmem_ld32(td + 32u * h, v);
        tmem_wait_ld();
        if (q4 < 2) {
          // row k = t of dS~ (columns 32h .. 32h + 31)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint4 hv, lv;
            uint32_t* hp = &hv.x;
            uint32_t* lp = &lv.x;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float y0 = v[8 * j + 2 * q], y1 = v[8 * j + 2 * q + 1];
              hp[q] = pack_bf16x2(y0, y1);
              const float2 g = bf16x2_to_float2(hp[q]);
              lp[q] = pack_bf16x2(y0 - g.x, y1 - g.y);
            }
            const uint32_t off = (uint32_t)t * 128u + ((uint32_t)(((4 * h + j) ^ t) & 7) << 4);
            *reinterpret_cast<uint4*>(st_hi + off) = hv;
            *reinterpret_cast<uint4*>(st_lo + off) = lv;
          }
        } else if (q4 == 2 && lane < 2) {
          // rows 64 and 65: sum_t (gamma/beta) dnum_t, high and low weights
#pragma unroll
          for (int k2 = 0; k2 < 32; ++k2) scratch[64 * lane + 32 * h + k2] = v[k2];
        }
      }
      float zc[16];
      tmem_ld16(td + 64u, zc);
      tmem_wait_ld();
      tc_fence_before();
      named_sync(6, kEpiThreads);
      if (et == 0) mbar_arrive(d2empty(d2));
      if (q4 < 2) {
        // dz~[k] = D2[k][64] + D2[k][65]
        uint32_t zh, zl;
        split1(zc[0] + zc[1], zh, zl);
        *reinterpret_cast<unsigned short*>(zv_hi + sw128_offset(0, t)) = (unsigned short)zh;
        *reinterpret_cast<unsigned short*>(zv_lo + sw128_offset(0, t)) = (unsigned short)zl;
      } else if (q4 == 2) {
        // dv~ = -(row 64 + row 65), two columns per lane (zero outside MALA)
        const int cc = 2 * lane;
        const float y0 = -(scratch[cc] + scratch[64 + cc]), y1 = -(scratch[cc + 1] + scratch[64 + cc + 1]);
        const uint32_t hv = pack_bf16x2(y0, y1);
        const float2 g = bf16x2_to_float2(hv);
        *reinterpret_cast<uint32_t*>(zv_hi + sw128_offset(1, cc)) = hv;
        *reinterpret_cast<uint32_t*>(zv_lo + sw128_offset(1, cc)) = pack_bf16x2(y0 - g.x, y1 - g.y);
        // row 66: dn~ of the piece = D2[66][67] + D2[66][68]
        if (lane == 2 && mala) a.dnp[w] = zc[3] + zc[4];
      }
      fence_proxy_async();
      named_sync(6, kEpiThreads);
      if (et == 0) {
        const int srow = w;   // record row: (u * M + i) * splits + piece
        tma_store_2d(&a.tmS_hi, smem_u32(st_hi), 0, srow * 66);
        tma_store_2d(&a.tmS_lo, smem_u32(st_lo), 0, srow * 66);
        tma_store_2d(&a.tmZV_hi, smem_u32(zv_hi), 0, srow * 66 + 64);
        tma_store_2d(&a.tmZV_lo, smem_u32(zv_lo), 0, srow * 66 + 64);
        bulk_commit();
      }
      ++m;
    }
    if (et == 0) bulk_wait<0>();
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

int launch_tc_bwd_output(const Plan& p, const void* q, const void* dout, const __nv_bfloat16* mixed_hi,
                         const __nv_bfloat16* mixed_lo, const float4* blkinfo, void* dq, __nv_bfloat16* dx_hi,
                         __nv_bfloat16* dx_lo, float* dnp, cudaStream_t s) {
  BoArgs a;
  memset(&a, 0, sizeof(a));
  const ChunkShape& c = p.chunk;
  const uint64_t dims5[5] = {64, (uint64_t)p.Wg, (uint64_t)p.Hg, (uint64_t)p.T, (uint64_t)p.BH};
  const uint64_t str5[4] = {128, 128ull * p.Wg, 128ull * p.Wg * p.Hg, 128ull * p.N};
  const uint32_t box5[5] = {64, (uint32_t)c.cw, (uint32_t)c.ch, (uint32_t)c.ct, 1};
  int e;
  if ((e = encode_tmap_bf16(&a.tmQ, q, 5, dims5, str5, box5)) != 0) return e;
  if ((e = encode_tmap_bf16(&a.tmG, dout, 5, dims5, str5, box5)) != 0) return e;
  if ((e = encode_tmap_bf16(&a.tmDQ, dq, 5, dims5, str5, box5)) != 0) return e;
  const uint64_t dims3[3] = {64, (uint64_t)(p.R / 64), (uint64_t)p.BH * p.M};
  const uint64_t str3[2] = {128, 2ull * p.R};
  const uint32_t box3[3] = {64, 64, 1};
  if ((e = encode_tmap_bf16(&a.tmB_hi, mixed_hi, 3, dims3, str3, box3)) != 0) return e;
  if ((e = encode_tmap_bf16(&a.tmB_lo, mixed_lo, 3, dims3, str3, box3)) != 0) return e;
  const uint64_t rec_rows = (uint64_t)p.BH * p.M * p.splits * 66ull;
  const uint64_t dims2[2] = {64, rec_rows};
  const uint64_t str2[1] = {128};
  const uint32_t boxS[2] = {64, 64}, boxZV[2] = {64, 2};
  if ((e = encode_tmap_bf16(&a.tmS_hi, dx_hi, 2, dims2, str2, boxS)) != 0) return e;
  if ((e = encode_tmap_bf16(&a.tmS_lo, dx_lo, 2, dims2, str2, boxS)) != 0) return e;
  if ((e = encode_tmap_bf16(&a.tmZV_hi, dx_hi, 2, dims2, str2, boxZV)) != 0) return e;
  if ((e = encode_tmap_bf16(&a.tmZV_lo, dx_lo, 2, dims2, str2, boxZV)) != 0) return e;
  a.mixed_hi = mixed_hi;
  a.mixed_lo = mixed_lo;
  a.blkinfo = blkinfo;
  a.dnp = dnp;
  a.R = p.R;
  a.splits = p.splits;
  a.cpp = p.cpp;
  a.units = p.BH * p.M * p.splits;
  a.f_head = make_fastdiv((uint32_t)(p.M * p.splits));
  a.f_splits = make_fastdiv((uint32_t)p.splits);
  a.c = c;
  a.err = p.err;
  cudaError_t ce =
      cudaFuncSetAttribute(tc_bwd_output_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (ce != cudaSuccess) return (int)ce;
  const int grid = a.units < num_sms() ? a.units : num_sms();
  tc_bwd_output_kernel<<<grid, kThreads, kSmemBytes, s>>>(a, p);
  return (int)cudaGetLastError();
}

}  // namespace mhla
