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
//   MMA2  D2 += [P | G2]^T [G | G2]  M = 128 (rows 0..63 features of P,
//         rows 64.. the columns of G2), N = 80, K = tokens; accumulated over
//         the tiles of a block piece
//   MMA3  D3 = [G | G2] [S~_i | Z]^T  M = 128 tokens, N = 64 (k), K = 64 + 16
// where G = dnum and G2 = (ds hi, ds lo, ds hi, e hi, e lo, w hi, w lo, 1)
// per token with e_t = (dO_t . v~_i) s_t / n~_i^2 and w_t = gamma_t / beta_t
// (the last five zero outside MALA): D2 rows 0..63 are dS~_i (columns 0..63)
// and dz~_i (columns 64 + 65), rows 69 + 70 give sum_t gamma_t dO_t (as
// sum_t w_t dnum_t), D2[71][67] + D2[71][68] = sum_t e_t.
// Every operand is split into bf16 high + low parts and contracted with three
// MMAs (hi hi + hi lo + lo hi), so the records carry about 16 significant
// bits: dMc contracts them against the forward records.
// The piece's D2 becomes one gradient record (hi and lo planes, the layout
// of the forward stack: dS~ rows, then dz~, dv~), stored from registers.
// Persistent, warp-specialised CTA (640 threads): warp 0 Q/dO producer,
// warp 1 TMEM + MMA, warp 2 block-operand producer, warp 3 Z and v~_i, warps
// 4-11 phi(Q) (two threads per row), warps 12-15 G and G2 from D1, warps
// 16-19 dq from D3 and the record from D2 (one thread per token row = TMEM
// lane).  D1, G lo and G2 are double-buffered and the MMA thread issues
// whichever of "MMA2+3 of this tile" and "MMA1 of the next" is ready, so the
// epilogue of one tile overlaps the MMAs of the other.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstring>

#include "common.cuh"
#include "tc_bwd.h"
#include "tc_common.cuh"

namespace mhla {
namespace {

using namespace tc;

constexpr int kThreads = 640;
constexpr int kXfThreads = 256;                 // warps 4..11
constexpr int kEpiThreads = 128;                // warps 12..15 (G), 16..19 (dq, record)
constexpr uint32_t kTile = 128 * 128;           // 128 token rows x 64 bf16
constexpr uint32_t kBTile = 64 * 128;           // 64 rows x 64 bf16
constexpr int kStages = 2;
constexpr int kBStages = 2;
// token stage: Q -> P hi -> dq | dO -> G hi | P lo
constexpr uint32_t kStageBytes = 3 * kTile;
constexpr uint32_t kOffGlo = kStages * kStageBytes;   // two G lo tiles
constexpr uint32_t kOffG2 = kOffGlo + 2 * kTile;      // two G2 tiles
constexpr uint32_t kOffZero = kOffG2 + 2 * kTile;     // 16 rows of zeros
// block-operand stage: S~ hi | S~ lo | Z | misc (v~ floats, aux rows, info)
constexpr uint32_t kOffSlo = kBTile;
constexpr uint32_t kOffZ = 2 * kBTile;
constexpr uint32_t kOffMisc = 3 * kBTile;
constexpr uint32_t kOffV = kOffMisc;            // 64 floats
constexpr uint32_t kOffAux = kOffMisc + 256;    // z~, v~ rows: hi (256 B), lo (256 B)
constexpr uint32_t kOffInfo = kOffMisc + 768;   // float4 {., n~_i, ., .}
constexpr uint32_t kBStageBytes = 3 * kBTile + 1024;
constexpr uint32_t kBBase = kOffZero + 2048;
constexpr uint32_t kScratch = kBBase + kBStages * kBStageBytes;  // 192 floats
constexpr uint32_t kBars = kScratch + 1024;
constexpr int kNumBars = 3 * kStages + 3 * kBStages + 13;  // + d1full[2], d1empty[2], gfree[2], gready, d3full, d3empty, d2full[2], d2empty[2]
constexpr uint32_t kSmemBytes = kBars + 8 * kNumBars + 16 + 1024;
constexpr uint32_t kTmemCols = 512;
// accumulators: D1 (80 columns, two), D3 (64), D2 (80, two)
__device__ __forceinline__ uint32_t col_d1(int x) { return x ? 96u : 0u; }
constexpr uint32_t kColD3 = 192;
__device__ __forceinline__ uint32_t col_d2(int x) { return x ? 384u : 256u; }
static_assert(kSmemBytes <= 232448, "shared memory");
static_assert(kBStageBytes % 1024 == 0 && kBBase % 1024 == 0, "alignment");

struct BoArgs {
  CUtensorMap tmQ, tmG, tmDQ;          // 5D (64, Wg, Hg, T, BH), box (64, cw, ch, ct, 1)
  CUtensorMap tmB_hi, tmB_lo;          // 3D (64, R/64, BH*M) over the mixed planes, box (64, 64, 1)
  const __nv_bfloat16* mixed_hi;
  const __nv_bfloat16* mixed_lo;
  const float4* blkinfo;
  __nv_bfloat16* dx_hi;                // gradient records [BH][Q][R]
  __nv_bfloat16* dx_lo;
  float* dnp;                          // [BH][Q] dn~ per piece (MALA)
  int R, units, splits, cpp;
  ChunkShape c;
  FastDiv f_head, f_splits;
  unsigned int* err;
};

// Walks this CTA's token tiles in order: unit w (head, block, piece) and
// tile c of the piece; n counts tiles, m units.
struct TileIt {
  int w, c, c0, c1, u, i;
  long long n, m;
  bool valid;
  __device__ bool first() const { return valid && c == c0; }
  __device__ bool last() const { return c == c1 - 1; }
};

__device__ __forceinline__ void it_load(const Plan& p, const BoArgs& a, TileIt& it) {
  it.valid = it.w < a.units;
  if (!it.valid) return;
  const uint32_t uu = fdiv((uint32_t)it.w, a.f_head);
  const uint32_t rem = (uint32_t)it.w - uu * (uint32_t)(p.M * a.splits);
  const uint32_t ii = fdiv(rem, a.f_splits);
  const int piece = (int)(rem - ii * (uint32_t)a.splits);
  it.u = (int)uu;
  it.i = (int)ii;
  it.c0 = piece * a.cpp;
  it.c1 = min(a.c.per_block, it.c0 + a.cpp);
  it.c = it.c0;
}

__device__ __forceinline__ void it_begin(const Plan& p, const BoArgs& a, TileIt& it) {
  it.w = blockIdx.x;
  it.n = 0;
  it.m = 0;
  it_load(p, a, it);
}

__device__ __forceinline__ void it_next(const Plan& p, const BoArgs& a, TileIt& it) {
  ++it.n;
  if (++it.c < it.c1) return;
  it.w += gridDim.x;
  ++it.m;
  it_load(p, a, it);
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
  auto bfull = [&](int x) { return bars + 8u * (3 * kStages + x); };
  auto bready = [&](int x) { return bars + 8u * (3 * kStages + kBStages + x); };
  auto bempty = [&](int x) { return bars + 8u * (3 * kStages + 2 * kBStages + x); };
  const uint32_t b0 = bars + 8u * (3 * kStages + 3 * kBStages);
  auto d1full = [&](int x) { return b0 + 8u * x; };           // 2
  auto d1empty = [&](int x) { return b0 + 16 + 8u * x; };     // 2
  auto gfree = [&](int x) { return b0 + 32 + 8u * x; };       // 2
  const uint32_t gready = b0 + 48, d3full = b0 + 56, d3empty = b0 + 64;
  auto d2full = [&](int x) { return b0 + 72 + 8u * x; };      // 2 (+ d2empty below)
  auto d2empty = [&](int x) { return b0 + 88 + 8u * x; };
  static_assert(8 * (3 * kStages + 3 * kBStages) + 104 == 8 * kNumBars, "barrier slots");
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gb + kBars + 8 * kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gb + kBars + 8 * kNumBars + 8);
  auto tst = [&](int s) { return base + (uint32_t)s * kStageBytes; };
  auto bst = [&](int x) { return base + kBBase + (uint32_t)x * kBStageBytes; };

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int rows = a.c.rows;
  const int rows_pad = a.c.rows_pad;
  const bool mala = p.norm == MHLA_NORM_MALA;

  // zero: token stages (rows past a tile stay finite), G lo, G2, the zero
  // rows, the Z tiles
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
    for (int x = 0; x < 2; ++x) {
      mbar_init(d1full(x), 1);
      mbar_init(d1empty(x), kEpiThreads / 32);
      mbar_init(gfree(x), 1);
      mbar_init(d2full(x), 1);
      mbar_init(d2empty(x), 1);
    }
    mbar_init(gready, kEpiThreads / 32);
    mbar_init(d3full, 1);
    mbar_init(d3empty, kEpiThreads / 32);
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
      TileIt it;
      long long issued = 0;
      for (it_begin(p, a, it); it.valid; it_next(p, a, it)) {
        const int s = (int)(it.n % kStages);
        const uint32_t par = (uint32_t)((it.n / kStages) & 1);
        if (!mbar_wait(tempty(s), par ^ 1u, a.err, 0x801, abort_flag)) break;
        int x0, y0, t0;
        chunk_origin(p, a.c, (uint32_t)it.i, (uint32_t)it.c, x0, y0, t0);
        const TileCoords g5 = token_tile_coords(p, it.u, x0, y0, t0);
        mbar_arrive_expect_tx(tfull(s), 2 * bytes);
        tma_load_5d(tst(s), &a.tmQ, tfull(s), g5.c[0], g5.c[1], g5.c[2], g5.c[3], g5.c[4], pol);
        tma_load_5d(tst(s) + kTile, &a.tmG, tfull(s), g5.c[0], g5.c[1], g5.c[2], g5.c[3], g5.c[4], pol);
        ++issued;
      }
      drain_loads(tfull(0), kStages, issued, a.err, 0x802);
    }
  } else if (warp == 2) {
    // ----------------------------------------- block-operand producer
    const uint64_t pol = policy_evict_last();
    long long issued = 0;
    TileIt it;
    for (it_begin(p, a, it); it.valid; it_next(p, a, it)) {
      if (!it.first()) continue;
      const int x = (int)(it.m % kBStages);
      const uint32_t par = (uint32_t)((it.m / kBStages) & 1);
      bool ok = true;
      if (lane == 0) ok = mbar_wait(bempty(x), par ^ 1u, a.err, 0x803, abort_flag);
      if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
      const uint32_t st = bst(x);
      const int rec = it.u * p.M + it.i;
      const __nv_bfloat16* src = (lane < 16 ? a.mixed_hi : a.mixed_lo) + (size_t)rec * a.R + 64 * 64 + (lane & 15) * 8;
      cp_async16(st + kOffAux + (lane < 16 ? 0u : 256u) + (lane & 15) * 16, src);
      if (lane == 0) cp_async16(st + kOffInfo, a.blkinfo + mc_index(p, it.u) * p.M + it.i);
      cp_async_arrive(bfull(x));
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_expect_tx(bfull(x), 2 * kBTile);
        tma_load_3d(st, &a.tmB_hi, bfull(x), 0, 0, rec, pol);
        tma_load_3d(st + kOffSlo, &a.tmB_lo, bfull(x), 0, 0, rec, pol);
      }
      ++issued;
    }
    if (lane == 0) drain_loads(bfull(0), kBStages, issued, a.err, 0x804);
  } else if (warp == 3) {
    // ------------------------------------- Z (z~ as hi, hi, lo) and v~
    TileIt it;
    for (it_begin(p, a, it); it.valid; it_next(p, a, it)) {
      if (!it.first()) continue;
      const int x = (int)(it.m % kBStages);
      const bool ok = mbar_wait(bfull(x), (uint32_t)((it.m / kBStages) & 1), a.err, 0x805, abort_flag);
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
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // --------------------------------------------------------------- MMA
      const uint32_t id1 = idesc_bf16_f32(128, 80, false, true);
      const uint32_t id1s = idesc_bf16_f32(128, 64, false, true);
      const uint32_t id2 = idesc_bf16_f32(128, 80, true, true);
      const uint32_t id3 = idesc_bf16_f32(128, 64, false, false);
      const uint32_t zero = base + kOffZero;
      const int ksteps2 = rows_pad / 16;
      // Descriptors are formed once per group and advanced by adding to their
      // fields (address: byte offset / 16; for operands whose second atom is
      // the zero tile, the leading offset shrinks as the address grows): the
      // issue of each MMA waits for the tensor pipe, so every instruction on
      // this thread adds to the tile's time.
      const uint64_t e_step = 128ull - (128ull << 16);
      // MMA1 of a tile: D1 = P [S~ | Z]
      auto mma1 = [&](const TileIt& it) -> bool {
        const int s = (int)(it.n % kStages), x = (int)(it.m % kBStages), d = (int)(it.n & 1);
        if (it.c == it.c0 && !mbar_wait(bready(x), (uint32_t)((it.m / kBStages) & 1), a.err, 0x806, abort_flag))
          return false;
        if (!mbar_wait(pready(s), (uint32_t)((it.n / kStages) & 1), a.err, 0x808, abort_flag)) return false;
        if (!mbar_wait(d1empty(d), (uint32_t)((it.n >> 1) & 1) ^ 1u, a.err, 0x809, abort_flag)) return false;
        tc_fence_after();
        const uint32_t phi = tst(s), plo = phi + 2 * kTile;
        const uint32_t sh = bst(x), sl = sh + kOffSlo, zt = sh + kOffZ;
        const uint32_t D1 = tmem + col_d1(d);
        const uint64_t ah0 = sdesc_sw128(phi, 0u, 1024u), al0 = sdesc_sw128(plo, 0u, 1024u);
        const uint64_t bh0 = sdesc_sw128(sh, zt - sh, 1024u), bl0 = sdesc_sw128(sl, 0u, 1024u);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint64_t ah = ah0 + 2 * ks, bh = bh0 + 128 * ks;  // + 32 / + 2048 bytes per K step
          umma_bf16(D1, ah, bh, id1, ks > 0 ? 1u : 0u);
          umma_bf16(D1, ah, bl0 + 128 * ks, id1s, 1u);
          umma_bf16(D1, al0 + 2 * ks, bh, id1, 1u);
        }
        umma_commit(d1full(d));
        return true;
      };
      // MMA2 and MMA3 of a tile
      auto mma23 = [&](const TileIt& it) -> bool {
        const int s = (int)(it.n % kStages), x = (int)(it.m % kBStages), g = (int)(it.n & 1);
        const int d2 = (int)(it.m & 1);
        if (it.c == it.c0 &&
            !mbar_wait(d2empty(d2), (uint32_t)((it.m >> 1) & 1) ^ 1u, a.err, 0x807, abort_flag))
          return false;
        if (!mbar_wait(gready, (uint32_t)(it.n & 1), a.err, 0x80a, abort_flag)) return false;
        if (!mbar_wait(d3empty, (uint32_t)(it.n & 1) ^ 1u, a.err, 0x80b, abort_flag)) return false;
        tc_fence_after();
        const uint32_t phi = tst(s), gt = phi + kTile, plo = phi + 2 * kTile;
        const uint32_t glo = base + kOffGlo + (uint32_t)g * kTile, g2 = base + kOffG2 + (uint32_t)g * kTile;
        const uint32_t sh = bst(x), sl = sh + kOffSlo, zt = sh + kOffZ;
        const uint32_t D2 = tmem + col_d2(d2), D3 = tmem + kColD3;
        uint64_t aw = sdesc_sw128(phi, g2 - phi, 1024u);    // P hi | G2
        uint64_t az = sdesc_sw128(plo, zero - plo, 1024u);  // P lo | 0
        uint64_t bg = sdesc_sw128(gt, g2 - gt, 1024u);      // G hi | G2
        uint64_t bz = sdesc_sw128(glo, zero - glo, 1024u);  // G lo | 0
        for (int kt = 0; kt < ksteps2; ++kt) {
          umma_bf16(D2, aw, bg, id2, (it.c > it.c0 || kt > 0) ? 1u : 0u);
          umma_bf16(D2, aw, bz, id2, 1u);
          umma_bf16(D2, az, bg, id2, 1u);
          aw += 128;  // + 2048 bytes; the leading offset to G2 stays
          bg += 128;
          az += e_step;
          bz += e_step;
        }
        const uint64_t gh0 = sdesc_sw128(gt, 0u, 1024u), gl0 = sdesc_sw128(glo, 0u, 1024u);
        const uint64_t sh0 = sdesc_sw128(sh, 0u, 1024u), sl0 = sdesc_sw128(sl, 0u, 1024u);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint64_t ah = gh0 + 2 * ks, bh = sh0 + 2 * ks;  // + 32 bytes per K step
          umma_bf16(D3, ah, bh, id3, ks > 0 ? 1u : 0u);
          umma_bf16(D3, ah, sl0 + 2 * ks, id3, 1u);
          umma_bf16(D3, gl0 + 2 * ks, bh, id3, 1u);
        }
        umma_bf16(D3, sdesc_sw128(g2, 0u, 1024u), sdesc_sw128(zt, 0u, 1024u), id3, 1u);
        umma_commit(gfree(g));
        umma_commit(d3full);
        if (it.last()) {
          umma_commit(d2full(d2));
          umma_commit(bempty(x));
        }
        return true;
      };
      // whether a tile's MMA1 / MMA2+3 could be issued now (no waiting)
      auto ready1 = [&](const TileIt& it) -> bool {
        const int s = (int)(it.n % kStages), x = (int)(it.m % kBStages), d = (int)(it.n & 1);
        if (it.c == it.c0 && !mbar_try_wait(bready(x), (uint32_t)((it.m / kBStages) & 1))) return false;
        return mbar_try_wait(pready(s), (uint32_t)((it.n / kStages) & 1)) &&
               mbar_try_wait(d1empty(d), (uint32_t)((it.n >> 1) & 1) ^ 1u);
      };
      auto ready23 = [&](const TileIt& it) -> bool {
        const int d2 = (int)(it.m & 1);
        if (it.c == it.c0 && !mbar_try_wait(d2empty(d2), (uint32_t)((it.m >> 1) & 1) ^ 1u)) return false;
        return mbar_try_wait(gready, (uint32_t)(it.n & 1)) && mbar_try_wait(d3empty, (uint32_t)(it.n & 1) ^ 1u);
      };
      // issue whichever is ready: MMA2+3 of the current tile first (the
      // epilogues wait on it), else MMA1 of the next tile (at most one ahead)
      TileIt cur, ahead;
      it_begin(p, a, cur);
      it_begin(p, a, ahead);
      bool ok = true;
      unsigned long long t_last = globaltimer();
      while (ok && cur.valid) {
        if (ahead.n > cur.n && ready23(cur)) {
          ok = mma23(cur);
          it_next(p, a, cur);
          t_last = globaltimer();
        } else if (ahead.valid && ahead.n <= cur.n + 1 && ready1(ahead)) {
          ok = mma1(ahead);
          it_next(p, a, ahead);
          t_last = globaltimer();
        } else {
          if (*abort_flag) break;
          if (globaltimer() - t_last > kWaitLimitNs) {
            report_timeout(a.err, 0x812);
            *abort_flag = 1;
            break;
          }
          __nanosleep(32);
        }
      }
    }
  } else if (warp >= 4 && warp < 12) {
    // ------------------------------------ phi(Q): P hi in place, P lo aside
    const int t = threadIdx.x - 128;
    const int row = t >> 1;
    const int half = t & 1;
    TileIt it;
    for (it_begin(p, a, it); it.valid; it_next(p, a, it)) {
      const int s = (int)(it.n % kStages);
      const bool ok = mbar_wait(tfull(s), (uint32_t)((it.n / kStages) & 1), a.err, 0x80c, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) break;
      uint8_t* rp = gb + s * kStageBytes + row * 128;
      if (row < rows) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t off = ((4 * half + j + row) & 7) << 4;
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
        for (int j = 0; j < 4; ++j) {
          const uint32_t off = (uint32_t)(4 * half + j) << 4;
          *reinterpret_cast<uint4*>(rp + off) = make_uint4(0u, 0u, 0u, 0u);
          *reinterpret_cast<uint4*>(rp + 2 * kTile + off) = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      fence_proxy_async();
      mbar_arrive_warp(pready(s));
    }
  } else if (warp >= 12 && warp < 16) {
    // --------------------------------------------------- D1 -> G, G2
    const int q4 = warp & 3;
    const int t = 32 * q4 + lane;       // token row = TMEM lane
    const uint32_t ta = tmem + ((uint32_t)(32 * q4) << 16);
    const float* vt = nullptr;
    float ntil = 1.f;
    TileIt it;
    for (it_begin(p, a, it); it.valid; it_next(p, a, it)) {
      const int s = (int)(it.n % kStages), d = (int)(it.n & 1), g = d;
      if (it.c == it.c0) {
        const int x = (int)(it.m % kBStages);
        const bool ok = mbar_wait(bready(x), (uint32_t)((it.m / kBStages) & 1), a.err, 0x80d, abort_flag);
        if (!named_all(5, kEpiThreads, ok)) break;
        const uint8_t* bp = gb + kBBase + x * kBStageBytes;
        vt = reinterpret_cast<const float*>(bp + kOffV);
        ntil = reinterpret_cast<const float4*>(bp + kOffInfo)->y;
      }
      uint8_t* grow = gb + s * kStageBytes + kTile + t * 128;   // dO -> G hi
      uint8_t* glo_row = gb + kOffGlo + g * kTile + t * 128;
      uint8_t* g2row = gb + kOffG2 + g * kTile + t * 128 + ((t & 7) << 4);   // logical chunk 0
      bool ok = mbar_wait(d1full(d), (uint32_t)((it.n >> 1) & 1), a.err, 0x80e, abort_flag);
      if (!named_all(5, kEpiThreads, ok)) break;
      tc_fence_after();
      float dot = 0.f, dgv = 0.f, sden;
      {
        float nm[32], zc[16];
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
          tmem_ld32(ta + col_d1(d) + 32u * h, nm);
          tmem_wait_ld();
          if (t < rows) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint4 gv = *reinterpret_cast<const uint4*>(grow + ((((4 * h + j) ^ t) & 7) << 4));
              const uint32_t* gp = &gv.x;
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const float2 gg = bf16x2_to_float2(gp[q]);
                const int cc = 8 * j + 2 * q;
                dot = fmaf(gg.x, nm[cc], fmaf(gg.y, nm[cc + 1], dot));
                dgv = fmaf(gg.x, vt[32 * h + cc], fmaf(gg.y, vt[32 * h + cc + 1], dgv));
              }
            }
          }
        }
        tmem_ld16(ta + col_d1(d) + 64u, zc);
        tmem_wait_ld();
        sden = zc[0] + zc[2];
      }
      tc_fence_before();
      mbar_arrive_warp(d1empty(d));
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
      if (p.norm != MHLA_NORM_NONE && sden == 0.f) {
        // no key mass: the output is constant 0 and passes no gradient
        scale = ds = wgt = e = 0.f;
      }
      // this G lo / G2 buffer is free once the MMAs of tile n - 2 are done
      ok = mbar_wait(gfree(g), (uint32_t)((it.n >> 1) & 1) ^ 1u, a.err, 0x80f, abort_flag);
      if (!named_all(5, kEpiThreads, ok)) break;
      if (t < rows) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t off = (uint32_t)(((j ^ t) & 7) << 4);
          uint4 gv = *reinterpret_cast<const uint4*>(grow + off), lv;
          uint32_t* gp = &gv.x;
          uint32_t* lp = &lv.x;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float2 gg = bf16x2_to_float2(gp[q]);
            const float y0 = gg.x * scale, y1 = gg.y * scale;
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
        *reinterpret_cast<uint4*>(g2row) =
            make_uint4(dh | (dl << 16), dh | (eh << 16), el | (wh << 16), wl | (mala ? 0x3F800000u : 0u));
      } else if (t < rows_pad) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          *reinterpret_cast<uint4*>(grow + (j << 4)) = make_uint4(0u, 0u, 0u, 0u);
          *reinterpret_cast<uint4*>(glo_row + (j << 4)) = make_uint4(0u, 0u, 0u, 0u);
        }
        *reinterpret_cast<uint4*>(g2row) = make_uint4(0u, 0u, 0u, 0u);
      }
      fence_proxy_async();
      mbar_arrive_warp(gready);
    }
  } else if (warp >= 16) {
    // ------------------------------------- dq from D3, records from D2
    const int q4 = warp & 3;
    const int t = 32 * q4 + lane;       // token row = TMEM lane
    const int et = threadIdx.x - 512;
    const uint32_t ta = tmem + ((uint32_t)(32 * q4) << 16);
    float* scratch = reinterpret_cast<float*>(gb + kScratch);
    TileIt it;
    for (it_begin(p, a, it); it.valid; it_next(p, a, it)) {
      const int s = (int)(it.n % kStages);
      uint8_t* qrow = gb + s * kStageBytes + t * 128;   // P hi -> dq
      const uint8_t* lrow = qrow + 2 * kTile;           // P lo
      bool ok = mbar_wait(d3full, (uint32_t)(it.n & 1), a.err, 0x810, abort_flag);
      if (!named_all(6, kEpiThreads, ok)) break;
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
              const float2 fh = bf16x2_to_float2(hp[q]), fl = bf16x2_to_float2(lp[q]);
              const float d0 = phi_deriv_from_phi(fh.x, fl.x, p.fmap);
              const float d1 = phi_deriv_from_phi(fh.y, fl.y, p.fmap);
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
        chunk_origin(p, a.c, (uint32_t)it.i, (uint32_t)it.c, x0, y0, t0);
        const TileCoords g5 = token_tile_coords(p, it.u, x0, y0, t0);
        tma_store_5d(&a.tmDQ, tst(s), g5.c[0], g5.c[1], g5.c[2], g5.c[3], g5.c[4]);
        bulk_commit();
        bulk_wait_read<0>();
        mbar_arrive(tempty(s));
      }
      if (!it.last()) continue;
      // ------------------------------------- piece record from D2
      const int d2 = (int)(it.m & 1);
      ok = mbar_wait(d2full(d2), (uint32_t)((it.m >> 1) & 1), a.err, 0x811, abort_flag);
      if (!named_all(6, kEpiThreads, ok)) break;
      tc_fence_after();
      const size_t rec = (size_t)it.w * a.R;   // record of the piece: (u * M + i) * splits + piece
      const uint32_t td = ta + col_d2(d2);
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        float v[32];
        tmem_ld32(td + 32u * h, v);
        tmem_wait_ld();
        if (q4 < 2) {
          // row k = t of dS~ (columns 32h .. 32h + 31), straight to the planes
          uint4* dh4 = reinterpret_cast<uint4*>(a.dx_hi + rec + (size_t)t * 64 + 32 * h);
          uint4* dl4 = reinterpret_cast<uint4*>(a.dx_lo + rec + (size_t)t * 64 + 32 * h);
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
            dh4[j] = hv;
            dl4[j] = lv;
          }
        } else if (q4 == 2 && (lane == 5 || lane == 6)) {
          // rows 69 and 70: sum_t w_t dnum_t with the high and low weights
#pragma unroll
          for (int k2 = 0; k2 < 32; ++k2) scratch[64 + 64 * (lane - 5) + 32 * h + k2] = v[k2];
        }
      }
      float zc[16];
      tmem_ld16(td + 64u, zc);
      tmem_wait_ld();
      if (q4 < 2) scratch[t] = zc[0] + zc[1];           // dz~[k]
      if (q4 == 2 && lane == 7 && mala) a.dnp[it.w] = zc[3] + zc[4];   // row 71: dn~ of the piece
      tc_fence_before();
      named_sync(6, kEpiThreads);
      if (et == 0) mbar_arrive(d2empty(d2));
      if (q4 == 2) {
        // rows 64 (dz~) and 65 (dv~ = -(row 69 + row 70)) of the record
        const int cc = 2 * lane;
        const float z0 = scratch[cc], z1 = scratch[cc + 1];
        const float y0 = -(scratch[64 + cc] + scratch[128 + cc]), y1 = -(scratch[64 + cc + 1] + scratch[128 + cc + 1]);
        const uint32_t zh = pack_bf16x2(z0, z1), yh = pack_bf16x2(y0, y1);
        const float2 zg = bf16x2_to_float2(zh), yg = bf16x2_to_float2(yh);
        uint32_t* rh = reinterpret_cast<uint32_t*>(a.dx_hi + rec + 64 * 64);
        uint32_t* rl = reinterpret_cast<uint32_t*>(a.dx_lo + rec + 64 * 64);
        rh[lane] = zh;
        rl[lane] = pack_bf16x2(z0 - zg.x, z1 - zg.y);
        rh[32 + lane] = yh;
        rl[32 + lane] = pack_bf16x2(y0 - yg.x, y1 - yg.y);
      }
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
  int e;
  if ((e = encode_token_map(&a.tmQ, p, q, c)) != 0) return e;
  if ((e = encode_token_map(&a.tmG, p, dout, c)) != 0) return e;
  if ((e = encode_token_map(&a.tmDQ, p, dq, c)) != 0) return e;
  const uint64_t dims3[3] = {64, (uint64_t)(p.R / 64), (uint64_t)p.BH * p.M};
  const uint64_t str3[2] = {128, 2ull * p.R};
  const uint32_t box3[3] = {64, 64, 1};
  if ((e = encode_tmap_bf16(&a.tmB_hi, mixed_hi, 3, dims3, str3, box3)) != 0) return e;
  if ((e = encode_tmap_bf16(&a.tmB_lo, mixed_lo, 3, dims3, str3, box3)) != 0) return e;
  a.mixed_hi = mixed_hi;
  a.mixed_lo = mixed_lo;
  a.blkinfo = blkinfo;
  a.dx_hi = dx_hi;
  a.dx_lo = dx_lo;
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
      (cudaError_t)set_max_dynamic_smem((const void*)tc_bwd_output_kernel, (int)kSmemBytes);
  if (ce != cudaSuccess) return (int)ce;
  const int grid = a.units < num_sms() ? a.units : num_sms();
  tc_bwd_output_kernel<<<grid, kThreads, kSmemBytes, s>>>(a, p);
  return (int)cudaGetLastError();
}

}  // namespace mhla
