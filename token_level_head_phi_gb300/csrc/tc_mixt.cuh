// Multi-Head Mixing with Mc held in tensor memory ("MHLA: Restoring
// Expressivity of Linear Attention via Token-Level Multi-Head", key design 2:
// the mixing is one product of Mc with the stack of block summaries).
//
// Per head, with the fp16 record stack X [Q][W] (one row per block piece)
// and the head's two fp16 Mc copies McS, McZ [M][Q] (Mc[i][q / splits] with
// the records' exponents folded in, built by the scale kernel):
//     Mixed[i][r] = sum_q Mc{S,Z}[i][q] X[q][r]
// computed as D[i][r] with M = 128 query blocks and N = 128 record entries:
//   A = the head's Mc copies, rows i0..i0+127, in TENSOR MEMORY (lane = query
//       block, column c holds entries 2c, 2c+1 of q; McS then McZ), loaded by
//       tcgen05.st when the CTA starts a head -- a CTA takes a contiguous run
//       of (head, r-tile) items, so it reloads once per head it touches;
//   B = X^T tile: MN-major (r contiguous), two 64-wide atoms, one 4D TMA box
//       per 64-deep K step: the only operand traffic through shared memory.
// Shared memory moves half as many bytes per FLOP as a kernel streaming both
// operands, which is what bounds the mixing GEMM.  The epilogue reads rows
// i of D, i.e. rows of the mixed summaries, and stores them without a
// transposition (swizzled staging, TMA store).
// Needs M <= 128 and Q <= 256 so that both copies and two 128-column
// accumulators fit the 512 TMEM columns.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "tc_common.cuh"
#include "tc_host.h"

namespace mhla {
namespace mt {

using namespace tc;

constexpr int kThreads = 384;                        // warps 0-3 control, 4-11 epilogue
constexpr int kMaxStages = 12;
constexpr uint32_t kAtom = 64 * 128;                 // 64 q-rows x 64 r (8 KB)
constexpr uint32_t kBTile = 2 * kAtom;               // 128 r x 64 q
constexpr uint32_t kStageArea = 160 * 1024;
constexpr uint32_t kStagingPart = 128 * 128;         // [128 i][64 r] bf16
constexpr uint32_t kStagingGroup = 2 * kStagingPart; // hi and lo
constexpr uint32_t kStaging = kStageArea;
constexpr uint32_t kBars = kStaging + 2 * kStagingGroup;
constexpr uint32_t kSmemBytes = kBars + 256 + 1024;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCol = 256;                    // accumulators at columns 256 and 384
static_assert(kSmemBytes <= 232448, "shared memory");

struct MixTArgs {
  CUtensorMap tmX;             // stack: 4D (64, Q, W / 64, slots), box (64, 64, 2, 1)
  CUtensorMap tmO, tmO_lo;     // mixed: 3D (R, M, slots), box (64, 128, 1), 128-byte swizzle
  const __half* mcx;           // [slots][2][M][Qp] the heads' fp16 Mc copies (S part, z part)
  int Q, Qp, kchunks, itiles, rtiles, items;  // items: (head, r-tile) pairs per query-block tile
  int stages;
  uint32_t stage_bytes;        // B tile
  unsigned int* err;
};

// Contiguous range [j0, j1) of the items of this CTA's query-block tile.
__device__ __forceinline__ void mixt_items(const MixTArgs& a, int& it, int& j0, int& j1) {
  it = (int)blockIdx.x % a.itiles;
  const int first = (int)blockIdx.x / a.itiles;
  const int ncta = ((int)gridDim.x - it + a.itiles - 1) / a.itiles;  // CTAs on this tile
  j0 = (int)((long long)first * a.items / ncta);
  j1 = (int)((long long)(first + 1) * a.items / ncta);
}

// The kernel body; `a` must live in kernel parameter space.
__device__ __forceinline__ void mixt_body(const MixTArgs& a, const Plan& p) {
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
  const uint32_t mc_ready = bars + 8u * (2 * kMaxStages + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gb + kBars + 8 * (2 * kMaxStages + 5));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gb + kBars + 8 * (2 * kMaxStages + 5) + 8);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  // this CTA's query-block tile and its run of (head, r-tile) items
  int it, j0, j1;
  mixt_items(a, it, j0, j1);
  const int i0 = it * 128;
  // first TMEM column of the part of a record tile starting at row r0
  const uint32_t zcol = (uint32_t)a.kchunks * 32u;
  auto a_col = [&](int r0) { return r0 >= p.d * p.d ? zcol : 0u; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(accfull(x), 1);
      mbar_init(accempty(x), 8);
    }
    mbar_init(mc_ready, 4);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) tma_prefetch_desc(&a.tmX);
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_launch_dependents();

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------- producer
      const uint64_t pol = policy_evict_first();
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      bool ok = true;
      // the stack comes from the preceding kernel
      pdl_wait();
      for (int j = j0; j < j1 && ok; ++j) {
        const int u = j / a.rtiles;
        const int r0 = (j % a.rtiles) * 128;
        for (int kc = 0; kc < a.kchunks; ++kc) {
          if (!(ok = mbar_wait(empty(stage), phase ^ 1u, a.err, 0x211, abort_flag))) break;
          const uint32_t st = base + (uint32_t)stage * a.stage_bytes;
          mbar_arrive_expect_tx(full(stage), a.stage_bytes);
          tma_load_4d(st, &a.tmX, full(stage), 0, kc * 64, r0 / 64, u, pol);
          ++issued;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      drain_loads(full(0), kStages, issued, a.err, 0x212);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // --------------------------------------------------------------- MMA
      const uint32_t idesc = idesc_f16_f32(128, 128, false, true);
      // stage 0's B descriptor, advanced by adding byte offset / 16 to its
      // address field (the issue of each MMA waits for the tensor pipe, so
      // every instruction on this thread adds to the step time)
      const uint64_t bd0 = sdesc_sw128(base, kAtom, 1024u);
      const uint32_t sstep = a.stage_bytes >> 4;
      int stage = 0, acc = 0, cur_u = -1;
      uint32_t phase = 0, accph = 0, loads = 0;
      bool ok = true;
      for (int j = j0; j < j1 && ok; ++j) {
        const int u = j / a.rtiles;
        const int r0 = (j % a.rtiles) * 128;
        if (u != cur_u) {
          // the A operand of head u is in tensor memory
          if (!(ok = mbar_wait(mc_ready, loads & 1u, a.err, 0x213, abort_flag))) break;
          ++loads;
          cur_u = u;
        }
        if (!(ok = mbar_wait(accempty(acc), accph ^ 1u, a.err, 0x214, abort_flag))) break;
        tc_fence_after();
        const uint32_t d = tmem + kAccCol + (uint32_t)acc * 128u;
        const uint32_t a_base = tmem + a_col(r0);
        for (int kc = 0; kc < a.kchunks; ++kc) {
          if (!(ok = mbar_wait(full(stage), phase, a.err, 0x215, abort_flag))) break;
          tc_fence_after();
          const uint64_t bd = bd0 + (uint64_t)((uint32_t)stage * sstep);
          const uint32_t ac = a_base + (uint32_t)kc * 32u;
          umma_tmem_a(d, ac, bd, idesc, kc > 0 ? 1u : 0u);
          umma_tmem_a(d, ac + 8u, bd + 128, idesc, 1u);
          umma_tmem_a(d, ac + 16u, bd + 256, idesc, 1u);
          umma_tmem_a(d, ac + 24u, bd + 384, idesc, 1u);
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
    const int q4 = warp & 3;                  // TMEM lane quarter
    const int g = (warp - 4) >> 2;            // record columns 64g .. 64g+63 of the tile
    const int gt = threadIdx.x - 128 - 128 * g;
    const int row = 32 * q4 + lane;           // query block i0 + row
    // Group 0 (warps 4-7) also writes the A operand: rows i0..i0+127 of head
    // u's two Mc copies, McS[i][q] and McZ[i][q] for q < 64 * kchunks (zero
    // past Q and past M), 16-bit pairs per 32-bit column.  The copies come
    // from the scale kernel, which has finished once the preceding kernel
    // (this CTA waits for it) has.
    const int i = i0 + 32 * q4 + lane;
    auto load_a = [&](int u) {
      for (int part = 0; part < 2; ++part) {
        const uint16_t* src = reinterpret_cast<const uint16_t*>(a.mcx) + (((size_t)u * 2 + part) * p.M + i) * a.Qp;
        for (int c0 = 0; c0 < a.kchunks * 32; c0 += 32) {
          // 64 entries of q from 2 * c0, eight at a time (the copies' rows are
          // zero from Q to the padded pitch Qp, a multiple of 8)
          uint32_t w[32];
#pragma unroll
          for (int g8 = 0; g8 < 8; ++g8) {
            const int q = 2 * c0 + 8 * g8;
            uint4 x = make_uint4(0u, 0u, 0u, 0u);
            if (i < p.M && q < a.Qp) x = *reinterpret_cast<const uint4*>(src + q);
            w[4 * g8] = x.x;
            w[4 * g8 + 1] = x.y;
            w[4 * g8 + 2] = x.z;
            w[4 * g8 + 3] = x.w;
          }
          tmem_st32(tmem + (uint32_t)part * zcol + (uint32_t)c0 + ((uint32_t)(32 * q4) << 16), w);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive_warp(mc_ready);
    };
    if (g == 0 && j0 < j1) {
      pdl_wait();
      load_a(j0 / a.rtiles);
    }
    // ------------------------------------------------------------ epilogue
    uint8_t* stg = gb + kStaging + g * kStagingGroup;
    const uint32_t stg_addr = base + kStaging + g * kStagingGroup;
    int acc = 0;
    uint32_t accph = 0;
    bool ok = true;
    for (int j = j0; j < j1 && ok; ++j) {
      const int u = j / a.rtiles;
      const int r0 = (j % a.rtiles) * 128 + 64 * g;
      const bool lo = r0 >= p.d * p.d;  // z~, v~ always carry their low residual
      ok = mbar_wait(accfull(acc), accph, a.err, 0x216, abort_flag);
      if (!(ok = named_all(1 + g, 128, ok))) break;
      tc_fence_after();
      // every MMA that read head u's A operand has completed: the next
      // item's head, if another, takes its place
      if (g == 0 && j + 1 < j1 && (j + 1) / a.rtiles != u) load_a((j + 1) / a.rtiles);
      float v0[32], v1[32];
      const uint32_t taddr = tmem + kAccCol + (uint32_t)acc * 128u + (uint32_t)(64 * g) + ((uint32_t)(32 * q4) << 16);
      tmem_ld32(taddr, v0);
      tmem_ld32(taddr + 32u, v1);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive_warp(accempty(acc));
      if (++acc == 2) {
        acc = 0;
        accph ^= 1u;
      }
      // the previous item's store has finished reading the staging tile
      if (gt == 0) bulk_wait_read<0>();
      named_sync(1 + g, 128);
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        const float* src = jj < 4 ? &v0[8 * jj] : &v1[8 * (jj - 4)];
        uint4 hv, lv;
        uint32_t* hp = &hv.x;
        uint32_t* lp = &lv.x;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          hp[q] = pack_bf16x2(src[2 * q], src[2 * q + 1]);
          if (lo) {
            const float2 h = bf16x2_to_float2(hp[q]);
            lp[q] = pack_bf16x2(src[2 * q] - h.x, src[2 * q + 1] - h.y);
          }
        }
        const uint32_t off = (uint32_t)row * 128u + ((uint32_t)((jj ^ row) & 7) << 4);
        *reinterpret_cast<uint4*>(stg + off) = hv;
        if (lo) *reinterpret_cast<uint4*>(stg + kStagingPart + off) = lv;
      }
      fence_proxy_async();
      named_sync(1 + g, 128);
      if (gt == 0) {
        tma_store_3d(&a.tmO, stg_addr, r0, i0, u);
        if (lo) tma_store_3d(&a.tmO_lo, stg_addr + kStagingPart, r0, i0, u);
        bulk_commit();
      }
    }
    if (gt == 0) bulk_wait<0>();
  }
  __syncwarp();

  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace mt

// Host side (tc_mix.cu): whether the TMEM-resident kernel can take the plan,
// and its tensor maps and scalars.
bool mixt_supported(const Plan& p, const TcBuffers& b);
int build_mixt_args(const Plan& p, const TcBuffers& b, mt::MixTArgs* out);

}  // namespace mhla
