// Output step on the tensor cores ("MHLA: Restoring Expressivity of Linear
// Attention via Token-Level Multi-Head", flowchart output node and key design
// 2; "Rectifying Magnitude Neglect in Linear Attention", key designs).
//
// For a token tile of query block i (up to 128 tokens, gathered by one TMA box
// from the token grid) one tcgen05 MMA of N = 80 yields numerators and
// denominators together:
//     D = phi(Q_tile) [S~_i | z~_i]   (M = 128 tokens, K = 64, N = 64 + 16)
//     D[t][c] = phi(q_t)^T S~_i[:, c],  s_t = D[t][64] + D[t][65]
// where the second B atom holds z~_i in two columns (high and low bf16
// parts) and zeros elsewhere.  The epilogue forms
//   DIVISIVE o = D / s,  NONE o = D,
//   MALA     o = (1 + 1/s) D - (s / n~_i) v~_i,   n~_i = n_b sum_b Mc[i, b]
// writes the bf16 result over the Q tile in shared memory, and one TMA store
// scatters it back to the grid positions of the tile.
//   A = phi(Q) tile: K-major (features contiguous), as TMA delivered it
//   B = S~_i: MN-major ([k][c], c contiguous), loaded by TMA from the mixed
//       stack (bf16 high part; MALA adds the low residual as a second MMA)
// Persistent, warp-specialised CTA (640 threads): warp 0 TMA producer,
// warp 1 TMEM + MMA, warps 4-11 phi(Q) (two threads per token row) and the
// z~/v~ operands, warps 12-19 epilogue (two warps per TMEM lane quarter,
// 32 output features each).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "tc_common.cuh"
#include "tc_host.h"

namespace mhla {
namespace ot {

using namespace tc;

constexpr int kStages = 5;
constexpr int kThreads = 640;
constexpr int kXfThreads = 256;                    // warps 4..11
constexpr int kEpiThreads = 256;                   // warps 12..19
constexpr uint32_t kQTile = 128 * 128;             // Q / O tile
constexpr uint32_t kBTile = 64 * 128;              // 64 k-rows x 64 columns
constexpr uint32_t kOffBhi = kQTile;               // S~_i high part
constexpr uint32_t kOffZt = kOffBhi + kBTile;      // z~_i as columns 0 (hi) and 1 (lo)
constexpr uint32_t kOffBlo = kOffZt + kBTile;      // S~_i low part (MALA)
constexpr uint32_t kOffV = kOffBlo + kBTile;       // v~_i, 64 floats (MALA)
constexpr uint32_t kOffAux = kOffV + 256;          // rows z~_i, v~_i of Mixed, bf16 hi (256 B)
constexpr uint32_t kOffAuxLo = kOffAux + 256;      // same, low residuals
constexpr uint32_t kOffInfo = kOffAuxLo + 256;     // float4 {output scale, n~_i, 0, 0}
constexpr uint32_t kStageBytes = kOffV + 1024;
static_assert(kOffInfo + 16 <= kStageBytes, "stage layout");
constexpr uint32_t kBars = kStages * kStageBytes;
constexpr uint32_t kSmemBytes = kBars + 256 + 1024;
constexpr int kAccSlots = 4;                       // TMEM accumulators (128 columns each, 80 used)
constexpr uint32_t kAccStride = 128;
constexpr uint32_t kTmemCols = 512;

static_assert(kStageBytes % 1024 == 0, "stage alignment");

struct OutArgs {
  CUtensorMap tmQ, tmO;        // 5D (64, Wg, Hg, T, BH), box (64, cw, ch, ct, 1)
  CUtensorMap tmB_hi, tmB_lo;  // 3D (64, R/64, BH*M), box (64, 64, 1)
  CUtensorMap tmA_hi, tmA_lo;  // same view, box (64, 2, 1), no swizzle: rows z~_i, v~_i
  const float4* blkinfo;       // per query block {output scale, n~_i, 0, 0}
  int units;
  int use_lo;
  ChunkShape c;
  unsigned int* err;
};

// The kernel body; `a` must live in kernel parameter space.
__device__ __forceinline__ void output_body(const OutArgs& a, const Plan& p, const FlowCtl& f) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gb = smem_raw + (base - raw);
  const uint32_t bars = base + kBars;
  auto full = [&](int s) { return bars + 8u * s; };
  auto tready = [&](int s) { return bars + 8u * (kStages + s); };
  auto mmadone = [&](int s) { return bars + 8u * (2 * kStages + s); };
  auto empty = [&](int s) { return bars + 8u * (3 * kStages + s); };
  auto accempty = [&](int x) { return bars + 8u * (4 * kStages + x); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gb + kBars + 8 * (4 * kStages + kAccSlots));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gb + kBars + 8 * (4 * kStages + kAccSlots) + 8);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int rows = a.c.rows;
  const int nck = a.c.per_block;
  const int per_head = p.M * nck;

  // z~ tiles: every column except 0 and 1 stays zero
  for (int s = 0; s < kStages; ++s)
    for (uint32_t off = threadIdx.x * 16u; off < kBTile; off += kThreads * 16u)
      *reinterpret_cast<uint4*>(gb + s * kStageBytes + kOffZt + off) = make_uint4(0u, 0u, 0u, 0u);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(tready(s), kXfThreads / 32);
      mbar_init(mmadone(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int x = 0; x < kAccSlots; ++x) mbar_init(accempty(x), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&a.tmQ);
    tma_prefetch_desc(&a.tmO);
    tma_prefetch_desc(&a.tmB_hi);
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
      // ---------------------------------------------------------- producer
      const uint64_t pol_q = policy_evict_first();
      const uint64_t pol_b = policy_evict_last();
      const uint32_t bytes = (uint32_t)rows * 128u + kBTile * (a.use_lo ? 2u : 1u) + 512u + 16u;
      int stage = 0, ready_u = -1;
      uint32_t phase = 0;
      for (int w = f.cta; w < a.units; w += f.ncta) {
        const int u = w / per_head;
        const int rem = w % per_head;
        const int i = rem / nck;
        const int c = rem % nck;
        // fused flow: the mixed summaries of head u are written
        if (f.x_done && u != ready_u && !flow_wait(&f.x_done[u], f.need_x, a.err, 0x307, abort_flag)) break;
        ready_u = u;
        if (!mbar_wait(empty(stage), phase ^ 1u, a.err, 0x301, abort_flag)) break;
        const int bx = i % p.Mw, by = (i / p.Mw) % p.Mh, bz = i / (p.Mw * p.Mh);
        const int x0 = bx * p.bw + (c % a.c.ncx) * a.c.cw;
        const int y0 = by * p.bh + ((c / a.c.ncx) % a.c.ncy) * a.c.ch;
        const int t0 = bz * p.bt + (c / (a.c.ncx * a.c.ncy)) * a.c.ct;
        const uint32_t st = base + (uint32_t)stage * kStageBytes;
        mbar_arrive_expect_tx(full(stage), bytes);
        tma_load_5d(st, &a.tmQ, full(stage), 0, x0, y0, t0, u, pol_q);
        const int rec = flow_slot(f, u) * p.M + i;  // record of S~_i in the mixed summaries
        tma_load_3d(st + kOffBhi, &a.tmB_hi, full(stage), 0, 0, rec, pol_b);
        if (a.use_lo) tma_load_3d(st + kOffBlo, &a.tmB_lo, full(stage), 0, 0, rec, pol_b);
        tma_load_3d(st + kOffAux, &a.tmA_hi, full(stage), 0, p.d, rec, pol_b);
        tma_load_3d(st + kOffAuxLo, &a.tmA_lo, full(stage), 0, p.d, rec, pol_b);
        bulk_load(st + kOffInfo, a.blkinfo + i, 16u, full(stage));
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // --------------------------------------------------------------- MMA
      const uint32_t idesc80 = idesc_bf16_f32(128, 80, false, true);
      const uint32_t idesc64 = idesc_bf16_f32(128, 64, false, true);
      int stage = 0, slot = 0;
      uint32_t phase = 0, slotph = 0;
      for (int w = f.cta; w < a.units; w += f.ncta) {
        if (!mbar_wait(tready(stage), phase, a.err, 0x302, abort_flag)) break;
        if (!mbar_wait(accempty(slot), slotph ^ 1u, a.err, 0x306, abort_flag)) break;
        tc_fence_after();
        const uint32_t st = base + (uint32_t)stage * kStageBytes;
        const uint32_t d = tmem + (uint32_t)slot * kAccStride;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint64_t ad = sdesc_sw128(st + (uint32_t)ks * 32u, 0u, 1024u);
          umma_bf16(d, ad, sdesc_sw128(st + kOffBhi + (uint32_t)ks * 2048u, kOffZt - kOffBhi, 1024u), idesc80,
                    ks > 0 ? 1u : 0u);
          if (a.use_lo)
            umma_bf16(d, ad, sdesc_sw128(st + kOffBlo + (uint32_t)ks * 2048u, kBTile, 1024u), idesc64, 1u);
        }
        umma_commit(mmadone(stage));
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
        if (++slot == kAccSlots) {
          slot = 0;
          slotph ^= 1u;
        }
      }
    }
  } else if (warp >= 4 && warp < 12) {
    // ----------------------------------- phi(Q) and the z~_i / v~_i operands
    const int t = threadIdx.x - 128;
    const int row = t >> 1;
    const int half = t & 1;
    int stage = 0;
    uint32_t phase = 0;
    for (int w = f.cta; w < a.units; w += f.ncta) {
      const bool ok = mbar_wait(full(stage), phase, a.err, 0x303, abort_flag);
      if (!named_all(2, kXfThreads, ok)) break;
      uint8_t* st = gb + stage * kStageBytes;
      // threads 0..63: z~_i[k] (hi, lo) into columns 0, 1 of the z~ operand;
      // threads 64..127: v~_i[c] = hi + lo as float for the MALA epilogue
      if (t < 128) {
        const __nv_bfloat16 zh = reinterpret_cast<const __nv_bfloat16*>(st + kOffAux)[t];
        const __nv_bfloat16 zl = reinterpret_cast<const __nv_bfloat16*>(st + kOffAuxLo)[t];
        if (t < 64) {
          *reinterpret_cast<__nv_bfloat16*>(st + kOffZt + sw128_offset(t, 0)) = zh;
          *reinterpret_cast<__nv_bfloat16*>(st + kOffZt + sw128_offset(t, 1)) = zl;
        } else {
          reinterpret_cast<float*>(st + kOffV)[t - 64] = __bfloat162float(zh) + __bfloat162float(zl);
        }
      }
      if (row < rows) {
        uint8_t* rp = st + row * 128;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t off = ((4 * half + j + row) & 7) << 4;
          uint4 x = *reinterpret_cast<uint4*>(rp + off);
          uint32_t* xp = &x.x;
          if (p.fmap == MHLA_FEATURE_ELU1) {
#pragma unroll
            for (int q = 0; q < 4; ++q) xp[q] = phi2_elu1_bf16(xp[q]);
          } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float2 f = bf16x2_to_float2(xp[q]);
              xp[q] = pack_bf16x2(phi_map(f.x, p.fmap), phi_map(f.y, p.fmap));
            }
          }
          *reinterpret_cast<uint4*>(rp + off) = x;
        }
      }
      fence_proxy_async();
      mbar_arrive_warp(tready(stage));
      if (++stage == kStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
  } else if (warp >= 12) {
    // ------------------------------------------------------------ epilogue
    const int q4 = warp & 3;            // TMEM lane quarter
    const int h = (warp - 12) >> 2;     // output features 32h .. 32h+31
    const int t = 32 * q4 + lane;       // token row = TMEM lane
    const int et = threadIdx.x - 384;
    int stage = 0, prev = -1, slot = 0;
    uint32_t phase = 0;
    unsigned int batch = 0;
    for (int w = f.cta; w < a.units; w += f.ncta) {
      const int u = w / per_head;
      const int rem = w % per_head;
      const int i = rem / nck;
      const int c = rem % nck;
      bool ok = mbar_wait(mmadone(stage), phase, a.err, 0x304, abort_flag);
      // the transform's shared-memory writes (v~)
      ok = ok && mbar_wait(tready(stage), phase, a.err, 0x305, abort_flag);
      if (!named_all(3, kEpiThreads, ok)) break;
      tc_fence_after();
      float o[32], s0, s1;
      const uint32_t taddr = tmem + (uint32_t)slot * kAccStride + ((uint32_t)(32 * q4) << 16);
      tmem_ld32(taddr + 32u * h, o);
      tmem_ld2(taddr + 64u, s0, s1);
      tmem_wait_ld();
      uint8_t* st = gb + stage * kStageBytes;
      if (t < rows) {
        const float s = s0 + s1;
        const float4 info = *reinterpret_cast<const float4*>(st + kOffInfo);
        // info.x undoes the fp16 mixing's power-of-two scale; under DIVISIVE
        // numerator and denominator carry the same scale, which cancels
        float scale = info.x, gamma = 0.f;
        if (p.norm == MHLA_NORM_DIVISIVE) {
          scale = __frcp_rn(s);
        } else if (p.norm == MHLA_NORM_MALA) {
          scale = 1.f + __frcp_rn(s);                       // beta
          gamma = s / info.y;                               // s / n~_i
        }
        const float* vs = reinterpret_cast<const float*>(st + kOffV) + 32 * h;
        uint8_t* rp = st + t * 128;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint4 x;
          uint32_t* xp = &x.x;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int cc = 8 * j + 2 * q;
            float y0 = o[cc] * scale, y1 = o[cc + 1] * scale;
            if (p.norm == MHLA_NORM_MALA) {
              y0 -= gamma * vs[cc];
              y1 -= gamma * vs[cc + 1];
            }
            xp[q] = pack_bf16x2(y0, y1);
          }
          *reinterpret_cast<uint4*>(rp + ((((4 * h + j) ^ t) & 7) << 4)) = x;
        }
      }
      fence_proxy_async();
      tc_fence_before();
      named_sync(3, kEpiThreads);
      if (et == 0) mbar_arrive(accempty(slot));  // every epilogue thread has read the accumulator
      if (++slot == kAccSlots) slot = 0;
      if (et == 0) {
        const int bx = i % p.Mw, by = (i / p.Mw) % p.Mh, bz = i / (p.Mw * p.Mh);
        const int x0 = bx * p.bw + (c % a.c.ncx) * a.c.cw;
        const int y0 = by * p.bh + ((c / a.c.ncx) % a.c.ncy) * a.c.ch;
        const int t0 = bz * p.bt + (c / (a.c.ncx * a.c.ncy)) * a.c.ct;
        tma_store_5d(&a.tmO, base + (uint32_t)stage * kStageBytes, 0, x0, y0, t0, u);
        bulk_commit();
        // this CTA's units of head u have read their S~_i (the slot may be
        // reused once every unit has)
        if (f.o_done && (++batch, flow_head_ends(f, w, a.units, per_head))) {
          flow_signal(&f.o_done[u], batch);
          batch = 0;
        }
        // the previous tile's store has finished reading its stage: release it
        bulk_wait_read<1>();
        if (prev >= 0) mbar_arrive(empty(prev));
      }
      prev = stage;
      if (++stage == kStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (et == 0) bulk_wait<0>();
  }
  __syncwarp();

  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace ot

// Host side (tc_output.cu): tensor maps and scalars for a launch whose mixed
// summaries hold `slots` heads.
int build_output_args(const Plan& p, const ChunkShape& c, const void* q, const TcBuffers& b, void* out, int slots,
                      ot::OutArgs* args);
constexpr uint32_t output_smem_bytes() { return ot::kSmemBytes; }

}  // namespace mhla
