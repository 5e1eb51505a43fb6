// Output step on the tensor cores ("MHLA: Restoring Expressivity of Linear
// Attention via Token-Level Multi-Head", flowchart output node and key design
// 2; "Rectifying Magnitude Neglect in Linear Attention", key designs).
//
// For a token tile of query block i (up to 128 tokens, gathered by one TMA box
// from the token grid) one tcgen05 MMA of N = 80 per K step yields numerators
// and denominators together:
//     D = phi(Q_tile) [S~_i | Z]   (M = 128 tokens, K = 64, N = 64 + 16)
//     D[t][c] = phi(q_t)^T S~_i[:, c],  s_t = D[t][64] + D[t][65]
// where Z, the second N atom of B, holds z~_i in two columns (high and low
// bf16 parts) and zeros elsewhere.
// The epilogue forms
//   DIVISIVE o = D / s,  NONE o = D,
//   MALA     o = (1 + 1/s) D - (s / n~_i) v~_i,   n~_i = n_b sum_b Mc[i, b]
// writes the bf16 result over the Q tile in shared memory, and one TMA store
// scatters it back to the grid positions of the tile.
//   A = phi(Q) tile: K-major (features contiguous), as TMA delivered it
//   B = S~_i: MN-major ([k][c], c contiguous), loaded by TMA from the mixed
//       stack (bf16 high part; MALA adds the low residual as a third MMA)
//   Z: MN-major like S~_i (8 KB), columns 0 and 1 written per unit
// Two rings of shared-memory stages: Q tiles (16 KB, streamed from HBM, the
// deep one: it sets how many bytes are in flight) and the per-block operands
// S~_i, Z, z~_i / v~_i rows and the output scale (read from L2, a few stages).
// With exponential features phi(Q) also goes in as bf16 high + low parts:
// the low parts through a third, short ring and one more MMA per K step.
// Persistent, warp-specialised CTA (640 threads): warp 0 Q producer, warp 1
// TMEM + MMA, warp 2 block-operand producer, warp 3 Z and v~_i, warps 4-11
// phi(Q) (two threads per token row), warps 12-19 epilogue (two warps per
// TMEM lane quarter, 32 output features each).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "tc_common.cuh"
#include "tc_host.h"

namespace mhla {
namespace ot {

using namespace tc;

constexpr int kThreads = 640;
constexpr int kXfThreads = 256;                    // warps 4..11
constexpr int kEpiThreads = 256;                   // warps 12..19
constexpr uint32_t kQTile = 128 * 128;             // Q / O tile
constexpr uint32_t kBTile = 64 * 128;              // 64 k-rows x 64 columns
constexpr int kBStages = 4;
constexpr int kPendStores = 4;                     // O stores in flight per CTA
constexpr int kAccSlots = 4;                       // TMEM accumulators (128 columns each, 80 used)
constexpr uint32_t kAccStride = 128;
constexpr uint32_t kTmemCols = 512;

// Shared-memory layout; kLo (MALA, exponential features) adds the low
// residual of S~_i, kQLo (exponential features) a ring of kQLoStages tiles
// for the low residual of phi(Q), each free again once its tile's MMAs have
// completed.
template <bool kLo, bool kQLo>
struct Layout {
  static constexpr int kQStages = (kLo ? 7 : 9) - (kQLo ? 2 : 0);
  static constexpr int kQLoStages = kQLo ? 2 : 0;
  static constexpr uint32_t kQLoBase = kQStages * kQTile;
  // block-operand stage: S~_i hi [, lo] | Z (the second N atom of B) | misc
  static constexpr uint32_t kOffBlo = kBTile;
  static constexpr uint32_t kOffZ = kLo ? 2 * kBTile : kBTile;
  static constexpr uint32_t kOffMisc = kOffZ + kBTile;
  static constexpr uint32_t kOffV = kOffMisc;               // v~_i, 64 floats (MALA)
  static constexpr uint32_t kOffAux = kOffMisc + 256;       // rows z~_i, v~_i of Mixed, bf16 hi (256 B)
  static constexpr uint32_t kOffAuxLo = kOffMisc + 512;     // same, low residuals
  static constexpr uint32_t kOffInfo = kOffMisc + 768;      // float4 {output scale, n~_i, 0, 0}
  static constexpr uint32_t kBStageBytes = kOffMisc + 1024;
  static constexpr uint32_t kBBase = kQLoBase + kQLoStages * kQTile;
  static constexpr uint32_t kBars = kBBase + kBStages * kBStageBytes;
  static constexpr int kNumBars = 4 * kQStages + 3 * kBStages + kAccSlots + kQLoStages;
  static constexpr uint32_t kSmemBytes = kBars + 8 * kNumBars + 16 + 1024;
  static_assert(kBStageBytes % 1024 == 0, "stage alignment");
};

static_assert(Layout<false, false>::kSmemBytes <= 232448 && Layout<true, false>::kSmemBytes <= 232448 &&
                  Layout<false, true>::kSmemBytes <= 232448 && Layout<true, true>::kSmemBytes <= 232448,
              "shared memory");

struct OutArgs {
  CUtensorMap tmQ, tmO;        // 5D (64, Wg, Hg, T, BH), box (64, cw, ch, ct, 1)
  const __nv_bfloat16* mixed_hi;  // records of the mixed summaries (rows z~_i, v~_i read by cp.async)
  const __nv_bfloat16* mixed_lo;
  int R;                          // record length
  CUtensorMap tmB_hi, tmB_lo;  // 3D (64, R/64, slots*M), box (64, 64, 1)
  const float4* blkinfo;       // per query block {output scale, n~_i, 0, 0}
  int info_per_slot;           // blkinfo rows per slot (fp16 path) instead of per mixing matrix
  int units;
  ChunkShape c;
  FastDiv f_head, f_nck;       // divisions by M * nck and by nck (units per head, per block)
  unsigned int* err;
};

// Head, query block and chunk of work unit w (head-major, then block, then
// chunk).
__device__ __forceinline__ void out_unit(const Plan& p, const OutArgs& a, int w, int& u, int& i, int& c) {
  const uint32_t uu = fdiv((uint32_t)w, a.f_head);
  const uint32_t rem = (uint32_t)w - uu * (uint32_t)(p.M * a.c.per_block);
  const uint32_t ii = fdiv(rem, a.f_nck);
  u = (int)uu;
  i = (int)ii;
  c = (int)(rem - ii * (uint32_t)a.c.per_block);
}

// The kernel body; `a` must live in kernel parameter space.
template <bool kLo, bool kQLo>
__device__ __forceinline__ void output_body(const OutArgs& a, const Plan& p, const FlowCtl& f) {
  using L = Layout<kLo, kQLo>;
  constexpr int kQStages = L::kQStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gb = smem_raw + (base - raw);
  const uint32_t bars = base + L::kBars;
  auto qfull = [&](int s) { return bars + 8u * s; };
  auto qready = [&](int s) { return bars + 8u * (kQStages + s); };
  auto qmma = [&](int s) { return bars + 8u * (2 * kQStages + s); };
  auto qempty = [&](int s) { return bars + 8u * (3 * kQStages + s); };
  auto bfull = [&](int b) { return bars + 8u * (4 * kQStages + b); };
  auto bready = [&](int b) { return bars + 8u * (4 * kQStages + kBStages + b); };
  auto bempty = [&](int b) { return bars + 8u * (4 * kQStages + 2 * kBStages + b); };
  auto accempty = [&](int x) { return bars + 8u * (4 * kQStages + 3 * kBStages + x); };
  // phi(Q) low-residual tile j is free (its tile's MMAs have completed)
  auto lofree = [&](int j) { return bars + 8u * (4 * kQStages + 3 * kBStages + kAccSlots + j); };
  auto qlo = [&](int j) { return base + L::kQLoBase + (uint32_t)j * kQTile; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gb + L::kBars + 8 * L::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gb + L::kBars + 8 * L::kNumBars + 8);
  auto qst = [&](int s) { return base + (uint32_t)s * kQTile; };
  auto bst = [&](int b) { return base + L::kBBase + (uint32_t)b * L::kBStageBytes; };

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int rows = a.c.rows;
  const int nck = a.c.per_block;
  const int per_head = p.M * nck;

  // Z operands: every row except 0 and 1 stays zero
  for (int b = 0; b < kBStages; ++b)
    for (uint32_t off = threadIdx.x * 16u; off < kBTile; off += kThreads * 16u)
      *reinterpret_cast<uint4*>(gb + L::kBBase + b * L::kBStageBytes + L::kOffZ + off) = make_uint4(0u, 0u, 0u, 0u);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kQStages; ++s) {
      mbar_init(qfull(s), 1);
      mbar_init(qready(s), kXfThreads / 32);
      mbar_init(qmma(s), 1);
      mbar_init(qempty(s), 1);
    }
    for (int b = 0; b < kBStages; ++b) {
      mbar_init(bfull(b), 1);
      mbar_init(bready(b), 1);
      mbar_init(bempty(b), 1);
    }
    for (int x = 0; x < kAccSlots; ++x) mbar_init(accempty(x), 1);
    for (int j = 0; j < L::kQLoStages; ++j) mbar_init(lofree(j), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&a.tmQ);
    tma_prefetch_desc(&a.tmO);
  }
  if (warp == 2 && lane == 0) tma_prefetch_desc(&a.tmB_hi);
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_launch_dependents();

  if (warp == 0) {
    if (lane == 0) {
      // -------------------------------------------------------- Q producer
      // (Q is an input: its loads need not wait for the mixing kernel)
      const uint64_t pol_q = policy_evict_first();
      const uint32_t bytes = (uint32_t)rows * 128u;
      int s = 0;
      uint32_t ph = 0;
      long long issued = 0;
      for (int w = f.cta; w < a.units; w += f.ncta) {
        int u, i, c, x0, y0, t0;
        out_unit(p, a, w, u, i, c);
        if (!mbar_wait(qempty(s), ph ^ 1u, a.err, 0x301, abort_flag)) break;
        chunk_origin(p, a.c, (uint32_t)i, (uint32_t)c, x0, y0, t0);
        const TileCoords g5 = token_tile_coords(p, u, x0, y0, t0);
        mbar_arrive_expect_tx(qfull(s), bytes);
        tma_load_5d(qst(s), &a.tmQ, qfull(s), g5.c[0], g5.c[1], g5.c[2], g5.c[3], g5.c[4], pol_q);
        ++issued;
        if (++s == kQStages) {
          s = 0;
          ph ^= 1u;
        }
      }
      drain_loads(qfull(0), kQStages, issued, a.err, 0x30b);
    }
  } else if (warp == 2) {
    // ---------------------------------------------- block-operand producer
    // lane 0: S~_i (hi [, lo]) by TMA; every lane: one 16-byte piece of the
    // z~_i / v~_i rows (hi: lanes 0-15, lo: 16-31) and lane 0 the block info,
    // by cp.async (small copies are cheaper outside the TMA engine)
    const uint64_t pol_b = policy_evict_last();
    const uint32_t bytes = kBTile * (kLo ? 2u : 1u);
    int b = 0, ready_u = -1;
    uint32_t ph = 0;
    long long issued = 0;
    // the mixed summaries and the block info come from the preceding kernels
    if (lane == 0) pdl_wait();
    __syncwarp();
    for (int w = f.cta; w < a.units; w += f.ncta) {
      int u, i, c;
      out_unit(p, a, w, u, i, c);
      bool ok = true;
      if (lane == 0) {
        // fused flow: the mixed summaries of head u are written
        if (f.x_done && u != ready_u) ok = flow_wait(&f.x_done[u], f.need_x + f.stall, a.err, 0x307, abort_flag, f.wait_ns);
        ok = ok && mbar_wait(bempty(b), ph ^ 1u, a.err, 0x308, abort_flag);
      }
      if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
      ready_u = u;
      const uint32_t st = bst(b);
      const int rec = flow_slot(f, u) * p.M + i;  // record of S~_i in the mixed summaries
      const __nv_bfloat16* src = (lane < 16 ? a.mixed_hi : a.mixed_lo) + (size_t)rec * a.R + 64 * 64 + (lane & 15) * 8;
      cp_async16(st + (lane < 16 ? L::kOffAux : L::kOffAuxLo) + (lane & 15) * 16, src);
      if (lane == 0)
        cp_async16(st + L::kOffInfo, a.blkinfo + (a.info_per_slot ? flow_slot(f, u) : mc_index(p, u)) * p.M + i);
      cp_async_arrive(bfull(b));
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_expect_tx(bfull(b), bytes);
        tma_load_3d(st, &a.tmB_hi, bfull(b), 0, 0, rec, pol_b);
        if (kLo) tma_load_3d(st + L::kOffBlo, &a.tmB_lo, bfull(b), 0, 0, rec, pol_b);
      }
      ++issued;
      if (++b == kBStages) {
        b = 0;
        ph ^= 1u;
      }
    }
    // the barrier completes only once this lane's cp.async copies and the
    // TMA bytes have landed
    if (lane == 0) drain_loads(bfull(0), kBStages, issued, a.err, 0x30c);
  } else if (warp == 3) {
    // ---------------------------- Z (z~_i hi, lo as rows 0, 1) and v~_i
    int b = 0;
    uint32_t ph = 0;
    for (int w = f.cta; w < a.units; w += f.ncta) {
      const bool ok = mbar_wait(bfull(b), ph, a.err, 0x309, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) break;
      uint8_t* st = gb + L::kBBase + b * L::kBStageBytes;
      const __nv_bfloat16* aux = reinterpret_cast<const __nv_bfloat16*>(st + L::kOffAux);
      const __nv_bfloat16* auxlo = reinterpret_cast<const __nv_bfloat16*>(st + L::kOffAuxLo);
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int k = lane + 32 * j;
        *reinterpret_cast<__nv_bfloat16*>(st + L::kOffZ + sw128_offset(k, 0)) = aux[k];
        *reinterpret_cast<__nv_bfloat16*>(st + L::kOffZ + sw128_offset(k, 1)) = auxlo[k];
        reinterpret_cast<float*>(st + L::kOffV)[k] = __bfloat162float(aux[64 + k]) + __bfloat162float(auxlo[64 + k]);
      }
      fence_proxy_async();
      mbar_arrive_warp(bready(b));
      if (++b == kBStages) {
        b = 0;
        ph ^= 1u;
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // --------------------------------------------------------------- MMA
      const uint32_t idesc80 = idesc_bf16_f32(128, 80, false, true);
      const uint32_t idesc64 = idesc_bf16_f32(128, 64, false, true);
      int s = 0, b = 0, slot = 0, lj = 0;
      uint32_t ph = 0, bph = 0, slotph = 0;
      for (int w = f.cta; w < a.units; w += f.ncta) {
        if (!mbar_wait(qready(s), ph, a.err, 0x302, abort_flag)) break;
        if (!mbar_wait(bready(b), bph, a.err, 0x30a, abort_flag)) break;
        if (!mbar_wait(accempty(slot), slotph ^ 1u, a.err, 0x306, abort_flag)) break;
        tc_fence_after();
        const uint32_t qs = qst(s), bs = bst(b);
        const uint32_t d = tmem + (uint32_t)slot * kAccStride;
        // descriptors of K step 0, advanced by adding byte offset / 16 to the
        // address field (the issue of each MMA waits for the tensor pipe, so
        // every instruction on this thread adds to the tile's time)
        const uint64_t ad0 = sdesc_sw128(qs, 0u, 1024u);
        const uint64_t bd0 = sdesc_sw128(bs, L::kOffZ, 1024u);
        const uint64_t bl0 = sdesc_sw128(bs + L::kOffBlo, kBTile, 1024u);
        const uint64_t ql0 = sdesc_sw128(kQLo ? qlo(lj) : qs, 0u, 1024u);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint64_t ad = ad0 + 2 * ks;     // + 32 bytes per K step
          const uint64_t bd = bd0 + 128 * ks;   // + 2048 bytes per K step
          const uint32_t acc = ks > 0 ? 1u : 0u;
          umma_bf16(d, ad, bd, idesc80, acc);
          if (kLo) umma_bf16(d, ad, bl0 + 128 * ks, idesc64, 1u);
          // the low residual of phi(Q) times [S~_i | Z]
          if (kQLo) umma_bf16(d, ql0 + 2 * ks, bd, idesc80, 1u);
        }
        if (kQLo) {
          umma_commit(lofree(lj));
          if (++lj == L::kQLoStages) lj = 0;
        }
        umma_commit(qmma(s));
        if (++s == kQStages) {
          s = 0;
          ph ^= 1u;
        }
        if (++b == kBStages) {
          b = 0;
          bph ^= 1u;
        }
        if (++slot == kAccSlots) {
          slot = 0;
          slotph ^= 1u;
        }
      }
    }
  } else if (warp >= 4 && warp < 12) {
    // -------------------------------------------------------------- phi(Q)
    const int t = threadIdx.x - 128;
    const int row = t >> 1;
    const int half = t & 1;
    int s = 0, lj = 0;
    uint32_t ph = 0, lph = 0;
    for (int w = f.cta; w < a.units; w += f.ncta) {
      bool ok = mbar_wait(qfull(s), ph, a.err, 0x303, abort_flag);
      if (kQLo) ok = ok && mbar_wait(lofree(lj), lph ^ 1u, a.err, 0x30d, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) break;
      if (row < rows) {
        uint8_t* rp = gb + s * kQTile + row * 128;
        uint8_t* lp = gb + L::kQLoBase + lj * kQTile + row * 128;
        uint4 xs[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) xs[j] = *reinterpret_cast<const uint4*>(rp + (((4 * half + j + row) & 7) << 4));
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t off = ((4 * half + j + row) & 7) << 4;
          uint4 x = xs[j], lo;
          uint32_t* xp = &x.x;
          uint32_t* lop = &lo.x;
          if (!kQLo && p.fmap == MHLA_FEATURE_ELU1) {
#pragma unroll
            for (int q = 0; q < 4; ++q) xp[q] = phi2_elu1_bf16(xp[q]);
          } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float2 fv = bf16x2_to_float2(xp[q]);
              const float p0 = phi_map(fv.x, p.fmap), p1 = phi_map(fv.y, p.fmap);
              xp[q] = pack_bf16x2(p0, p1);
              if (kQLo) {
                const float2 hv = bf16x2_to_float2(xp[q]);
                lop[q] = pack_bf16x2(p0 - hv.x, p1 - hv.y);
              }
            }
          }
          *reinterpret_cast<uint4*>(rp + off) = x;
          if (kQLo) *reinterpret_cast<uint4*>(lp + off) = lo;
        }
      }
      if (kQLo && ++lj == L::kQLoStages) {
        lj = 0;
        lph ^= 1u;
      }
      fence_proxy_async();
      mbar_arrive_warp(qready(s));
      if (++s == kQStages) {
        s = 0;
        ph ^= 1u;
      }
    }
  } else if (warp >= 12) {
    // ------------------------------------------------------------ epilogue
    const int q4 = warp & 3;            // TMEM lane quarter
    const int h = (warp - 12) >> 2;     // output features 32h .. 32h+31
    const int t = 32 * q4 + lane;       // token row = TMEM lane
    const int et = threadIdx.x - 384;
    int s = 0, b = 0, n_out = 0, slot = 0;
    uint32_t ph = 0, bph = 0;
    unsigned int batch = 0;
    for (int w = f.cta; w < a.units; w += f.ncta) {
      int u, i, c;
      out_unit(p, a, w, u, i, c);
      bool ok = mbar_wait(qmma(s), ph, a.err, 0x304, abort_flag);
      // the block operands (v~_i floats written by warp 3)
      ok = ok && mbar_wait(bready(b), bph, a.err, 0x305, abort_flag);
      if (!named_all(3, kEpiThreads, ok)) break;
      tc_fence_after();
      float o[32], s0, s1;
      const uint32_t taddr = tmem + (uint32_t)slot * kAccStride + ((uint32_t)(32 * q4) << 16);
      tmem_ld32(taddr + 32u * h, o);
      tmem_ld2(taddr + 64u, s0, s1);
      tmem_wait_ld();
      if (t < rows) {
        const uint8_t* bp = gb + L::kBBase + b * L::kBStageBytes;
        const float sden = s0 + s1;
        const float4 info = *reinterpret_cast<const float4*>(bp + L::kOffInfo);
        // info.x undoes the powers of two of the fp16 records: 2^(ES - EZ)
        // under DIVISIVE, 2^ES under NONE (1 for split records)
        float scale = info.x, gamma = 0.f;
        if (p.norm == MHLA_NORM_DIVISIVE) {
          scale = sden != 0.f ? info.x * __frcp_rn(sden) : 0.f;  // s = 0: no key mass, output 0
        } else if (p.norm == MHLA_NORM_MALA) {
          scale = sden != 0.f ? 1.f + __frcp_rn(sden) : 0.f;  // beta
          gamma = sden / info.y;                            // s / n~_i
        }
        const float* vs = reinterpret_cast<const float*>(bp + L::kOffV) + 32 * h;
        uint8_t* rp = gb + s * kQTile + t * 128;
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
      if (et == 0) {
        // every epilogue thread has read the accumulator and the block operands
        mbar_arrive(accempty(slot));
        mbar_arrive(bempty(b));
        int x0, y0, t0;
        chunk_origin(p, a.c, (uint32_t)i, (uint32_t)c, x0, y0, t0);
        const TileCoords g5 = token_tile_coords(p, u, x0, y0, t0);
        tma_store_5d(&a.tmO, qst(s), g5.c[0], g5.c[1], g5.c[2], g5.c[3], g5.c[4]);
        bulk_commit();
        // this CTA's units of head u have read their S~_i (the slot may be
        // reused once every unit has)
        if (f.o_done && (++batch, flow_head_ends(f, w, a.units, per_head))) {
          flow_signal(&f.o_done[u], batch);
          batch = 0;
        }
        // release the stage of the store kPendStores - 1 units back once it
        // has been read (later stores may still be queued behind Q loads)
        bulk_wait_read<kPendStores - 1>();
        if (n_out >= kPendStores - 1) mbar_arrive(qempty((s + kQStages - (kPendStores - 1)) % kQStages));
      }
      ++n_out;
      if (++s == kQStages) {
        s = 0;
        ph ^= 1u;
      }
      if (++b == kBStages) {
        b = 0;
        bph ^= 1u;
      }
      if (++slot == kAccSlots) slot = 0;
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
constexpr uint32_t output_smem_bytes(bool lo, bool qlo) {
  return lo ? (qlo ? ot::Layout<true, true>::kSmemBytes : ot::Layout<true, false>::kSmemBytes)
            : (qlo ? ot::Layout<false, true>::kSmemBytes : ot::Layout<false, false>::kSmemBytes);
}

}  // namespace mhla
