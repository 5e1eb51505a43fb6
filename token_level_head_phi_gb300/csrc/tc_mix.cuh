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
//   kF16  (DIVISIVE/NONE): X = the fp16 records (S_q 2^-eS[q], z_q 2^-eZ[q]),
//         B = the head's fp16 copy of Mc with those exponents folded in
//         (McS for the tiles of S rows, McZ for the tile of z and v rows);
//         one MMA per K step; Mixed holds S~_i 2^-ES[i] and z~_i 2^-EZ[i],
//         which the output step scales back.
//   split (MALA, causal, fused): X and Mc as bf16 high + low parts,
//         D = Xh Mh + Xh Ml + Xl Mh in two MMAs per K step: Xh [Mh | Ml]
//         (N = 2 NT: the two B tiles lie back to back in shared memory, so
//         one descriptor spans both) into accumulator columns [0, 2 NT), and
//         Xl Mh into [0, NT); the epilogue adds columns c and NT + c.
// The epilogue writes Mixed as bf16 (plus the low residual where the output
// step needs it): 32 query blocks x 128 r at a time, transposed through a
// shared-memory tile and stored by TMA.
//
// Also here: the small preparation kernel that builds the Mc copies.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "tc_common.cuh"
#include "tc_host.h"

namespace mhla {
namespace mx {

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
  CUtensorMap tmA, tmA_lo;     // 4D (64, Q, W / 64, slots), box (64, 64, 2, 1): two r atoms
  CUtensorMap tmB, tmB_lo;     // 2D (Q, rows), box (64, NT): Mc copies, [mc_heads][M] or [slots][2][M] rows
  CUtensorMap tmO, tmO_lo;     // 3D (R, M, BH) view of Mixed, box (128, 32, 1), no swizzle
  int Q, NT, itiles, rtiles, kchunks, units;
  int r_off;                   // column of Mixed where this part starts
  int write_lo;                // write the low residual of every value
  int b_per_slot;              // B rows per slot and part (fp16 path) instead of per mixing matrix
  int stages;
  uint32_t stage_bytes, off_alo, off_b, off_blo;
  unsigned int* err;
};

// The kernel body; `a` must live in kernel parameter space.
template <bool kF16>
__device__ __forceinline__ void mix_body(const MixArgs& a, const Plan& p, const FlowCtl& f) {
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
      mbar_init(accempty(x), 4 * kEpiGroups);
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
  pdl_launch_dependents();

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------- producer
      const uint64_t pol_a = policy_evict_first();
      const uint64_t pol_b = policy_evict_last();
      const uint32_t bytes = kF16 ? kATile + (uint32_t)a.NT * 128u : 2u * kATile + 2u * (uint32_t)a.NT * 128u;
      int stage = 0, ready_u = -1;
      uint32_t phase = 0;
      long long issued = 0;
      bool ok = true;
      // the stack and the Mc copies come from the preceding kernels
      pdl_wait();
      for (int w = f.cta; w < a.units && ok; w += f.ncta) {
        const int u = w / per_head;
        const int rem = w % per_head;
        const int r0 = (rem / a.itiles) * 128;
        const int i0 = (rem % a.itiles) * a.NT;
        const int ss = flow_slot(f, u);
        // fused flow: every summary of head u is written, and the mixed slot
        // is no longer read by the outputs of the head that last used it
        if (f.s_done && u != ready_u) {
          if (!(ok = flow_wait(&f.s_done[u], f.need_s, a.err, 0x205, abort_flag, f.wait_ns))) break;
          if (f.ring && u >= f.ring &&
              !(ok = flow_wait(&f.o_done[u - f.ring], f.need_o, a.err, 0x206, abort_flag, f.wait_ns)))
            break;
          ready_u = u;
        }
        for (int kc = 0; kc < a.kchunks; ++kc) {
          if (!(ok = mbar_wait(empty(stage), phase ^ 1u, a.err, 0x201, abort_flag))) break;
          const uint32_t st = base + (uint32_t)stage * a.stage_bytes;
          mbar_arrive_expect_tx(full(stage), bytes);
          tma_load_4d(st, &a.tmA, full(stage), 0, kc * 64, r0 / 64, ss, pol_a);
          // rows of this head's mixing matrix: its own fp16 copy for the S
          // or the z part of the record, or the matrix it shares
          const int ib = i0 + (a.b_per_slot ? (2 * ss + (r0 >= p.d * p.d ? 1 : 0)) : mc_index(p, u)) * p.M;
          tma_load_2d(st + a.off_b, &a.tmB, full(stage), kc * 64, ib, pol_b);
          if (!kF16) {
            tma_load_4d(st + a.off_alo, &a.tmA_lo, full(stage), 0, kc * 64, r0 / 64, ss, pol_a);
            tma_load_2d(st + a.off_blo, &a.tmB_lo, full(stage), kc * 64, ib, pol_b);
          }
          ++issued;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      drain_loads(full(0), kStages, issued, a.err, 0x207);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // --------------------------------------------------------------- MMA
      const uint32_t idesc = kF16 ? idesc_f16_f32(128, a.NT, true, false) : idesc_bf16_f32(128, a.NT, true, false);
      const uint32_t idesc2 = idesc_bf16_f32(128, 2 * a.NT, true, false);  // split: Xh [Mh | Ml]
      // Descriptors of stage 0, advanced by adding byte offset / 16 to their
      // address field (the shared memory window is below 256 KB, so the
      // field never carries): the issue of each MMA waits for the tensor
      // pipe, so every instruction on this thread adds to the step time.
      const uint64_t ad0 = sdesc_sw128(base, kAtom, 1024u);
      const uint64_t bd0 = sdesc_sw128(base + a.off_b, 0u, 1024u);
      const uint64_t ld0 = sdesc_sw128(base + a.off_alo, kAtom, 1024u);
      const uint32_t sstep = a.stage_bytes >> 4;
      int stage = 0, acc = 0;
      uint32_t phase = 0, accph = 0;
      bool ok = true;
      for (int w = f.cta; w < a.units && ok; w += f.ncta) {
        if (!(ok = mbar_wait(accempty(acc), accph ^ 1u, a.err, 0x202, abort_flag))) break;
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)acc * 256u;
        for (int kc = 0; kc < a.kchunks; ++kc) {
          if (!(ok = mbar_wait(full(stage), phase, a.err, 0x203, abort_flag))) break;
          tc_fence_after();
          const uint64_t so = (uint64_t)((uint32_t)stage * sstep);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const uint64_t ahi = ad0 + so + 128 * ks;  // + 2048 bytes per K step
            const uint64_t bhi = bd0 + so + 2 * ks;    // + 32 bytes per K step
            const uint32_t accum = (kc > 0 || ks > 0) ? 1u : 0u;
            if (kF16) {
              umma_bf16(d, ahi, bhi, idesc, accum);
            } else {
              // the B descriptor at Mh spans Ml too (off_blo = off_b + NT rows)
              umma_bf16(d, ahi, bhi, idesc2, accum);
              umma_bf16(d, ld0 + so + 128 * ks, bhi, idesc, 1u);
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
  } else if (warp >= 4 && warp < 4 + 4 * kEpiGroups) {
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
    uint32_t accph = 0, sbuf = 0;
    bool prev_both = false;
    unsigned int batch = 0;
    bool ok = true;
    for (int w = f.cta; w < a.units && ok; w += f.ncta) {
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
        if (!kF16) {
          // split: add the Xh Ml products, NT columns further
          float v2[32];
          tmem_ld32(taddr + (uint32_t)(a.NT + c0), v2);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] += v2[j];
        }
        tmem_wait_ld();
        // Slices without low residuals alternate between the two halves of
        // the staging area, so a slice waits only for the store before the
        // previous one; a slice with residuals takes both halves.
        const uint32_t off = lo ? 0u : sbuf * 8192u;
        if (gt == 0) {
          if (lo || prev_both) bulk_wait_read<0>();
          else bulk_wait_read<1>();
        }
        named_sync(1 + g, 128);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const __nv_bfloat16 h = __float2bfloat16_rn(v[j]);
          reinterpret_cast<__nv_bfloat16*>(stg + off)[j * 128 + rl] = h;
          if (lo)
            reinterpret_cast<__nv_bfloat16*>(stg + 8192)[j * 128 + rl] = __float2bfloat16_rn(v[j] - __bfloat162float(h));
        }
        fence_proxy_async();
        named_sync(1 + g, 128);
        if (gt == 0) {
          tma_store_3d(&a.tmO, stg_addr + off, r0, i0 + c0, flow_slot(f, u));
          if (lo) tma_store_3d(&a.tmO_lo, stg_addr + 8192, r0, i0 + c0, flow_slot(f, u));
          bulk_commit();
        }
        prev_both = lo;
        if (!lo) sbuf ^= 1u;
      }
      if (f.x_done && gt == 0 && (++batch, flow_head_ends(f, w, a.units, per_head))) {
        // this group's rows of the head are written: publish them
        bulk_wait<0>();
        flow_signal(&f.x_done[u], batch);
        batch = 0;
      }
      tc_fence_before();
      mbar_arrive_warp(accempty(acc));
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

}  // namespace mx

// Host side (tc_mix.cu): tensor maps and scalars for a launch whose stack and
// mixed summaries hold `slots` heads.
int build_mix_args(const Plan& p, const TcBuffers& b, int slots, mx::MixArgs* out);
constexpr uint32_t mix_smem_bytes() { return mx::kSmemBytes; }

}  // namespace mhla
