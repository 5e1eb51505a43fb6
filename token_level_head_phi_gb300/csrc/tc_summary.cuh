// Block summaries on the tensor cores (head dimension 64, bf16 inputs).
//
// For every block b of every head ("MHLA: Restoring Expressivity of Linear
// Attention via Token-Level Multi-Head", overall framework):
//   S_b = sum_{j in b} phi(K_j) V_j^T,  z_b = sum_{j in b} phi(K_j),
//   v_b = sum_{j in b} V_j  (the last one feeds the MALA normalisation).
// All three come out of ONE 128x80 tcgen05 MMA per 16 tokens:
//   A = [phi(K_b)^T ; 1^T]  (rows 0..63 features of phi(K), rows 64..127 ones)
//   B = [V_b | 1]           (cols 0..63 features of V, cols 64..79 ones)
//   D = A B:  D[k][c] = S_b[k][c], D[k][64] = z_b[k], D[64][c] = v_b[c].
// Both operands are MN-major: the token tile arrives by TMA exactly as it
// lies in memory ([token][feature], 128-byte rows, 128-byte swizzle).  The
// second M atom of A and the second N atom of B (the ones) are reached
// through the descriptors' leading-byte offset; since one MMA reads only 16
// token rows of each atom, that offset is set per K step so that both land
// on the same 16-row (2 KB) tile of ones.  phi = ELU+1 is applied in place to the
// K tile by the transform warps; padding rows stay zero.  For MALA the low
// bf16 residual of phi(K) goes through a second MMA (its ones rows add v_b a
// second time, which the epilogue halves).
//
// Persistent, warp-specialised CTA (one per SM, 640 threads):
//   warp 0       TMA producer (K and V tiles of one token chunk per stage)
//   warp 1       TMEM allocation; warps 1, 2 MMA issue (even / odd units,
//                each through its own ring of stages and its own two of the
//                four TMEM accumulators)
//   warps 4-6, 16-17  epilogue: TMEM rows 0..64 -> the record (S_b, z_b,
//                v_b) as fp16 (DIVISIVE/NONE: S_b and z_b each scaled by a
//                power of two taken from its own largest entry, the two
//                exponents stored beside the record; v_b, which only MALA
//                reads, as zeros) or as bf16 high + low parts (split) ->
//                swizzled staging tiles (two, used in turn) -> TMA stores
//                into the summary stack
//   warps 8-15   phi(K) transform, two threads per token row
// Each CTA walks work units (head, block, piece) with a static stride; long
// blocks are cut into pieces whose partial summaries the mixing step adds.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "tc_common.cuh"
#include "tc_host.h"

namespace mhla {
namespace sm {

using namespace tc;

constexpr int kThreads = 640;
constexpr int kEpiThreads = 160;                        // warps 4, 5, 6, 16, 17
constexpr int kXfThreads = 256;                         // warps 8..15
constexpr uint32_t kTile = 128 * 128;                   // 128 rows of 128 bytes
constexpr uint32_t kStagePart = 8192 + 1024;            // staging: S 8 KB + zv 1 KB
constexpr uint32_t kStagingBuf = 2 * kStagePart;        // hi and lo
constexpr int kAccs = 4;                                // TMEM accumulators: unit it uses it % 4
constexpr uint32_t kTmemCols = 512;                     // four 128-column accumulators (80 columns used)
constexpr int kN = 80;                                  // MMA N: 64 value features + 16 ones

// Shared-memory layout.  kLo adds the low bf16 residual of phi(K) as a third
// tile per stage (MALA); the stage count shrinks (and one staging buffer
// is kept) to keep everything resident.
template <bool kLo>
struct Layout {
  static constexpr int kStages = kLo ? 4 : 6;
  static constexpr int kIssuers = 2;                                 // MMA-issuing warps (1, 2)
  static constexpr int kStagingBufs = kLo ? 1 : 2;
  static constexpr uint32_t kStageBytes = (kLo ? 3 : 2) * kTile;  // K, V [, K lo]
  static constexpr uint32_t kOnes = kStages * kStageBytes;          // 16 token rows of ones (2 KB)
  static constexpr uint32_t kStaging = kOnes + 2048;                // staging buffers
  static constexpr uint32_t kStagingStride = kLo ? kStagingBuf : kStagePart;
  static constexpr uint32_t kBars = kStaging + kStagingBufs * kStagingStride;
  static constexpr uint32_t kSmemBytes = kBars + 256 + 1024;        // + barriers + alignment slack
  static_assert(kStaging % 1024 == 0 && kStagingStride % 1024 == 0 && kSmemBytes <= 232448, "layout");
};

struct SummaryArgs {
  CUtensorMap tmK, tmV;              // 5D (64, Wg, Hg, T, BH), box (64, cw, ch, ct, 1)
  CUtensorMap tmS, tmS_lo;           // 2D view (64, BH*Q*66) of the stack, box (64, 64): S_b rows
  CUtensorMap tmZV, tmZV_lo;         // same view, box (64, 2): the z_b and v_b rows
  int units, splits, cpp;            // work units, pieces per block, chunks per piece
  int wait_prev;                     // no prep kernel before this one: wait for the stream's previous work
  int2* rexp;                        // fp16 records: [slots * M * splits] exponents {eS, eZ}
  ChunkShape c;
  FastDiv f_head, f_splits;          // divisions by M * splits and by splits
  unsigned int* err;
};

struct UnitCoord {
  int u, b, c0, c1;
};

__device__ __forceinline__ UnitCoord unit_coord(const Plan& p, const SummaryArgs& a, int w) {
  UnitCoord r;
  const uint32_t u = fdiv((uint32_t)w, a.f_head);
  const uint32_t rem = (uint32_t)w - u * (uint32_t)(p.M * a.splits);
  const uint32_t b = fdiv(rem, a.f_splits);
  r.u = (int)u;
  r.b = (int)b;
  r.c0 = (int)(rem - b * (uint32_t)a.splits) * a.cpp;
  r.c1 = min(a.c.per_block, r.c0 + a.cpp);
  return r;
}

// phi of 8 bf16 (one 16-byte chunk), rounded to bf16; optionally also the
// low bf16 residual.
template <bool kLo>
__device__ __forceinline__ void phi_chunk(uint4& x, uint4& lo, int fmap) {
  uint32_t* xp = &x.x;
  uint32_t* lp = &lo.x;
  if (!kLo && fmap == MHLA_FEATURE_ELU1) {
#pragma unroll
    for (int q = 0; q < 4; ++q) xp[q] = phi2_elu1_bf16(xp[q]);
    return;
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float2 f = bf16x2_to_float2(xp[q]);
    const float a = phi_map(f.x, fmap), b = phi_map(f.y, fmap);
    xp[q] = pack_bf16x2(a, b);
    if (kLo) {
      const float2 g = bf16x2_to_float2(xp[q]);
      lp[q] = pack_bf16x2(a - g.x, b - g.y);
    }
  }
}

// Exponent e of an fp16 record part whose largest magnitude has the float
// bits `amax_bits` (sign cleared): the part is stored times 2^-e, which puts
// that entry in [2^14, 2^15) -- every entry down to 2^-29 of it stays a normal
// fp16 number, and no rounding can reach the fp16 limit 65504.  Read from the
// exponent field (amax in [2^k, 2^(k+1)) gives e = k - 14); clamped so that
// 2^-e is a normal float (a part whose largest entry is below 2^-106 counts
// as zero).  An infinite entry stays infinite, NaN stays NaN.
__device__ __forceinline__ int record_exponent(uint32_t amax_bits) {
  const int e = (int)((amax_bits >> 23) & 0xFFu) - 141;
  return min(max(e, -120), 113);
}

// Largest |v[j]| of 32 floats as float bits (for non-negative floats the
// bit patterns order as the values do): a tree of maxima, five deep (|x| is
// an operand modifier of the max, not an instruction).
__device__ __forceinline__ uint32_t abs_max_bits32(const float (&v)[32]) {
  float m[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) m[j] = fmaxf(fabsf(v[2 * j]), fabsf(v[2 * j + 1]));
#pragma unroll
  for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
    for (int j = 0; j < w; ++j) m[j] = fmaxf(m[j], m[j + w]);
  return __float_as_uint(m[0]);
}


// 2^-e as a float, for e in [-120, 113].
__device__ __forceinline__ float pow2_neg(int e) { return __uint_as_float((uint32_t)(127 - e) << 23); }

// 8 floats (times scale) -> 8 bf16 (hi) and optionally their low residuals.
__device__ __forceinline__ void split8(const float* src, uint4& hv, uint4& lv, float scale, bool want_lo) {
  uint32_t* hp = &hv.x;
  uint32_t* lp = &lv.x;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float x0 = src[2 * q] * scale, x1 = src[2 * q + 1] * scale;
    hp[q] = pack_bf16x2(x0, x1);
    if (want_lo) {
      const float2 g = bf16x2_to_float2(hp[q]);
      lp[q] = pack_bf16x2(x0 - g.x, x1 - g.y);
    }
  }
}

// The kernel body; `a` must live in kernel parameter space (TMA reads the
// tensor maps from there).
template <bool kLo>
__device__ __forceinline__ void summary_body(const SummaryArgs& a, const Plan& p, const FlowCtl& f) {
  using L = Layout<kLo>;
  constexpr int kStages = L::kStages;
  constexpr uint32_t kStageBytes = L::kStageBytes;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gb = smem_raw + (base - raw);
  const uint32_t bars = base + L::kBars;
  auto full = [&](int s) { return bars + 8u * s; };
  auto kready = [&](int s) { return bars + 8u * (kStages + s); };
  auto empty = [&](int s) { return bars + 8u * (2 * kStages + s); };
  auto accfull = [&](int x) { return bars + 8u * (3 * kStages + x); };
  auto accempty = [&](int x) { return bars + 8u * (3 * kStages + kAccs + x); };
  // Stage rings: with two MMA issuers (kIssuers), unit number `it` of this
  // CTA goes through ring it % kIssuers, the stages j, j + kIssuers, ...; each
  // ring is filled in order by the producer and drained in order by ONE
  // issuer, so no waiter ever falls two phases behind a stage's barriers.
  // (one issuer when a unit has more chunks than a ring has stages: its
  // chunks would wait on their own ring's reuse)
  const int kIssuers = (L::kIssuers == 2 && a.cpp <= kStages / 2) ? 2 : 1;
  auto ring_len = [&](int j) { return (kStages - j + kIssuers - 1) / kIssuers; };
  auto ring_stage = [&](int j, long long k) { return j + kIssuers * (int)(k % ring_len(j)); };
  auto ring_phase = [&](int j, long long k) { return (uint32_t)((k / ring_len(j)) & 1); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gb + L::kBars + 8 * (3 * kStages + 2 * kAccs));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gb + L::kBars + 8 * (3 * kStages + 2 * kAccs) + 8);
  // epilogue: per-warp maxima of the fp16 record parts (float bits)
  uint32_t* red = reinterpret_cast<uint32_t*>(gb + L::kBars + 224);
  static_assert(8 * (3 * kStages + 2 * kAccs) + 12 <= 224 && 224 + 4 * 6 <= 256, "barrier area");

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int rows = a.c.rows;

  // Stage tiles start zeroed (padding rows must stay zero, so they add
  // nothing against the ones); the ones tile holds 1.0 everywhere.
  for (uint32_t off = threadIdx.x * 16u; off < L::kStaging; off += kThreads * 16u) {
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    if (off >= L::kOnes) val = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
    *reinterpret_cast<uint4*>(gb + off) = val;
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(kready(s), kXfThreads / 32);
      mbar_init(empty(s), 1);
    }
    for (int x = 0; x < kAccs; ++x) {
      mbar_init(accfull(x), 1);
      mbar_init(accempty(x), kEpiThreads / 32);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&a.tmK);
    tma_prefetch_desc(&a.tmV);
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
  // First kernel of a call: what came before in the stream (the previous
  // call, whose kernels read the stack this one writes, or the producer of K
  // and V) has finished.  After the prep kernel, which waited for it, K and V
  // are inputs with nothing to wait for.
  if (a.wait_prev) pdl_wait();
  // the next kernel may start its set-up as SMs free up
  pdl_launch_dependents();

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      const uint32_t bytes = 2u * (uint32_t)rows * 128u;
      int ready_u = -1, it = 0;
      long long rk0 = 0, rk1 = 0;   // loads issued per ring
      bool ok = true;
      for (int w = f.cta; w < a.units && ok; w += f.ncta, ++it) {
        const UnitCoord uc = unit_coord(p, a, w);
        // fused flow: the stack slot of this head is free once the mixing of
        // the head that last used it has read it
        if (f.x_done && f.ring && uc.u >= f.ring && uc.u != ready_u &&
            !(ok = flow_wait(&f.x_done[uc.u - f.ring], f.need_x, a.err, 0x108, abort_flag, f.wait_ns)))
          break;
        ready_u = uc.u;
        const int j = it % kIssuers;
        for (int c = uc.c0; c < uc.c1; ++c) {
          const long long k = j ? rk1 : rk0;
          const int stage = ring_stage(j, k);
          if (!(ok = mbar_wait(empty(stage), ring_phase(j, k) ^ 1u, a.err, 0x101, abort_flag))) break;
          int x0, y0, t0;
          chunk_origin(p, a.c, uc.b, c, x0, y0, t0);
          const TileCoords g5 = token_tile_coords(p, uc.u, x0, y0, t0);
          const uint32_t kt = base + (uint32_t)stage * kStageBytes;
          mbar_arrive_expect_tx(full(stage), bytes);
          tma_load_5d(kt, &a.tmK, full(stage), g5.c[0], g5.c[1], g5.c[2], g5.c[3], g5.c[4], pol);
          tma_load_5d(kt + kTile, &a.tmV, full(stage), g5.c[0], g5.c[1], g5.c[2], g5.c[3], g5.c[4], pol);
          if (j) ++rk1;
          else ++rk0;
        }
      }
      // before the CTA's memory is released: the last loads of each ring
      // have landed (bounded, whatever the abort flag says)
      for (int j = 0; j < kIssuers; ++j) {
        const long long n = j ? rk1 : rk0;
        const long long first = n > ring_len(j) ? n - ring_len(j) : 0;
        for (long long k = first; k < n; ++k) {
          const uint32_t bar = full(ring_stage(j, k)), par = ring_phase(j, k);
          if (mbar_try_wait(bar, par)) continue;
          const unsigned long long t0 = globaltimer();
          while (!mbar_try_wait_sleep(bar, par, 20000u)) {
            if (globaltimer() - t0 > kWaitLimitNs) {
              report_timeout(a.err, 0x109);
              break;
            }
          }
        }
      }
    }
  } else if (warp == 1 || warp == 2) {
    // --------------------------------------------------------------- MMA
    // A tcgen05.mma holds its issuing warp for a fixed time whatever its N,
    // so with two issuers warp 1 takes this CTA's even units (accumulator 0,
    // ring 0) and warp 2 the odd ones (accumulator 1, ring 1); with one,
    // warp 1 takes every unit and alternates the accumulators.
    const int j = warp - 1;
    if (lane == 0 && j < kIssuers) {
      const uint32_t idesc = idesc_bf16_f32(128, kN, true, true);
      const int ksteps = a.c.rows_pad / 16;
      long long rk = 0;       // chunks taken from ring j
      int it = 0;
      bool ok = true;
      for (int w = f.cta; w < a.units && ok; w += f.ncta, ++it) {
        if (it % kIssuers != j) continue;
        const UnitCoord uc = unit_coord(p, a, w);
        // unit it accumulates in slot it % 4: each issuer alternates two
        // slots, so it can start a unit before the epilogue has read the
        // previous one out of tensor memory
        const int acc = it & (kAccs - 1);
        if (!(ok = mbar_wait(accempty(acc), ((uint32_t)(it / kAccs) & 1u) ^ 1u, a.err, 0x102, abort_flag))) break;
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)acc * 128u;
        for (int c = uc.c0; c < uc.c1; ++c) {
          const int stage = ring_stage(j, rk);
          if (!(ok = mbar_wait(kready(stage), ring_phase(j, rk), a.err, 0x103, abort_flag))) break;
          tc_fence_after();
          const uint32_t kt = base + (uint32_t)stage * kStageBytes;
          const uint32_t vt = kt + kTile;
          const uint32_t ones = base + L::kOnes;
          // the second atoms of A and B: the ones tile, whatever the K step.
          // Descriptors advance by adding to their fields (address + 2048
          // bytes, leading offset to the ones tile - 2048 bytes per K step):
          // the issue of each MMA waits for the tensor pipe, so every
          // instruction on this thread adds to the unit's time.
          const uint64_t e_step = 128ull - (128ull << 16);
          uint64_t kd = sdesc_sw128(kt, ones - kt, 1024u), vd = sdesc_sw128(vt, ones - vt, 1024u);
          uint64_t ld = sdesc_sw128(kt + 2 * kTile, ones - (kt + 2 * kTile), 1024u);
          for (int ks = 0; ks < ksteps; ++ks) {
            umma_bf16(d, kd, vd, idesc, (c > uc.c0 || ks > 0) ? 1u : 0u);
            if (kLo) umma_bf16(d, ld, vd, idesc, 1u);
            kd += e_step;
            vd += e_step;
            ld += e_step;
          }
          umma_commit(empty(stage));
          ++rk;
        }
        if (!ok) break;
        umma_commit(accfull(acc));
      }
    }
  } else if (warp >= 8 && warp < 16) {
    // ------------------------------------------------ phi(K) transform
    // thread t: row t/2, chunks 4*(t%2) .. +3 at physical positions rotated
    // by the row so that 8 consecutive threads hit 8 distinct bank groups
    const int t = threadIdx.x - 256;
    const int row = t >> 1;
    const int half = t & 1;
    long long rk0 = 0, rk1 = 0;   // chunks taken from rings 0, 1
    int it = 0;
    bool ok = true;
    for (int w = f.cta; w < a.units && ok; w += f.ncta, ++it) {
      const UnitCoord uc = unit_coord(p, a, w);
      const int ring = it % kIssuers;
      for (int c = uc.c0; c < uc.c1; ++c) {
        const long long k = ring ? rk1 : rk0;
        const int stage = ring_stage(ring, k);
        if (!(ok = mbar_wait(full(stage), ring_phase(ring, k), a.err, 0x104, abort_flag))) break;
        if (row < rows) {
          uint8_t* rp = gb + stage * kStageBytes + row * 128;
          uint4 x[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) x[j] = *reinterpret_cast<const uint4*>(rp + (((4 * half + j + row) & 7) << 4));
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t off = ((4 * half + j + row) & 7) << 4;
            uint4 lo;
            phi_chunk<kLo>(x[j], lo, p.fmap);
            *reinterpret_cast<uint4*>(rp + off) = x[j];
            if (kLo) *reinterpret_cast<uint4*>(rp + 2 * kTile + off) = lo;
          }
        }
        fence_proxy_async();
        mbar_arrive_warp(kready(stage));
        if (ring) ++rk1;
        else ++rk0;
      }
    }
  } else if (warp == 4 || warp == 5 || warp == 6 || warp == 16 || warp == 17) {
    // ------------------------------------------------------------ epilogue
    // warps 4/16 -> rows 0..31, 5/17 -> rows 32..63 (columns 0..31 / 32..63),
    // warp 6 -> row 64 (v_b)
    const int e = warp & 3;                   // TMEM lane quarter
    const int h = warp >= 16 ? 1 : 0;         // column half of S_b
    const int et = warp < 16 ? threadIdx.x - 128 : 96 + threadIdx.x - 512;
    const int r = 32 * e + lane;  // TMEM lane = row of D
    int it = 0;
    unsigned int batch = 0;
    bool ok = true;
    for (int w = f.cta; w < a.units && ok; w += f.ncta, ++it) {
      const UnitCoord uc = unit_coord(p, a, w);
      const int acc = it & (kAccs - 1);
      ok = mbar_wait(accfull(acc), (uint32_t)(it / kAccs) & 1u, a.err, 0x105, abort_flag);
      if (!(ok = named_all(1, kEpiThreads, ok))) break;
      tc_fence_after();
      const uint32_t taddr = tmem + (uint32_t)acc * 128u + ((uint32_t)(32 * e) << 16);
      float s0[32], s1[32], zval = 0.f, znext;
      tmem_ld32(taddr + 32u * h, s0);
      if (e == 2) tmem_ld32(taddr + 32u, s1);
      tmem_ld2(taddr + 64u, zval, znext);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive_warp(accempty(acc));

      uint8_t* st_hi = gb + L::kStaging + (it % L::kStagingBufs) * L::kStagingStride;
      uint8_t* st_lo = st_hi + kStagePart;
      if (!kLo && e < 2) {
        // largest magnitudes (float bits) of this warp's share of S_b and
        // z_b, gathered in shared memory: red[2e + h] (S_b), red[4 + e] (z_b)
        const uint32_t am = __reduce_max_sync(0xffffffffu, abs_max_bits32(s0));
        const uint32_t amz = __reduce_max_sync(0xffffffffu, h == 0 ? __float_as_uint(fabsf(zval)) : 0u);
        if (lane == 0) {
          red[2 * e + h] = am;
          if (h == 0) red[4 + e] = amz;
        }
      }
      if (et == 0) {
        // the store that last read this staging buffer has finished reading it
        bulk_wait_read<L::kStagingBufs - 1>();
      }
      named_sync(1, kEpiThreads);
      int eS = 0, eZ = 0;
      if (!kLo) {
        eS = record_exponent(max(max(red[0], red[1]), max(red[2], red[3])));
        eZ = record_exponent(max(red[4], red[5]));
      }
      if (e < 2) {
        // row r of S_b (columns 32h .. 32h+31) and, for h = 0, z_b[r]
        const float scS = kLo ? 1.f : pow2_neg(eS);
        const float2 sc2 = make_float2(scS, scS);
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const int j = 4 * h + jj;
          const float* src = &s0[8 * jj];
          uint4 hv, lv;
          if (!kLo) {
            uint32_t* hp = &hv.x;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              // two products per instruction (exact: a power of two)
              const float2 y = __fmul2_rn(make_float2(src[2 * q], src[2 * q + 1]), sc2);
              __half2 hh = __floats2half2_rn(y.x, y.y);
              hp[q] = *reinterpret_cast<uint32_t*>(&hh);
            }
          } else {
            split8(src, hv, lv, 1.f, true);
          }
          const uint32_t off = (uint32_t)r * 128u + ((uint32_t)((j ^ (r & 7)) & 7) << 4);
          *reinterpret_cast<uint4*>(st_hi + off) = hv;
          if (kLo) *reinterpret_cast<uint4*>(st_lo + off) = lv;
        }
        if (h == 0) {
          if (!kLo) {
            *reinterpret_cast<__half*>(st_hi + 8192 + sw128_offset(0, r)) = __float2half_rn(zval * pow2_neg(eZ));
          } else {
            const __nv_bfloat16 zh = __float2bfloat16_rn(zval);
            *reinterpret_cast<__nv_bfloat16*>(st_hi + 8192 + sw128_offset(0, r)) = zh;
            *reinterpret_cast<__nv_bfloat16*>(st_lo + 8192 + sw128_offset(0, r)) =
                __float2bfloat16_rn(zval - __bfloat162float(zh));
          }
        }
      } else if (lane == 0) {
        // row 64 of D: v_b (every row 64..127 holds the same values; the
        // low-residual MMA of MALA adds them twice).  The fp16 records feed
        // DIVISIVE and NONE only, which never read v_b: zeros.
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float* src = j < 4 ? &s0[8 * j] : &s1[8 * (j - 4)];
          uint4 hv = make_uint4(0u, 0u, 0u, 0u), lv;
          if (kLo) split8(src, hv, lv, 0.5f, true);
          const uint32_t off = 128u + ((uint32_t)((j ^ 1) & 7) << 4);
          *reinterpret_cast<uint4*>(st_hi + 8192 + off) = hv;
          if (kLo) *reinterpret_cast<uint4*>(st_lo + 8192 + off) = lv;
        }
      }
      fence_proxy_async();
      named_sync(1, kEpiThreads);
      if (et == 0) {
        const int srow = (flow_slot(f, uc.u) * p.M + uc.b) * a.splits + (uc.c0 / a.cpp);
        if (!kLo) a.rexp[srow] = make_int2(eS, eZ);
        tma_store_2d(&a.tmS, smem_u32(st_hi), 0, srow * 66);
        tma_store_2d(&a.tmZV, smem_u32(st_hi + 8192), 0, srow * 66 + 64);
        if (kLo) {
          tma_store_2d(&a.tmS_lo, smem_u32(st_lo), 0, srow * 66);
          tma_store_2d(&a.tmZV_lo, smem_u32(st_lo + 8192), 0, srow * 66 + 64);
        }
        bulk_commit();
        // fused flow: after this CTA's last unit of the head, publish the
        // head's rows once they are stored
        if (f.s_done && (++batch, flow_head_ends(f, w, a.units, p.M * a.splits))) {
          bulk_wait<0>();
          flow_signal(&f.s_done[uc.u], batch);
          batch = 0;
        }
      }
    }
    if (et == 0) bulk_wait<0>();
  }
  __syncwarp();

  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
  // this kernel completes only after its predecessor (the prep kernel, whose
  // Mc copies the mixing reads) has
  if (threadIdx.x == 0) pdl_wait();
}

}  // namespace sm

// Host side (tc_summary.cu): tensor maps and scalars for a launch whose stack
// holds `slots` heads; shared-memory bytes of the kernel body.
int build_summary_args(const Plan& p, const ChunkShape& c, const void* k, const void* v, const TcBuffers& b,
                       int slots, sm::SummaryArgs* out);
uint32_t summary_smem_bytes(bool lo);

}  // namespace mhla
