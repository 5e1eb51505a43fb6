// Key and value gradients on the tensor cores (head dimension 64, bf16).
//
// The block summaries S_b = sum_j phi(K_j) V_j^T, z_b = sum_j phi(K_j),
// v_b = sum_j V_j ("MHLA: Restoring Expressivity of Linear Attention via
// Token-Level Multi-Head", overall framework) are linear in each token's
// contribution, so with dS_b, dz_b, dv_b the gradients of the loss with
// respect to them (Mc^T times the gradients of the mixed summaries):
//     dK_j = (dS_b V_j + dz_b) * phi'(K_j)
//     dV_j = dS_b^T phi(K_j) + dv_b
// For a token tile of block b (up to 128 tokens, one TMA box from the grid):
//     D_K = [V | 1] [dS_b | dz_b]^T      M = 128 tokens, N = 64 (k), K = 64 + 16
//     D_V = [phi(K) | 1] [dS_b ; dv_b^T]  M = 128 tokens, N = 64 (c), K = 64 + 16
//   A = V tile (K-major, exact bf16) or phi(K) tile (K-major, bf16 high + low
//       parts: two MMAs), as TMA delivered the token rows
//   B = dS_b as loaded from the gradient record ([k][c], c contiguous):
//       K-major for D_K, MN-major for D_V; bf16 high + low planes
//   the bias K step: A = a tile of ones (columns 0 and 1), B = dz_b (K-major,
//       columns 0, 1 = high, low) or dv_b (MN-major, rows 0, 1 = high, low)
// phi'(K) comes from the two parts of phi(K): min(phi, 1) for ELU+1 (1 above
// zero, exp(K) = phi(K) at and below it), [phi > 0] for ReLU, phi for exp.  The epilogue
// writes dK over the phi(K) tile and dV over the V tile and stores both by
// TMA to the grid positions of the tile.
// Persistent, warp-specialised CTA (512 threads): warp 0 K/V producer, warp 1
// TMEM + MMA, warp 2 gradient-record producer, warp 3 bias operands, warps
// 4-11 phi(K) (two threads per token row), warps 12-15 epilogue (one thread
// per token row = TMEM lane).
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
constexpr int kXfThreads = 256;                // warps 4..11
constexpr int kEpiThreads = 128;               // warps 12..15
constexpr uint32_t kTile = 128 * 128;          // 128 token rows of 64 bf16
constexpr uint32_t kBTile = 64 * 128;          // 64 rows of 64 bf16
constexpr int kStages = 3;
constexpr int kBStages = 2;
constexpr int kPendStores = 2;
// token stage: K -> phi(K) high part -> dK | V -> dV | phi(K) low part
constexpr uint32_t kStageBytes = 3 * kTile;
// gradient-record stage: dS hi | dS lo | Zk (dz as K-major columns 0, 1) |
// Zv (dv as MN-major rows 0, 1; 16 rows) | aux rows (dz, dv hi and lo)
constexpr uint32_t kOffSlo = kBTile;
constexpr uint32_t kOffZk = 2 * kBTile;
constexpr uint32_t kOffZv = 3 * kBTile;
constexpr uint32_t kOffAux = 3 * kBTile + 2048;     // 4 rows x 128 bytes: dz hi, dv hi, dz lo, dv lo
constexpr uint32_t kBStageBytes = 3 * kBTile + 3072;
constexpr uint32_t kOnes = kStages * kStageBytes;   // 128 x 64 tile, columns 0 and 1 one
constexpr uint32_t kBBase = kOnes + kTile;
constexpr uint32_t kBars = kBBase + kBStages * kBStageBytes;
constexpr int kNumBars = 4 * kStages + 3 * kBStages + 2 * 2;
constexpr uint32_t kSmemBytes = kBars + 8 * kNumBars + 16 + 1024;
constexpr uint32_t kTmemCols = 256;               // two accumulator sets of 128 columns (D_K | D_V)
static_assert(kSmemBytes <= 232448, "shared memory");
static_assert(kBStageBytes % 1024 == 0, "stage alignment");

struct SumArgs {
  CUtensorMap tmK, tmV, tmDK, tmDV;   // 5D (64, Wg, Hg, T, BH), box (64, cw, ch, ct, 1)
  CUtensorMap tmS_hi, tmS_lo;         // 3D (64, R/64, BH*M) over the gradient planes, box (64, 64, 1)
  const __nv_bfloat16* dx_hi;         // gradient records (rows dz, dv read by cp.async)
  const __nv_bfloat16* dx_lo;
  int R, units;
  ChunkShape c;
  FastDiv f_head, f_nck;
  unsigned int* err;
};

__device__ __forceinline__ void sum_unit(const Plan& p, const SumArgs& a, int w, int& u, int& b, int& c) {
  const uint32_t uu = fdiv((uint32_t)w, a.f_head);
  const uint32_t rem = (uint32_t)w - uu * (uint32_t)(p.M * a.c.per_block);
  const uint32_t bb = fdiv(rem, a.f_nck);
  u = (int)uu;
  b = (int)bb;
  c = (int)(rem - bb * (uint32_t)a.c.per_block);
}

__global__ void __launch_bounds__(kThreads, 1) tc_bwd_summary_kernel(const __grid_constant__ SumArgs a, const Plan p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gb = smem_raw + (base - raw);
  const uint32_t bars = base + kBars;
  auto kvfull = [&](int s) { return bars + 8u * s; };
  auto kready = [&](int s) { return bars + 8u * (kStages + s); };
  auto mmadone = [&](int s) { return bars + 8u * (2 * kStages + s); };
  auto kvempty = [&](int s) { return bars + 8u * (3 * kStages + s); };
  auto bfull = [&](int x) { return bars + 8u * (4 * kStages + x); };
  auto bready = [&](int x) { return bars + 8u * (4 * kStages + kBStages + x); };
  auto bempty = [&](int x) { return bars + 8u * (4 * kStages + 2 * kBStages + x); };
  auto accempty = [&](int x) { return bars + 8u * (4 * kStages + 3 * kBStages + x); };
  auto accfull = [&](int x) { return bars + 8u * (4 * kStages + 3 * kBStages + 2 + x); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gb + kBars + 8 * kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gb + kBars + 8 * kNumBars + 8);
  auto kst = [&](int s) { return base + (uint32_t)s * kStageBytes; };
  auto bst = [&](int x) { return base + kBBase + (uint32_t)x * kBStageBytes; };

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int rows = a.c.rows;

  // ones tile (columns 0 and 1 of every row) and zeroed bias operands
  for (uint32_t off = threadIdx.x * 16u; off < kTile; off += kThreads * 16u) {
    const uint32_t r = off / 128u, chunk = (off % 128u) / 16u;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (chunk == (r & 7u)) v.x = 0x3F803F80u;  // logical chunk 0 = columns 0..7: columns 0, 1 = 1.0
    *reinterpret_cast<uint4*>(gb + kOnes + off) = v;
  }
  for (int x = 0; x < kBStages; ++x)
    for (uint32_t off = threadIdx.x * 16u; off < kBTile + 2048u; off += kThreads * 16u)
      *reinterpret_cast<uint4*>(gb + kBBase + x * kBStageBytes + kOffZk + off) = make_uint4(0u, 0u, 0u, 0u);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(kvfull(s), 1);
      mbar_init(kready(s), kXfThreads / 32);
      mbar_init(mmadone(s), 1);
      mbar_init(kvempty(s), 1);
    }
    for (int x = 0; x < kBStages; ++x) {
      mbar_init(bfull(x), 1);
      mbar_init(bready(x), 1);
      mbar_init(bempty(x), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(accempty(x), 1);
      mbar_init(accfull(x), 1);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&a.tmK);
    tma_prefetch_desc(&a.tmV);
    tma_prefetch_desc(&a.tmDK);
    tma_prefetch_desc(&a.tmDV);
  }
  if (warp == 2 && lane == 0) {
    tma_prefetch_desc(&a.tmS_hi);
    tma_prefetch_desc(&a.tmS_lo);
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
      // ------------------------------------------------ K, V tile producer
      const uint64_t pol = policy_evict_first();
      const uint32_t bytes = (uint32_t)rows * 128u;
      int s = 0;
      uint32_t ph = 0;
      long long issued = 0;
      for (int w = blockIdx.x; w < a.units; w += gridDim.x) {
        int u, b, c, x0, y0, t0;
        sum_unit(p, a, w, u, b, c);
        if (!mbar_wait(kvempty(s), ph ^ 1u, a.err, 0x701, abort_flag)) break;
        chunk_origin(p, a.c, (uint32_t)b, (uint32_t)c, x0, y0, t0);
        const TileCoords g5 = token_tile_coords(p, u, x0, y0, t0);
        mbar_arrive_expect_tx(kvfull(s), 2 * bytes);
        tma_load_5d(kst(s), &a.tmK, kvfull(s), g5.c[0], g5.c[1], g5.c[2], g5.c[3], g5.c[4], pol);
        tma_load_5d(kst(s) + kTile, &a.tmV, kvfull(s), g5.c[0], g5.c[1], g5.c[2], g5.c[3], g5.c[4], pol);
        ++issued;
        if (++s == kStages) {
          s = 0;
          ph ^= 1u;
        }
      }
      drain_loads(kvfull(0), kStages, issued, a.err, 0x702);
    }
  } else if (warp == 2) {
    // ------------------------------------------ gradient-record producer
    // lane 0: dS_b (hi, lo) by TMA; lanes 0-31: the dz_b, dv_b rows (hi:
    // lanes 0-15, lo: 16-31) by cp.async, 16 bytes each
    const uint64_t pol = policy_evict_last();
    int x = 0;
    uint32_t ph = 0;
    long long issued = 0;
    for (int w = blockIdx.x; w < a.units; w += gridDim.x) {
      int u, b, c;
      sum_unit(p, a, w, u, b, c);
      bool ok = true;
      if (lane == 0) ok = mbar_wait(bempty(x), ph ^ 1u, a.err, 0x703, abort_flag);
      if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
      const uint32_t st = bst(x);
      const int rec = u * p.M + b;
      const __nv_bfloat16* src = (lane < 16 ? a.dx_hi : a.dx_lo) + (size_t)rec * a.R + 64 * 64 + (lane & 15) * 8;
      cp_async16(st + kOffAux + (lane < 16 ? 0u : 256u) + (lane & 15) * 16, src);
      cp_async_arrive(bfull(x));
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_expect_tx(bfull(x), 2 * kBTile);
        tma_load_3d(st, &a.tmS_hi, bfull(x), 0, 0, rec, pol);
        tma_load_3d(st + kOffSlo, &a.tmS_lo, bfull(x), 0, 0, rec, pol);
      }
      ++issued;
      if (++x == kBStages) {
        x = 0;
        ph ^= 1u;
      }
    }
    if (lane == 0) drain_loads(bfull(0), kBStages, issued, a.err, 0x704);
  } else if (warp == 3) {
    // ------------------------------------------------- bias operands
    // Zk[k][0..1] = dz_b[k] hi, lo (K-major, 64 rows); Zv[0..1][c] = dv_b[c]
    // hi, lo (MN-major rows of the bias K step)
    int x = 0;
    uint32_t ph = 0;
    for (int w = blockIdx.x; w < a.units; w += gridDim.x) {
      const bool ok = mbar_wait(bfull(x), ph, a.err, 0x705, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) break;
      uint8_t* st = gb + kBBase + x * kBStageBytes;
      const __nv_bfloat16* aux = reinterpret_cast<const __nv_bfloat16*>(st + kOffAux);
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int k = lane + 32 * j;
        *reinterpret_cast<__nv_bfloat16*>(st + kOffZk + sw128_offset(k, 0)) = aux[k];          // dz hi
        *reinterpret_cast<__nv_bfloat16*>(st + kOffZk + sw128_offset(k, 1)) = aux[128 + k];    // dz lo
        *reinterpret_cast<__nv_bfloat16*>(st + kOffZv + sw128_offset(0, k)) = aux[64 + k];     // dv hi
        *reinterpret_cast<__nv_bfloat16*>(st + kOffZv + sw128_offset(1, k)) = aux[192 + k];    // dv lo
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
      const uint32_t id_k = idesc_bf16_f32(128, 64, false, false);  // D_K: B = dS K-major
      const uint32_t id_v = idesc_bf16_f32(128, 64, false, true);   // D_V: B = dS MN-major
      int s = 0, x = 0, acc = 0;
      uint32_t ph = 0, bph = 0, accph = 0;
      const uint32_t ones = base + kOnes;
      for (int w = blockIdx.x; w < a.units; w += gridDim.x) {
        if (!mbar_wait(kready(s), ph, a.err, 0x706, abort_flag)) break;
        if (!mbar_wait(bready(x), bph, a.err, 0x707, abort_flag)) break;
        if (!mbar_wait(accempty(acc), accph ^ 1u, a.err, 0x708, abort_flag)) break;
        tc_fence_after();
        const uint32_t ks_ = kst(s), phi_hi = ks_, vt = ks_ + kTile, phi_lo = ks_ + 2 * kTile;
        const uint32_t bs = bst(x);
        const uint32_t dK = tmem + (uint32_t)acc * 128u, dV = dK + 64u;
        // descriptors of K step 0, advanced by adding byte offset / 16 to the
        // address field (the issue of each MMA waits for the tensor pipe, so
        // every instruction on this thread adds to the unit's time)
        const uint64_t v0 = sdesc_sw128(vt, 0u, 1024u), b0 = sdesc_sw128(bs, 0u, 1024u);
        const uint64_t bl0 = sdesc_sw128(bs + kOffSlo, 0u, 1024u);
        const uint64_t h0 = sdesc_sw128(phi_hi, 0u, 1024u), l0 = sdesc_sw128(phi_lo, 0u, 1024u);
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
          // D_K += V dS^T (B K-major: rows k, 16 c per step; + 32 bytes per step)
          const uint64_t av = v0 + 2 * k4;
          umma_bf16(dK, av, b0 + 2 * k4, id_k, k4 > 0 ? 1u : 0u);
          umma_bf16(dK, av, bl0 + 2 * k4, id_k, 1u);
          // D_V += phi(K) dS (B MN-major: 16 k rows per step, + 2048 bytes)
          const uint64_t ah = h0 + 2 * k4, bh = b0 + 128 * k4;
          umma_bf16(dV, ah, bh, id_v, k4 > 0 ? 1u : 0u);
          umma_bf16(dV, ah, bl0 + 128 * k4, id_v, 1u);
          umma_bf16(dV, l0 + 2 * k4, bh, id_v, 1u);
        }
        // bias K step: ones columns 0, 1 against (dz hi, lo) and (dv hi, lo)
        const uint64_t a1 = sdesc_sw128(ones, 0u, 1024u);
        umma_bf16(dK, a1, sdesc_sw128(bs + kOffZk, 0u, 1024u), id_k, 1u);
        umma_bf16(dV, a1, sdesc_sw128(bs + kOffZv, 0u, 1024u), id_v, 1u);
        umma_commit(mmadone(s));
        umma_commit(bempty(x));
        umma_commit(accfull(acc));
        if (++s == kStages) {
          s = 0;
          ph ^= 1u;
        }
        if (++x == kBStages) {
          x = 0;
          bph ^= 1u;
        }
        if (++acc == 2) {
          acc = 0;
          accph ^= 1u;
        }
      }
    }
  } else if (warp >= 4 && warp < 12) {
    // ----------------------------------------- phi(K): high part in place, low part aside
    const int t = threadIdx.x - 128;
    const int row = t >> 1;
    const int half = t & 1;
    int s = 0;
    uint32_t ph = 0;
    for (int w = blockIdx.x; w < a.units; w += gridDim.x) {
      const bool ok = mbar_wait(kvfull(s), ph, a.err, 0x709, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) break;
      if (row < rows) {
        uint8_t* rp = gb + s * kStageBytes + row * 128;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t off = ((4 * half + j + row) & 7) << 4;
          uint4 x = *reinterpret_cast<const uint4*>(rp + off), lo;
          uint32_t* xp = &x.x;
          uint32_t* lp = &lo.x;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float2 f = bf16x2_to_float2(xp[q]);
            const float f0 = phi_map(f.x, p.fmap), f1 = phi_map(f.y, p.fmap);
            xp[q] = pack_bf16x2(f0, f1);
            const float2 g = bf16x2_to_float2(xp[q]);
            lp[q] = pack_bf16x2(f0 - g.x, f1 - g.y);
          }
          *reinterpret_cast<uint4*>(rp + off) = x;
          *reinterpret_cast<uint4*>(rp + 2 * kTile + off) = lo;
        }
      }
      fence_proxy_async();
      mbar_arrive_warp(kready(s));
      if (++s == kStages) {
        s = 0;
        ph ^= 1u;
      }
    }
  } else if (warp >= 12) {
    // ------------------------------------------------------------ epilogue
    const int q4 = warp & 3;
    const int t = 32 * q4 + lane;   // token row = TMEM lane
    const int et = threadIdx.x - 384;
    int s = 0, acc = 0, n_out = 0;
    uint32_t ph = 0, accph = 0;
    for (int w = blockIdx.x; w < a.units; w += gridDim.x) {
      int u, b, c;
      sum_unit(p, a, w, u, b, c);
      bool ok = mbar_wait(accfull(acc), accph, a.err, 0x70a, abort_flag);
      ok = ok && mbar_wait(mmadone(s), ph, a.err, 0x70b, abort_flag);
      if (!named_all(4, kEpiThreads, ok)) break;
      tc_fence_after();
      const uint32_t taddr = tmem + (uint32_t)acc * 128u + ((uint32_t)(32 * q4) << 16);
      uint8_t* rk = gb + s * kStageBytes + t * 128;   // phi(K) hi -> dK
      uint8_t* rv = rk + kTile;                       // V -> dV
      const uint8_t* rl = rk + 2 * kTile;             // phi(K) lo
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        float gk[32], gv[32];
        tmem_ld32(taddr + 32u * h, gk);
        tmem_ld32(taddr + 64u + 32u * h, gv);
        tmem_wait_ld();
        if (t < rows) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t off = (uint32_t)((((4 * h + j) ^ t) & 7) << 4);
            uint4 xh = *reinterpret_cast<const uint4*>(rk + off);
            const uint4 xl = *reinterpret_cast<const uint4*>(rl + off);
            uint4 ov;
            const uint32_t* hp = &xh.x;
            const uint32_t* lp = &xl.x;
            uint32_t* kp = &xh.x;
            uint32_t* vp = &ov.x;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int cc = 8 * j + 2 * q;
              const float2 fh = bf16x2_to_float2(hp[q]), fl = bf16x2_to_float2(lp[q]);
              const float d0 = phi_deriv_from_phi(fh.x, fl.x, p.fmap);
              const float d1 = phi_deriv_from_phi(fh.y, fl.y, p.fmap);
              kp[q] = pack_bf16x2(gk[cc] * d0, gk[cc + 1] * d1);
              vp[q] = pack_bf16x2(gv[cc], gv[cc + 1]);
            }
            *reinterpret_cast<uint4*>(rk + off) = xh;
            *reinterpret_cast<uint4*>(rv + off) = ov;
          }
        }
      }
      fence_proxy_async();
      tc_fence_before();
      named_sync(4, kEpiThreads);
      if (et == 0) {
        mbar_arrive(accempty(acc));
        int x0, y0, t0;
        chunk_origin(p, a.c, (uint32_t)b, (uint32_t)c, x0, y0, t0);
        const TileCoords g5 = token_tile_coords(p, u, x0, y0, t0);
        tma_store_5d(&a.tmDK, kst(s), g5.c[0], g5.c[1], g5.c[2], g5.c[3], g5.c[4]);
        tma_store_5d(&a.tmDV, kst(s) + kTile, g5.c[0], g5.c[1], g5.c[2], g5.c[3], g5.c[4]);
        bulk_commit();
        bulk_wait_read<kPendStores - 1>();
        if (n_out >= kPendStores - 1) mbar_arrive(kvempty((s + kStages - (kPendStores - 1)) % kStages));
      }
      ++n_out;
      if (++s == kStages) {
        s = 0;
        ph ^= 1u;
      }
      if (++acc == 2) {
        acc = 0;
        accph ^= 1u;
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

int launch_tc_bwd_summary(const Plan& p, const void* k, const void* v, const __nv_bfloat16* dx_hi,
                          const __nv_bfloat16* dx_lo, void* dk, void* dv, cudaStream_t s) {
  SumArgs a;
  memset(&a, 0, sizeof(a));
  const ChunkShape& c = p.chunk;
  int e;
  if ((e = encode_token_map(&a.tmK, p, k, c)) != 0) return e;
  if ((e = encode_token_map(&a.tmV, p, v, c)) != 0) return e;
  if ((e = encode_token_map(&a.tmDK, p, dk, c)) != 0) return e;
  if ((e = encode_token_map(&a.tmDV, p, dv, c)) != 0) return e;
  const uint64_t dims3[3] = {64, (uint64_t)(p.R / 64), (uint64_t)p.BH * p.M};
  const uint64_t str3[2] = {128, 2ull * p.R};
  const uint32_t box3[3] = {64, 64, 1};
  if ((e = encode_tmap_bf16(&a.tmS_hi, dx_hi, 3, dims3, str3, box3)) != 0) return e;
  if ((e = encode_tmap_bf16(&a.tmS_lo, dx_lo, 3, dims3, str3, box3)) != 0) return e;
  a.dx_hi = dx_hi;
  a.dx_lo = dx_lo;
  a.R = p.R;
  a.units = p.BH * p.M * c.per_block;
  a.f_head = make_fastdiv((uint32_t)(p.M * c.per_block));
  a.f_nck = make_fastdiv((uint32_t)c.per_block);
  a.c = c;
  a.err = p.err;
  cudaError_t ce =
      (cudaError_t)set_max_dynamic_smem((const void*)tc_bwd_summary_kernel, (int)kSmemBytes);
  if (ce != cudaSuccess) return (int)ce;
  const int grid = a.units < num_sms() ? a.units : num_sms();
  tc_bwd_summary_kernel<<<grid, kThreads, kSmemBytes, s>>>(a, p);
  return (int)cudaGetLastError();
}

}  // namespace mhla
