// Block-ordered causal output step on the tensor cores (head dimension 64,
// bf16 tensors).
//
// Query t of block i sees the earlier blocks through the strict lower
// triangle of Mc and its own block up to itself through w = Mc[i, i] (the
// block-ordered reading of "MHLA: Restoring Expressivity of Linear Attention
// via Token-Level Multi-Head", key design 2 and its chunkwise remarks).  One
// CTA walks the token chunks of one block in order (each chunk a contiguous
// run of the block's local order); with P = phi(Q_c), F = phi(K_c):
//   prefix  D_a  = P [S_state | Z_state]            (N = 80: numerator, s)
//   scores  D_s  = P F^T                             (N = 128)
//   intra   P~   = w * mask(D_s)  (j <= t; bf16)     rows summed in float32
//           D_a += P~ V                              (numerator columns)
//   MALA    D_v  = L V,  L = lower-triangular ones   (in-chunk prefix of V)
//   state   D_u += F^T [V | 1]  (+ ones rows: sum V) for the next chunk:
//           S_state = S<_i + w * D_u  (bf16 high + low planes)
// where S<_i, z<_i, v<_i, n<_i are the records mixed with the strict lower
// triangle (high + low planes).  Then
//   s = D_a[64] + D_a[66] + rowsum(P~),  DIVISIVE o = num / s,  NONE o = num,
//   MALA o = (1 + 1/s) num - (s / n~_t) v~_t,  v~_t = v_state + w D_v[t],
//   n~_t = n_state + w (t + 1);  s = 0 gives o = 0.
// Each CTA (128 threads, one row per thread) runs the chunk's phases in turn;
// two CTAs share an SM so that one's MMAs overlap the other's epilogues.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstring>

#include "common.cuh"
#include "tc_causal.h"
#include "tc_common.cuh"

namespace mhla {
namespace {

using namespace tc;

constexpr int kThreads = 128;
constexpr uint32_t kTile = 128 * 128;   // 128 rows x 64 bf16
constexpr uint32_t kBTile = 64 * 128;   // 64 rows x 64 bf16
// shared memory (offsets from the 1024-aligned base)
constexpr uint32_t kOffQ = 0;                    // Q -> P -> O
constexpr uint32_t kOffK = kTile;                // K -> F
constexpr uint32_t kOffV = 2 * kTile;            // V
constexpr uint32_t kOffPt = 3 * kTile;           // P~: two K-major atoms (j 0..63, 64..127)
constexpr uint32_t kOffSt = 5 * kTile;           // state: S hi | S lo | Z (3 x 8 KB)
constexpr uint32_t kOffOnes = kOffSt + 3 * kBTile;  // 16 rows of ones (bias atoms of the state MMA)
constexpr uint32_t kOffZst = kOffOnes + 2048;    // z_state, 64 floats
constexpr uint32_t kOffBars = kOffZst + 256;     // load barrier, MMA barrier, abort flag, TMEM slot
constexpr uint32_t kSmemBytes = kOffBars + 32 + 1024;
constexpr uint32_t kTmemCols = 256;
// TMEM columns: D_a 0..79; D_s 128..255, reused by D_u 128..207 once read
constexpr uint32_t kColA = 0, kColS = 128, kColU = 128;
static_assert(kSmemBytes <= 232448 / 2, "two CTAs per SM");
static_assert(kOffSt % 1024 == 0 && kOffOnes % 1024 == 0, "alignment");

struct CausalArgs {
  CUtensorMap tmQ, tmK, tmV, tmO;   // token maps (encode_token_map)
  CUtensorMap tmS_hi, tmS_lo;       // 3D (64, R/64, BH*M) over the prefix-mixed planes, box (64, 64, 1)
  const __nv_bfloat16* mixed_hi;    // prefix-mixed records (z< rows read directly)
  const __nv_bfloat16* mixed_lo;
  const float* mc;                  // Mc (its diagonal weighs the block's own tokens)
  int R;
  ChunkShape c;
  unsigned int* err;
};

// all threads agree whether a bounded wait succeeded
__device__ __forceinline__ bool wait_all(uint32_t bar, uint32_t parity, unsigned int* err, unsigned int where,
                                         volatile int* abort_flag) {
  const bool ok = mbar_wait(bar, parity, err, where, abort_flag);
  return !__syncthreads_or(ok ? 0 : 1);
}

// Writes this thread's state rows k (< 64): S = hi + lo split again, and the
// Z bias row (z hi, z hi, z lo) of the same k.
__device__ __forceinline__ void put_z_row(uint8_t* gb, int k, float z) {
  const __nv_bfloat16 zh = __float2bfloat16_rn(z);
  const __nv_bfloat16 zl = __float2bfloat16_rn(z - __bfloat162float(zh));
  uint8_t* zt = gb + kOffSt + 2 * kBTile;
  *reinterpret_cast<__nv_bfloat16*>(zt + sw128_offset(k, 0)) = zh;
  *reinterpret_cast<__nv_bfloat16*>(zt + sw128_offset(k, 1)) = zh;
  *reinterpret_cast<__nv_bfloat16*>(zt + sw128_offset(k, 2)) = zl;
}

__global__ void __launch_bounds__(kThreads, 2) tc_causal_kernel(const __grid_constant__ CausalArgs a, const Plan p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gb = smem_raw + (base - raw);
  const uint32_t bar_ld = base + kOffBars, bar_mma = base + kOffBars + 8;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gb + kOffBars + 16);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gb + kOffBars + 24);
  float* zst = reinterpret_cast<float*>(gb + kOffZst);
  const int t = threadIdx.x;
  const int warp = t / 32;
  const int u = blockIdx.y, i = blockIdx.x;
  const int rows = a.c.rows, rows_pad = a.c.rows_pad, nck = a.c.per_block;
  const float w = a.mc[((size_t)mc_index(p, u) * p.M + i) * p.M + i];

  // zero every tile (rows past a chunk stay finite), ones rows for the state MMA
  for (uint32_t off = t * 16u; off < kOffOnes; off += kThreads * 16u)
    *reinterpret_cast<uint4*>(gb + off) = make_uint4(0u, 0u, 0u, 0u);
  for (uint32_t off = t * 16u; off < 2048u; off += kThreads * 16u)
    *reinterpret_cast<uint4*>(gb + kOffOnes + off) = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
  if (t == 0) {
    mbar_init(bar_ld, 1);
    mbar_init(bar_mma, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  fence_proxy_async();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t ta = tmem + ((uint32_t)(32 * warp) << 16);   // this warp's TMEM lanes
  uint32_t ph_ld = 0, ph_mma = 0;
  bool ok = true;

  // ------------------------------------------- prefix record S<_i, z<_i
  const int rec = u * p.M + i;
  if (t == 0) {
    mbar_arrive_expect_tx(bar_ld, 2 * kBTile);
    tma_load_3d(base + kOffSt, &a.tmS_hi, bar_ld, 0, 0, rec, policy_evict_first());
    tma_load_3d(base + kOffSt + kBTile, &a.tmS_lo, bar_ld, 0, 0, rec, policy_evict_first());
  }
  if (t < 64) {
    const size_t zo = (size_t)rec * a.R + 64 * 64 + t;
    zst[t] = __bfloat162float(a.mixed_hi[zo]) + __bfloat162float(a.mixed_lo[zo]);
    put_z_row(gb, t, zst[t]);
  }
  ok = wait_all(bar_ld, ph_ld, a.err, 0x901, abort_flag);
  ph_ld ^= 1u;

  const uint32_t id_a = idesc_bf16_f32(128, 80, false, true);
  const uint32_t id_a64 = idesc_bf16_f32(128, 64, false, true);
  const uint32_t id_s = idesc_bf16_f32(128, 128, false, false);
  const uint32_t id_v = idesc_bf16_f32(128, 64, false, true);
  const uint32_t id_u = idesc_bf16_f32(128, 80, true, true);
  const uint32_t q_s = base + kOffQ, k_s = base + kOffK, v_s = base + kOffV, pt_s = base + kOffPt;
  const uint32_t sh = base + kOffSt, sl = sh + kBTile, zt = sh + 2 * kBTile, ones = base + kOffOnes;

  for (int c = 0; c < nck && ok; ++c) {
    int x0, y0, t0;
    chunk_origin(p, a.c, (uint32_t)i, (uint32_t)c, x0, y0, t0);
    const TileCoords g5 = token_tile_coords(p, u, x0, y0, t0);
    // ------------------------------------------------------ loads
    if (t == 0) {
      bulk_wait_read<0>();   // the previous chunk's output has left the Q tile
      const uint32_t bytes = (uint32_t)rows * 128u;
      const uint64_t pol = policy_evict_first();
      mbar_arrive_expect_tx(bar_ld, 3 * bytes);
      tma_load_5d(q_s, &a.tmQ, bar_ld, g5.c[0], g5.c[1], g5.c[2], g5.c[3], g5.c[4], pol);
      tma_load_5d(k_s, &a.tmK, bar_ld, g5.c[0], g5.c[1], g5.c[2], g5.c[3], g5.c[4], pol);
      tma_load_5d(v_s, &a.tmV, bar_ld, g5.c[0], g5.c[1], g5.c[2], g5.c[3], g5.c[4], pol);
    }
    if (!(ok = wait_all(bar_ld, ph_ld, a.err, 0x902, abort_flag))) break;
    ph_ld ^= 1u;
    // ---------------------------------------- P = phi(Q), F = phi(K)
    {
      uint8_t* qr = gb + kOffQ + t * 128;
      uint8_t* kr = gb + kOffK + t * 128;
      if (t < rows) {
#pragma unroll 2
        for (int j = 0; j < 8; ++j) {
          const uint32_t off = (uint32_t)(j << 4);
          uint4 xq = *reinterpret_cast<const uint4*>(qr + off), xk = *reinterpret_cast<const uint4*>(kr + off);
          uint32_t* pq = &xq.x;
          uint32_t* pk = &xk.x;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 fq = bf16x2_to_float2(pq[e]), fk = bf16x2_to_float2(pk[e]);
            pq[e] = pack_bf16x2(phi_map(fq.x, p.fmap), phi_map(fq.y, p.fmap));
            pk[e] = pack_bf16x2(phi_map(fk.x, p.fmap), phi_map(fk.y, p.fmap));
          }
          *reinterpret_cast<uint4*>(qr + off) = xq;
          *reinterpret_cast<uint4*>(kr + off) = xk;
        }
      } else if (t < rows_pad) {
        for (int j = 0; j < 8; ++j) {
          *reinterpret_cast<uint4*>(qr + (j << 4)) = make_uint4(0u, 0u, 0u, 0u);
          *reinterpret_cast<uint4*>(kr + (j << 4)) = make_uint4(0u, 0u, 0u, 0u);
        }
      }
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    // --------------------------------------------- MMA: prefix, scores
    if (t == 0) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        const uint64_t ap = sdesc_sw128(q_s + (uint32_t)ks * 32u, 0u, 1024u);
        umma_bf16(tmem + kColA, ap, sdesc_sw128(sh + (uint32_t)ks * 2048u, zt - sh, 1024u), id_a, ks > 0 ? 1u : 0u);
        umma_bf16(tmem + kColA, ap, sdesc_sw128(sl + (uint32_t)ks * 2048u, 0u, 1024u), id_a64, 1u);
        umma_bf16(tmem + kColS, ap, sdesc_sw128(k_s + (uint32_t)ks * 32u, 0u, 1024u), id_s, ks > 0 ? 1u : 0u);
      }
      umma_commit(bar_mma);
    }
    if (!(ok = wait_all(bar_mma, ph_mma, a.err, 0x903, abort_flag))) break;
    ph_mma ^= 1u;
    tc_fence_after();
    // ------------------------------ P~ = w mask(D_s), its row sums
    float rsum = 0.f;
    {
      uint8_t* prow = gb + kOffPt + t * 128;
#pragma unroll 1
      for (int h = 0; h < 4; ++h) {
        float sc[32];
        tmem_ld32(ta + kColS + 32u * h, sc);
        tmem_wait_ld();
        uint8_t* atom = prow + (h >> 1) * kTile;   // j 0..63 -> atom 0, 64..127 -> atom 1
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4 pk;
          uint32_t* pp = &pk.x;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j0 = 32 * h + 8 * q + 2 * e;
            const float v0 = (j0 <= t && t < rows) ? w * sc[8 * q + 2 * e] : 0.f;
            const float v1 = (j0 + 1 <= t && t < rows) ? w * sc[8 * q + 2 * e + 1] : 0.f;
            rsum += v0 + v1;
            pp[e] = pack_bf16x2(v0, v1);
          }
          const int chunk = ((h & 1) * 4 + q);   // logical 16-byte chunk in the atom row
          *reinterpret_cast<uint4*>(atom + (((chunk ^ t) & 7) << 4)) = pk;
        }
      }
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    // -------------------------------------- MMA: intra, state update
    const bool more = c + 1 < nck;
    if (t == 0) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t ao = (uint32_t)(ks >> 2) * kTile + (uint32_t)(ks & 3) * 32u;
        umma_bf16(tmem + kColA, sdesc_sw128(pt_s + ao, 0u, 1024u), sdesc_sw128(v_s + (uint32_t)ks * 2048u, 0u, 1024u),
                  id_v, 1u);
      }
      if (more) {
        // D_u = F^T [V | 1] over this chunk's tokens (the summary's form)
        for (int kt = 0; kt < rows_pad / 16; ++kt) {
          const uint32_t fa = k_s + (uint32_t)kt * 2048u, va = v_s + (uint32_t)kt * 2048u;
          umma_bf16(tmem + kColU, sdesc_sw128(fa, ones - fa, 1024u), sdesc_sw128(va, ones - va, 1024u), id_u,
                    kt > 0 ? 1u : 0u);
        }
      }
      umma_commit(bar_mma);
    }
    if (!(ok = wait_all(bar_mma, ph_mma, a.err, 0x904, abort_flag))) break;
    ph_mma ^= 1u;
    tc_fence_after();
    // ------------------------------------------------------ output
    {
      float nm[32], zc[16];
      tmem_ld16(ta + kColA + 64u, zc);
      tmem_wait_ld();
      const float s = zc[0] + zc[2] + rsum;
      float scale = 1.f;
      if (p.norm == MHLA_NORM_DIVISIVE) scale = s != 0.f ? 1.f / s : 0.f;
      uint8_t* orow = gb + kOffQ + t * 128;
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        tmem_ld32(ta + kColA + 32u * h, nm);
        tmem_wait_ld();
        if (t < rows) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 ov;
            uint32_t* op = &ov.x;
#pragma unroll
            for (int e = 0; e < 4; ++e) op[e] = pack_bf16x2(nm[8 * q + 2 * e] * scale, nm[8 * q + 2 * e + 1] * scale);
            *reinterpret_cast<uint4*>(orow + ((((4 * h + q) ^ t) & 7) << 4)) = ov;
          }
        }
      }
    }
    // ------------------------------------ state for the next chunk
    if (more && warp < 2) {
      float dv[32], zc[16];
      uint8_t* shr = gb + kOffSt + t * 128;
      uint8_t* slr = shr + kBTile;
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        tmem_ld32(ta + kColU + 32u * h, dv);
        tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t off = (uint32_t)((((4 * h + q) ^ t) & 7) << 4);
          uint4 hv = *reinterpret_cast<const uint4*>(shr + off), lv = *reinterpret_cast<const uint4*>(slr + off);
          uint32_t* hp = &hv.x;
          uint32_t* lp = &lv.x;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 fh = bf16x2_to_float2(hp[e]), fl = bf16x2_to_float2(lp[e]);
            const float y0 = fh.x + fl.x + w * dv[8 * q + 2 * e], y1 = fh.y + fl.y + w * dv[8 * q + 2 * e + 1];
            hp[e] = pack_bf16x2(y0, y1);
            const float2 g = bf16x2_to_float2(hp[e]);
            lp[e] = pack_bf16x2(y0 - g.x, y1 - g.y);
          }
          *reinterpret_cast<uint4*>(shr + off) = hv;
          *reinterpret_cast<uint4*>(slr + off) = lv;
        }
      }
      tmem_ld16(ta + kColU + 64u, zc);
      tmem_wait_ld();
      zst[t] += w * zc[0];
      put_z_row(gb, t, zst[t]);
    } else if (more) {
      // warps 2, 3 hold TMEM lanes 64..127 of D_u (the ones rows): nothing to keep
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    if (t == 0) {
      tma_store_5d(&a.tmO, q_s, g5.c[0], g5.c[1], g5.c[2], g5.c[3], g5.c[4]);
      bulk_commit();
    }
  }
  if (t == 0) bulk_wait<0>();
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace
}  // namespace mhla

namespace mhla {

bool tc_causal_supported(const Plan& p) {
  const ChunkShape& c = p.chunk;
  // every chunk must be a contiguous run of the block's local (raster) order
  const bool run = (c.ct == 1 && c.ch == 1) || (c.cw == p.bw && c.ct == 1) || (c.cw == p.bw && c.ch == p.bh);
  return run && p.norm != MHLA_NORM_MALA;
}

int launch_tc_causal(const Plan& p, const void* q, const void* k, const void* v, const __nv_bfloat16* mixed_hi,
                     const __nv_bfloat16* mixed_lo, const float* mc, void* out, cudaStream_t s) {
  CausalArgs a;
  memset(&a, 0, sizeof(a));
  const ChunkShape& c = p.chunk;
  int e;
  if ((e = encode_token_map(&a.tmQ, p, q, c)) != 0) return e;
  if ((e = encode_token_map(&a.tmK, p, k, c)) != 0) return e;
  if ((e = encode_token_map(&a.tmV, p, v, c)) != 0) return e;
  if ((e = encode_token_map(&a.tmO, p, out, c)) != 0) return e;
  const uint64_t dims3[3] = {64, (uint64_t)(p.R / 64), (uint64_t)p.BH * p.M};
  const uint64_t str3[2] = {128, 2ull * p.R};
  const uint32_t box3[3] = {64, 64, 1};
  if ((e = encode_tmap_bf16(&a.tmS_hi, mixed_hi, 3, dims3, str3, box3)) != 0) return e;
  if ((e = encode_tmap_bf16(&a.tmS_lo, mixed_lo, 3, dims3, str3, box3)) != 0) return e;
  a.mixed_hi = mixed_hi;
  a.mixed_lo = mixed_lo;
  a.mc = mc;
  a.R = p.R;
  a.c = c;
  a.err = p.err;
  cudaError_t ce = cudaFuncSetAttribute(tc_causal_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (ce != cudaSuccess) return (int)ce;
  tc_causal_kernel<<<dim3(p.M, p.BH), kThreads, kSmemBytes, s>>>(a, p);
  return (int)cudaGetLastError();
}

}  // namespace mhla
