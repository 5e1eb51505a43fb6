// Output step on the tensor cores ("MHLA: Restoring Expressivity of Linear
// Attention via Token-Level Multi-Head", flowchart output node and key design
// 2; "Rectifying Magnitude Neglect in Linear Attention", key designs).
//
// For a token tile of query block i (up to 128 tokens, gathered by one TMA box
// from the token grid):
//     D = phi(Q_tile) S~_i            (tcgen05, M = 128 tokens, N = 64, K = 64)
//     s_t = phi(q_t) . z~_i           (CUDA cores, while phi is applied)
//   DIVISIVE o = D / s,  NONE o = D,
//   MALA     o = (1 + 1/s) D - (s / n~_i) v~_i,   n~_i = n_b sum_b Mc[i, b]
// then the bf16 result overwrites the Q tile in shared memory and one TMA
// store scatters it back to the grid positions of the tile.
//   A = phi(Q) tile: K-major (features contiguous), as TMA delivered it
//   B = S~_i: MN-major ([k][c], c contiguous), loaded by TMA from the mixed
//       stack (bf16 high part; MALA adds the low residual as a second MMA)
// Persistent, warp-specialised CTA (384 threads): warp 0 TMA producer,
// warp 1 TMEM + MMA, warps 4-7 phi + denominators, warps 8-11 epilogue.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstring>

#include "common.cuh"
#include "tc_common.cuh"
#include "tc_host.h"

namespace mhla {
namespace {

using namespace tc;

constexpr int kStages = 4;
constexpr int kThreads = 384;
constexpr uint32_t kQTile = 128 * 128;           // Q / O tile
constexpr uint32_t kBTile = 64 * 128;            // S~_i, 64 k-rows x 64 c
constexpr uint32_t kOffBhi = kQTile;
constexpr uint32_t kOffBlo = kQTile + kBTile;
constexpr uint32_t kOffDen = kQTile + 2 * kBTile;  // 128 floats
constexpr uint32_t kOffZ = kOffDen + 512;          // z~ (64 floats)
constexpr uint32_t kOffV = kOffZ + 256;            // v~ (64 floats)
constexpr uint32_t kStageBytes = 34 * 1024;
constexpr uint32_t kBars = kStages * kStageBytes;
constexpr uint32_t kSmemBytes = kBars + 256 + 1024;
constexpr uint32_t kTmemCols = 256;              // one 64-column accumulator per stage

static_assert(kOffV + 256 <= kStageBytes, "stage layout overflow");

struct OutArgs {
  CUtensorMap tmQ, tmO;        // 5D (64, Wg, Hg, T, BH), box (64, cw, ch, ct, 1)
  CUtensorMap tmB_hi, tmB_lo;  // 3D (64, R/64, BH*M), box (64, 64, 1)
  const __nv_bfloat16* mixed_hi;
  const __nv_bfloat16* mixed_lo;
  const float* rowsum;
  int units;
  int use_lo;
  ChunkShape c;
  unsigned int* err;
};

__device__ __forceinline__ float phi_fast(float x, int fmap) {
  if (fmap == MHLA_FEATURE_IDENTITY) return x;
  return x > 0.f ? x + 1.f : __expf(x);
}

__global__ void __launch_bounds__(kThreads, 1) tc_output_kernel(const __grid_constant__ OutArgs a, const Plan p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gb = smem_raw + (base - raw);
  const uint32_t bars = base + kBars;
  auto full = [&](int s) { return bars + 8u * s; };
  auto tready = [&](int s) { return bars + 8u * (kStages + s); };
  auto mmadone = [&](int s) { return bars + 8u * (2 * kStages + s); };
  auto empty = [&](int s) { return bars + 8u * (3 * kStages + s); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gb + kBars + 8 * (4 * kStages));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gb + kBars + 8 * (4 * kStages) + 8);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int rows = a.c.rows;
  const int nck = a.c.per_block;
  const int per_head = p.M * nck;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(tready(s), 128);
      mbar_init(mmadone(s), 1);
      mbar_init(empty(s), 1);
    }
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
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------- producer
      const uint64_t pol_q = policy_evict_first();
      const uint64_t pol_b = policy_evict_last();
      const uint32_t bytes = (uint32_t)rows * 128u + kBTile * (a.use_lo ? 2u : 1u);
      int stage = 0;
      uint32_t phase = 0;
      for (int w = blockIdx.x; w < a.units; w += gridDim.x) {
        if (!mbar_wait(empty(stage), phase ^ 1u, a.err, 0x301, abort_flag)) break;
        const int u = w / per_head;
        const int rem = w % per_head;
        const int i = rem / nck;
        const int c = rem % nck;
        const int bx = i % p.Mw, by = (i / p.Mw) % p.Mh, bz = i / (p.Mw * p.Mh);
        const int x0 = bx * p.bw + (c % a.c.ncx) * a.c.cw;
        const int y0 = by * p.bh + ((c / a.c.ncx) % a.c.ncy) * a.c.ch;
        const int t0 = bz * p.bt + (c / (a.c.ncx * a.c.ncy)) * a.c.ct;
        const uint32_t st = base + (uint32_t)stage * kStageBytes;
        mbar_arrive_expect_tx(full(stage), bytes);
        tma_load_5d(st, &a.tmQ, full(stage), 0, x0, y0, t0, u, pol_q);
        tma_load_3d(st + kOffBhi, &a.tmB_hi, full(stage), 0, 0, u * p.M + i, pol_b);
        if (a.use_lo) tma_load_3d(st + kOffBlo, &a.tmB_lo, full(stage), 0, 0, u * p.M + i, pol_b);
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // --------------------------------------------------------------- MMA
      const uint32_t idesc = idesc_bf16_f32(128, 64, false, true);
      int stage = 0;
      uint32_t phase = 0;
      for (int w = blockIdx.x; w < a.units; w += gridDim.x) {
        if (!mbar_wait(tready(stage), phase, a.err, 0x302, abort_flag)) break;
        tc_fence_after();
        const uint32_t st = base + (uint32_t)stage * kStageBytes;
        const uint32_t d = tmem + (uint32_t)stage * 64u;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint64_t ad = sdesc_sw128(st + (uint32_t)ks * 32u, 0u, 1024u);
          umma_bf16(d, ad, sdesc_sw128(st + kOffBhi + (uint32_t)ks * 2048u, kBTile, 1024u), idesc, ks > 0 ? 1u : 0u);
          if (a.use_lo) umma_bf16(d, ad, sdesc_sw128(st + kOffBlo + (uint32_t)ks * 2048u, kBTile, 1024u), idesc, 1u);
        }
        umma_commit(mmadone(stage));
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------- phi(Q) and denominators
    const int t = threadIdx.x - 128;
    int stage = 0;
    uint32_t phase = 0;
    for (int w = blockIdx.x; w < a.units; w += gridDim.x) {
      const int u = w / per_head;
      const int i = (w % per_head) / nck;
      // z~_i (threads 0..63) and v~_i (threads 64..127), hi + lo parts
      const size_t aux = ((size_t)u * p.M + i) * p.R + (size_t)p.d * p.d + t;
      const float zv = __bfloat162float(a.mixed_hi[aux]) + __bfloat162float(a.mixed_lo[aux]);
      const bool ok = mbar_wait(full(stage), phase, a.err, 0x303, abort_flag);
      if (!named_all(2, 128, ok)) break;
      uint8_t* st = gb + stage * kStageBytes;
      float* zs = reinterpret_cast<float*>(st + kOffZ);  // z at [0,64), v at [64,128)
      zs[t] = zv;
      named_sync(4, 128);
      if (t < rows) {
        uint8_t* row = st + t * 128;
        float s = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          uint4* ptr = reinterpret_cast<uint4*>(row + (((j ^ t) & 7) << 4));
          uint4 x = *ptr;
          uint32_t* xp = &x.x;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&xp[q]);
            float2 f = __bfloat1622float2(h);
            xp[q] = pack_bf16x2(phi_fast(f.x, p.fmap), phi_fast(f.y, p.fmap));
            float2 g = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&xp[q]));
            s = fmaf(g.x, zs[8 * j + 2 * q], s);
            s = fmaf(g.y, zs[8 * j + 2 * q + 1], s);
          }
          *ptr = x;
        }
        reinterpret_cast<float*>(st + kOffDen)[t] = s;
      }
      fence_proxy_async();
      mbar_arrive(tready(stage));
      if (++stage == kStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
  } else if (warp >= 8) {
    // ------------------------------------------------------------ epilogue
    const int e = warp - 8;
    const int t = threadIdx.x - 256;  // token row = TMEM lane
    int stage = 0, prev = -1;
    uint32_t phase = 0;
    for (int w = blockIdx.x; w < a.units; w += gridDim.x) {
      const int u = w / per_head;
      const int rem = w % per_head;
      const int i = rem / nck;
      const int c = rem % nck;
      bool ok = mbar_wait(mmadone(stage), phase, a.err, 0x304, abort_flag);
      // the transform's shared-memory writes (denominators, z~, v~)
      ok = ok && mbar_wait(tready(stage), phase, a.err, 0x305, abort_flag);
      if (!named_all(3, 128, ok)) break;
      tc_fence_after();
      float o0[32], o1[32];
      const uint32_t taddr = tmem + (uint32_t)stage * 64u + ((uint32_t)(32 * e) << 16);
      tmem_ld32(taddr, o0);
      tmem_ld32(taddr + 32u, o1);
      tmem_wait_ld();
      uint8_t* st = gb + stage * kStageBytes;
      if (t < rows) {
        const float s = reinterpret_cast<const float*>(st + kOffDen)[t];
        const float* vs = reinterpret_cast<const float*>(st + kOffV);
        // MALA: beta = 1 + 1/s, gamma = s / n~_i
        const float beta = 1.f + 1.f / s;
        const float gamma = p.norm == MHLA_NORM_MALA ? s / ((float)p.nb * a.rowsum[i]) : 0.f;
        uint8_t* row = st + t * 128;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float* src = j < 4 ? &o0[8 * j] : &o1[8 * (j - 4)];
          uint4 x;
          uint32_t* xp = &x.x;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int cidx = 8 * j + 2 * q;
            float y0 = src[2 * q], y1 = src[2 * q + 1];
            if (p.norm == MHLA_NORM_DIVISIVE) {
              y0 = y0 / s;
              y1 = y1 / s;
            } else if (p.norm == MHLA_NORM_MALA) {
              y0 = beta * y0 - gamma * vs[cidx];
              y1 = beta * y1 - gamma * vs[cidx + 1];
            }
            xp[q] = pack_bf16x2(y0, y1);
          }
          *reinterpret_cast<uint4*>(row + (((j ^ t) & 7) << 4)) = x;
        }
      }
      fence_proxy_async();
      tc_fence_before();
      named_sync(3, 128);
      if (t == 0) {
        const int bx = i % p.Mw, by = (i / p.Mw) % p.Mh, bz = i / (p.Mw * p.Mh);
        const int x0 = bx * p.bw + (c % a.c.ncx) * a.c.cw;
        const int y0 = by * p.bh + ((c / a.c.ncx) % a.c.ncy) * a.c.ch;
        const int t0 = bz * p.bt + (c / (a.c.ncx * a.c.ncy)) * a.c.ct;
        tma_store_5d(&a.tmO, base + (uint32_t)stage * kStageBytes, 0, x0, y0, t0, u);
        bulk_commit();
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
    if (t == 0) bulk_wait<0>();
  }
  __syncwarp();

  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

int launch_tc_output(const Plan& p, const ChunkShape& c, const void* q, const TcBuffers& b, void* out,
                     cudaStream_t s) {
  OutArgs a;
  memset(&a, 0, sizeof(a));
  const uint64_t dims5[5] = {64, (uint64_t)p.Wg, (uint64_t)p.Hg, (uint64_t)p.T, (uint64_t)p.BH};
  const uint64_t str5[4] = {128, 128ull * p.Wg, 128ull * p.Wg * p.Hg, 128ull * p.N};
  const uint32_t box5[5] = {64, (uint32_t)c.cw, (uint32_t)c.ch, (uint32_t)c.ct, 1};
  int e;
  if ((e = encode_tmap_bf16(&a.tmQ, q, 5, dims5, str5, box5)) != 0) return e;
  if ((e = encode_tmap_bf16(&a.tmO, out, 5, dims5, str5, box5)) != 0) return e;
  const uint64_t dims3[3] = {64, (uint64_t)(p.R / 64), (uint64_t)p.BH * p.M};
  const uint64_t str3[2] = {128, 2ull * p.R};
  const uint32_t box3[3] = {64, 64, 1};
  if ((e = encode_tmap_bf16(&a.tmB_hi, b.mixed_hi, 3, dims3, str3, box3)) != 0) return e;
  if ((e = encode_tmap_bf16(&a.tmB_lo, b.mixed_lo, 3, dims3, str3, box3)) != 0) return e;
  a.mixed_hi = b.mixed_hi;
  a.mixed_lo = b.mixed_lo;
  a.rowsum = b.rowsum;
  a.units = p.BH * p.M * c.per_block;
  a.use_lo = p.norm == MHLA_NORM_MALA;
  a.c = c;
  a.err = p.err;
  cudaError_t ce = cudaFuncSetAttribute(tc_output_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (ce != cudaSuccess) return (int)ce;
  const int grid = a.units < num_sms() ? a.units : num_sms();
  tc_output_kernel<<<grid, kThreads, kSmemBytes, s>>>(a, p);
  return (int)cudaGetLastError();
}

}  // namespace mhla
