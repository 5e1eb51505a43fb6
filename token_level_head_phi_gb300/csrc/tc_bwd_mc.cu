// Gradient of the mixing matrix on the tensor cores (head dimension 64).
//
// The output of query block i depends on Mc[i, b] only through the mixed
// record X~_i = sum_b Mc[i, b] X_b ("MHLA: Restoring Expressivity of Linear
// Attention via Token-Level Multi-Head", key design 2; Mc is learned end to
// end, key design 3), so
//     dMc[i, b] = sum over heads of < dX~_i , X_b >
// where X_b = (S_b, z_b, v_b) is the record of block b and dX~_i the
// gradient of the loss with respect to the mixed record of block i (plus, for
// the MALA normalisation, n_b times the gradient of n~_i).  Over every head
// this is one GEMM  dMc = dX~ X^T  with a contraction length of
// heads x (d^2 + 2d); records are kept per block piece, so it runs over piece
// rows and the pieces are summed afterwards.
//
// Both operands arrive as bf16 high + low parts (a float32 value split as
// hi = bf16(x), lo = bf16(x - hi)); three MMAs per K step form
//     A_hi B_hi + A_hi B_lo + A_lo B_hi
// so the products carry about 16 significant bits, which the cancellation
// inside a row of dMc needs (for DIVISIVE, sum_b Mc[i,b] dMc[i,b] = 0).
//
// Kernel 1 (persistent, one CTA per SM): work item = (head, 128-row tile of
// i, 128-row tile of b); warp 0 streams the four 128 x 64 operand tiles of a
// K step by TMA (3 stages), warp 1 issues the MMAs into one of two TMEM
// accumulators, warps 4-7 copy the finished 128 x 128 float32 tile to a
// per-head partial.  Items run head-major so that the tiles of one head,
// which share their operands, are in flight together and hit L2.
// Kernel 2 sums the partials over heads and pieces in a fixed order (and
// adds the MALA term), so the result does not depend on scheduling.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstring>

#include "tc_bwd.h"
#include "tc_common.cuh"

namespace mhla {
namespace {

using namespace tc;

constexpr int kThreads = 256;
constexpr uint32_t kTile = 128 * 128;           // 128 rows x 64 bf16, 128-byte swizzle
constexpr uint32_t kStageBytes = 4 * kTile;     // A hi, A lo, B hi, B lo
constexpr int kStages = 3;
constexpr uint32_t kTmemCols = 512;             // two 256-column accumulators
constexpr uint32_t kBars = kStages * kStageBytes;
constexpr int kNumBars = 2 * kStages + 4;
constexpr uint32_t kSmemBytes = kBars + 8 * kNumBars + 16 + 1024;
static_assert(kSmemBytes <= 232448, "shared memory");

struct McArgs {
  CUtensorMap tmA_hi, tmA_lo, tmB_hi, tmB_lo;  // 3D (R, Q, BH), box (64, 128, 1)
  float* partial;                              // [BH][QP][QP], QP = 128 * qt
  int qt;                                      // 128-row tiles per side
  int kchunks;                                 // R / 64
  int items;                                   // BH * qt * qt
  unsigned int* err;
};

__global__ void __launch_bounds__(kThreads, 1) tc_bwd_mc_kernel(const __grid_constant__ McArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gb = smem_raw + (base - raw);
  const uint32_t bars = base + kBars;
  auto full = [&](int s) { return bars + 8u * s; };
  auto empty = [&](int s) { return bars + 8u * (kStages + s); };
  auto accfull = [&](int x) { return bars + 8u * (2 * kStages + x); };
  auto accempty = [&](int x) { return bars + 8u * (2 * kStages + 2 + x); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gb + kBars + 8 * kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gb + kBars + 8 * kNumBars + 8);
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int per_head = a.qt * a.qt;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(accfull(x), 1);
      mbar_init(accempty(x), 4);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&a.tmA_hi);
    tma_prefetch_desc(&a.tmA_lo);
    tma_prefetch_desc(&a.tmB_hi);
    tma_prefetch_desc(&a.tmB_lo);
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
      // ------------------------------------------------------- producer
      const uint64_t pol = policy_evict_last();
      int s = 0;
      uint32_t ph = 0;
      long long issued = 0;
      for (int w = blockIdx.x; w < a.items; w += gridDim.x) {
        const int u = w / per_head, rem = w - u * per_head;
        const int ti = rem / a.qt, tb = rem - ti * a.qt;
        bool ok = true;
        for (int kc = 0; kc < a.kchunks; ++kc) {
          if (!(ok = mbar_wait(empty(s), ph ^ 1u, a.err, 0x601, abort_flag))) break;
          const uint32_t st = base + (uint32_t)s * kStageBytes;
          mbar_arrive_expect_tx(full(s), kStageBytes);
          tma_load_3d(st, &a.tmA_hi, full(s), kc * 64, ti * 128, u, pol);
          tma_load_3d(st + kTile, &a.tmA_lo, full(s), kc * 64, ti * 128, u, pol);
          tma_load_3d(st + 2 * kTile, &a.tmB_hi, full(s), kc * 64, tb * 128, u, pol);
          tma_load_3d(st + 3 * kTile, &a.tmB_lo, full(s), kc * 64, tb * 128, u, pol);
          ++issued;
          if (++s == kStages) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
      }
      drain_loads(full(0), kStages, issued, a.err, 0x602);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA
      // B hi and B lo are adjacent 128-row K-major tiles: one N = 256 MMA
      // takes A hi against both (columns 0..127 and 128..255; the epilogue adds
      // them), as an MMA costs the same issue time whatever its N
      const uint32_t idesc = idesc_bf16_f32(128, 128, false, false);
      const uint32_t idesc2 = idesc_bf16_f32(128, 256, false, false);
      int s = 0, acc = 0;
      uint32_t ph = 0, accph = 0;
      bool ok = true;
      for (int w = blockIdx.x; w < a.items && ok; w += gridDim.x) {
        if (!(ok = mbar_wait(accempty(acc), accph ^ 1u, a.err, 0x603, abort_flag))) break;
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)acc * 256u;
        for (int kc = 0; kc < a.kchunks; ++kc) {
          if (!(ok = mbar_wait(full(s), ph, a.err, 0x604, abort_flag))) break;
          tc_fence_after();
          const uint32_t st = base + (uint32_t)s * kStageBytes;
          // descriptors of K step 0 advanced by 32 bytes (2 in the address
          // field) per step: the issuing thread's scalar work adds to every MMA
          const uint64_t ah0 = sdesc_sw128(st, 0u, 1024u), al0 = sdesc_sw128(st + kTile, 0u, 1024u);
          const uint64_t bh0 = sdesc_sw128(st + 2 * kTile, 0u, 1024u);   // rows 0..127 hi, 128..255 lo
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            umma_bf16(d, ah0 + 2 * ks, bh0 + 2 * ks, idesc2, (kc > 0 || ks > 0) ? 1u : 0u);
            umma_bf16(d, al0 + 2 * ks, bh0 + 2 * ks, idesc, 1u);
          }
          umma_commit(empty(s));
          if (++s == kStages) {
            s = 0;
            ph ^= 1u;
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
    // ------------------------------------------------------- epilogue
    const int q4 = warp & 3;
    const int row = 32 * q4 + lane;
    const size_t qp = (size_t)a.qt * 128;
    int acc = 0;
    uint32_t accph = 0;
    for (int w = blockIdx.x; w < a.items; w += gridDim.x) {
      const int u = w / per_head, rem = w - u * per_head;
      const int ti = rem / a.qt, tb = rem - ti * a.qt;
      const bool ok = mbar_wait(accfull(acc), accph, a.err, 0x605, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const uint32_t taddr = tmem + (uint32_t)acc * 256u + ((uint32_t)(32 * q4) << 16);
      float* dst = a.partial + ((size_t)u * qp + (size_t)ti * 128 + row) * qp + (size_t)tb * 128;
#pragma unroll 1
      for (int j = 0; j < 4; ++j) {
        float v[32], w2[32];
        tmem_ld32(taddr + 32u * j, v);
        tmem_ld32(taddr + 128u + 32u * j, w2);
        tmem_wait_ld();
#pragma unroll
        for (int x = 0; x < 32; ++x) v[x] += w2[x];
#pragma unroll
        for (int x = 0; x < 8; ++x)
          reinterpret_cast<float4*>(dst + 32 * j)[x] = make_float4(v[4 * x], v[4 * x + 1], v[4 * x + 2], v[4 * x + 3]);
      }
      tc_fence_before();
      mbar_arrive_warp(accempty(acc));
      if (++acc == 2) {
        acc = 0;
        accph ^= 1u;
      }
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// dmc[h][i][b] = sum_u sum_{s, s'} partial[u][i*splits + s][b*splits + s']
//                (+ MALA: n_b sum_u sum_s dnp[u][i*splits + s])
// with u over every unit (heads == 1, one shared Mc) or over the units of
// head h (heads == H, one Mc per head).
__global__ void bwd_mc_reduce_kernel(const float* __restrict__ partial, const float* __restrict__ dnp, int M,
                                     int splits, int BH, int qp, int Q, float nb, int mala, int heads,
                                     float* __restrict__ dmc) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= heads * M * M) return;
  const int h = idx / (M * M), rem = idx - h * M * M;
  const int i = rem / M, b = rem - i * M;
  float acc = 0.f;
  for (int u = h; u < BH; u += heads) {
    const float* pu = partial + (size_t)u * qp * qp;
    float au = 0.f;
    for (int s = 0; s < splits; ++s)
      for (int t = 0; t < splits; ++t) au += pu[(size_t)(i * splits + s) * qp + b * splits + t];
    acc += au;
  }
  if (mala) {
    float dn = 0.f;
    for (int u = h; u < BH; u += heads)
      for (int s = 0; s < splits; ++s) dn += dnp[(size_t)u * Q + i * splits + s];
    acc = fmaf(nb, dn, acc);
  }
  dmc[idx] = acc;
}

}  // namespace

size_t tc_bwd_mc_partial_bytes(const Plan& p) {
  const size_t qp = (size_t)(p.M * p.splits + 127) / 128 * 128;
  return sizeof(float) * (size_t)p.BH * qp * qp;
}

int launch_tc_bwd_mc(const Plan& p, const __nv_bfloat16* dx_hi, const __nv_bfloat16* dx_lo,
                     const __nv_bfloat16* x_hi, const __nv_bfloat16* x_lo, const float* dnp, float* partial,
                     float* dmc, cudaStream_t s) {
  McArgs a;
  memset(&a, 0, sizeof(a));
  const int Q = p.M * p.splits;
  const uint64_t dims[3] = {(uint64_t)p.R, (uint64_t)Q, (uint64_t)p.BH};
  const uint64_t str[2] = {2ull * p.R, 2ull * p.R * Q};
  const uint32_t box[3] = {64, 128, 1};
  int e;
  if ((e = encode_tmap_bf16(&a.tmA_hi, dx_hi, 3, dims, str, box)) != 0) return e;
  if ((e = encode_tmap_bf16(&a.tmA_lo, dx_lo, 3, dims, str, box)) != 0) return e;
  if ((e = encode_tmap_bf16(&a.tmB_hi, x_hi, 3, dims, str, box)) != 0) return e;
  if ((e = encode_tmap_bf16(&a.tmB_lo, x_lo, 3, dims, str, box)) != 0) return e;
  a.qt = (Q + 127) / 128;
  a.kchunks = p.R / 64;
  a.items = p.BH * a.qt * a.qt;
  a.partial = partial;
  a.err = p.err;
  cudaError_t ce = (cudaError_t)set_max_dynamic_smem((const void*)tc_bwd_mc_kernel, (int)kSmemBytes);
  if (ce != cudaSuccess) return (int)ce;
  const int grid = a.items < num_sms() ? a.items : num_sms();
  tc_bwd_mc_kernel<<<grid, kThreads, kSmemBytes, s>>>(a);
  if ((ce = cudaGetLastError()) != cudaSuccess) return (int)ce;
  const int n = p.M * p.M * p.mc_heads;
  bwd_mc_reduce_kernel<<<(n + 255) / 256, 256, 0, s>>>(partial, dnp, p.M, p.splits, p.BH, a.qt * 128, Q,
                                                       (float)p.nb, p.norm == MHLA_NORM_MALA ? 1 : 0, p.mc_heads,
                                                       dmc);
  return (int)cudaGetLastError();
}

}  // namespace mhla
