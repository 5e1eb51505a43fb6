// Block-ordered causal output step on the tensor cores (head dimension 64,
// bf16 tensors).
//
// Query t of block i sees the earlier blocks through the strict lower
// triangle of Mc and its own block up to itself through w = Mc[i, i] (the
// block-ordered reading of "MHLA: Restoring Expressivity of Linear Attention
// via Token-Level Multi-Head", key design 2 and its chunkwise remarks).  The
// token chunks of a block (each a contiguous run of the block's local order)
// are taken in order; with P = phi(Q_c), F = phi(K_c):
//   prefix  D_a  = P S_hi + P S_lo  |  P Z          (numerator columns | s parts)
//   scores  D_s  = P F^T                           (N = 128)
//   intra   P~   = w * mask(D_s)  (j <= t; bf16, kept in TMEM)
//           D_a += P~ [V | e0]                     (numerator; row sum of P~ in column 64)
//   state   D_u  = [F | e0]^T [V | e0]  for the next chunk:
//           S_state = S<_i + w * sum of F^T V, z_state likewise with F^T 1
//           (S as bf16 high + low planes; Z a K-major tile with z_state's
//           bf16 high part in row 0 and low part in row 1)
// where S<_i, z<_i are the records mixed with the strict lower triangle
// (high + low planes) and e0 is a tile with a one in its first column.  Then
//   s = D_a[64] + D_a[65],  DIVISIVE o = num / s,  NONE o = num;  s = 0 gives o = 0.
// Persistent, warp-specialised CTA (512 threads, one per SM): warp 0 loads
// Q, K, V (three token stages), warp 1 allocates TMEM and issues the MMAs,
// warp 2 loads each unit's prefix record (two state buffers), warps 4-7
// apply phi, warps 8-11 write P~, warps 12-15 update the state and write the
// outputs.  A CTA takes its (head, block) units two at a time and alternates
// their chunks, so one unit's carried-state chain overlaps the other's; the
// MMA warp issues whichever group is ready, so a chunk's prefix and scores
// run while the previous chunk's scores epilogue works; D_a and the output
// staging tile are double-buffered.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstring>

#include "common.cuh"
#include "tc_causal.h"
#include "tc_common.cuh"

namespace mhla {
namespace {

using namespace tc;

// Non-blocking test whether the phase of `bar` with parity `parity` has
// completed (acquire semantics when it has).
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

constexpr int kThreads = 512;
constexpr int kGrpThreads = 128;                 // warps 4-7 (phi), 8-11 (scores), 12-15 (outputs, state)
constexpr uint32_t kTile = 128 * 128;            // 128 rows x 64 bf16
constexpr uint32_t kBTile = 64 * 128;            // 64 rows x 64 bf16
constexpr int kStages = 3;
// shared memory (offsets from the 1024-aligned base)
constexpr uint32_t kStageBytes = 3 * kTile;            // Q -> P | K -> F | V
constexpr uint32_t kOffSt = kStages * kStageBytes;     // two state buffers: S hi | S lo | Z (K-major, 16 rows)
constexpr uint32_t kStBytes = 2 * kBTile + 2048;
constexpr uint32_t kOffO = kOffSt + 2 * kStBytes;      // two output staging tiles
constexpr uint32_t kOffE0 = kOffO + 2 * kTile;         // 16 rows x 64, a one in column 0
constexpr uint32_t kOffBars = kOffE0 + 2048;
constexpr int kNumBars = 3 * kStages + 5 * 2 + 6;
constexpr uint32_t kSmemBytes = kOffBars + 8 * kNumBars + 16 + 1024;
constexpr uint32_t kTmemCols = 512;
// TMEM columns: D_a (two, 80 used) at 0 and 96, D_s 192..319, D_u 320..399,
// P~ 416..479 (bf16 pairs, the A operand of the numerator MMA)
constexpr uint32_t kColS = 192, kColU = 320, kColP = 416;
__device__ __forceinline__ uint32_t col_a(int acc) { return acc ? 96u : 0u; }
static_assert(kSmemBytes <= 232448, "shared memory");
static_assert(kOffSt % 1024 == 0 && kOffO % 1024 == 0 && kOffE0 % 1024 == 0 && kStBytes % 1024 == 0, "alignment");

struct CausalArgs {
  CUtensorMap tmQ, tmK, tmV, tmO;   // token maps (encode_token_map)
  CUtensorMap tmS_hi, tmS_lo;       // 3D (64, R/64, BH*M) over the prefix-mixed planes, box (64, 64, 1)
  const __nv_bfloat16* mixed_hi;    // prefix-mixed records (z< rows read directly)
  const __nv_bfloat16* mixed_lo;
  const float* mc;                  // Mc (its diagonal weighs the block's own tokens)
  int R, units;                     // record length, (head, block) units
  FastDiv f_m;                      // division by M
  ChunkShape c;
  unsigned int* err;
};

// The chunks of this CTA in issue order.  Its units k = 0, 1, 2, ... (unit
// w = blockIdx.x + k * gridDim.x, head u = w / M, block i = w % M) are taken
// in pairs whose chunks alternate, (k, 0), (k+1, 0), (k, 1), (k+1, 1), ...:
// each unit's chunks depend on one another through the carried state, the
// two units of a pair do not.  n counts chunks; state buffer x = k & 1.
struct ChunkIt {
  int k0, side, k, w, u, i, c;
  bool pair, valid;
  long long n;
};

__device__ __forceinline__ void ci_set(const CausalArgs& a, const Plan& p, ChunkIt& it) {
  it.k = it.k0 + it.side;
  it.w = (int)blockIdx.x + it.k * (int)gridDim.x;
  it.u = (int)fdiv((uint32_t)it.w, a.f_m);
  it.i = it.w - it.u * p.M;
}

__device__ __forceinline__ void ci_pair(const CausalArgs& a, ChunkIt& it) {
  it.valid = (int)blockIdx.x + it.k0 * (int)gridDim.x < a.units;
  it.pair = (int)blockIdx.x + (it.k0 + 1) * (int)gridDim.x < a.units;
}

__device__ __forceinline__ void ci_begin(const CausalArgs& a, const Plan& p, ChunkIt& it) {
  it.k0 = 0;
  it.side = 0;
  it.c = 0;
  it.n = 0;
  ci_pair(a, it);
  if (it.valid) ci_set(a, p, it);
}

__device__ __forceinline__ void ci_next(const CausalArgs& a, const Plan& p, ChunkIt& it) {
  ++it.n;
  if (it.side == 0 && it.pair) {
    it.side = 1;
  } else {
    it.side = 0;
    if (++it.c == a.c.per_block) {
      it.c = 0;
      it.k0 += 2;
      ci_pair(a, it);
    }
  }
  if (it.valid) ci_set(a, p, it);
}

__device__ __forceinline__ float diag_weight(const CausalArgs& a, const Plan& p, const ChunkIt& it) {
  return a.mc[((size_t)mc_index(p, it.u) * p.M + it.i) * p.M + it.i];
}

// Feature k of the z state in the K-major Z tile: bf16 high part in row 0,
// low part in row 1 (rows 2..15 stay zero).
__device__ __forceinline__ void put_z(uint8_t* zt, int k, float z) {
  const __nv_bfloat16 zh = __float2bfloat16_rn(z);
  const __nv_bfloat16 zl = __float2bfloat16_rn(z - __bfloat162float(zh));
  *reinterpret_cast<__nv_bfloat16*>(zt + sw128_offset(0, k)) = zh;
  *reinterpret_cast<__nv_bfloat16*>(zt + sw128_offset(1, k)) = zl;
}

__global__ void __launch_bounds__(kThreads, 1) tc_causal_kernel(const __grid_constant__ CausalArgs a, const Plan p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gb = smem_raw + (base - raw);
  const uint32_t bars = base + kOffBars;
  auto tfull = [&](int s) { return bars + 8u * (uint32_t)s; };                 // Q, K, V landed (tx)
  auto pready = [&](int s) { return bars + 8u * (uint32_t)(kStages + s); };    // P, F written (4 warps)
  auto tempty = [&](int s) { return bars + 8u * (uint32_t)(2 * kStages + s); };  // the stage's MMAs done
  const uint32_t b2 = bars + 8u * (uint32_t)(3 * kStages);
  auto stfull = [&](int x) { return b2 + 8u * (uint32_t)x; };        // S<, Z< of a unit in place (tx)
  auto stfree = [&](int x) { return b2 + 16u + 8u * (uint32_t)x; };  // the unit's last prefix MMA done
  auto stupd = [&](int x) { return b2 + 32u + 8u * (uint32_t)x; };   // state updated for the next chunk (2 warps)
  auto afull = [&](int x) { return b2 + 48u + 8u * (uint32_t)x; };   // numerator complete (commit)
  auto afree = [&](int x) { return b2 + 64u + 8u * (uint32_t)x; };   // numerator read (4 warps)
  const uint32_t b1 = b2 + 80u;
  const uint32_t sfull = b1, sfree = b1 + 8, ptready = b1 + 16, ptfree = b1 + 24, ufree = b1 + 32, mdone = b1 + 40;
  static_assert(8 * (3 * kStages) + 80 + 48 == 8 * kNumBars, "barrier slots");
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gb + kOffBars + 8 * kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gb + kOffBars + 8 * kNumBars + 8);
  auto tst = [&](int s) { return base + (uint32_t)s * kStageBytes; };
  auto stb = [&](int x) { return base + kOffSt + (uint32_t)x * kStBytes; };
  auto obuf = [&](int x) { return base + kOffO + (uint32_t)x * kTile; };

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int rows = a.c.rows, rows_pad = a.c.rows_pad, nck = a.c.per_block;

  // every tile starts zero (rows and columns past a chunk stay zero), e0 tile
  for (uint32_t off = threadIdx.x * 16u; off < kOffBars; off += kThreads * 16u)
    *reinterpret_cast<uint4*>(gb + off) = make_uint4(0u, 0u, 0u, 0u);
  __syncthreads();
  if (threadIdx.x < 16)
    *reinterpret_cast<__nv_bfloat16*>(gb + kOffE0 + sw128_offset(threadIdx.x, 0)) = __float2bfloat16_rn(1.f);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(tfull(s), 1);
      mbar_init(pready(s), kGrpThreads / 32);
      mbar_init(tempty(s), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(stfull(x), 1);
      mbar_init(stfree(x), 1);
      mbar_init(stupd(x), 2);   // warps 12, 13 (state rows 0..63)
      mbar_init(afull(x), 1);
      mbar_init(afree(x), kGrpThreads / 32);
    }
    mbar_init(sfull, 1);
    mbar_init(sfree, kGrpThreads / 32);
    mbar_init(ptready, kGrpThreads / 32);
    mbar_init(ptfree, 1);
    mbar_init(ufree, 2);
    mbar_init(mdone, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&a.tmQ);
    tma_prefetch_desc(&a.tmK);
    tma_prefetch_desc(&a.tmV);
    tma_prefetch_desc(&a.tmO);
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
      // -------------------------------------------- Q, K, V producer
      const uint64_t pol = policy_evict_first();
      const uint32_t bytes = (uint32_t)rows * 128u;
      long long issued = 0;
      ChunkIt it;
      for (ci_begin(a, p, it); it.valid; ci_next(a, p, it)) {
        const int s = (int)(it.n % kStages);
        if (!mbar_wait(tempty(s), (uint32_t)((it.n / kStages) & 1) ^ 1u, a.err, 0x911, abort_flag)) break;
        int x0, y0, t0;
        chunk_origin(p, a.c, (uint32_t)it.i, (uint32_t)it.c, x0, y0, t0);
        const TileCoords g5 = token_tile_coords(p, it.u, x0, y0, t0);
        mbar_arrive_expect_tx(tfull(s), 3 * bytes);
        tma_load_5d(tst(s), &a.tmQ, tfull(s), g5.c[0], g5.c[1], g5.c[2], g5.c[3], g5.c[4], pol);
        tma_load_5d(tst(s) + kTile, &a.tmK, tfull(s), g5.c[0], g5.c[1], g5.c[2], g5.c[3], g5.c[4], pol);
        tma_load_5d(tst(s) + 2 * kTile, &a.tmV, tfull(s), g5.c[0], g5.c[1], g5.c[2], g5.c[3], g5.c[4], pol);
        ++issued;
      }
      drain_loads(tfull(0), kStages, issued, a.err, 0x912);
    }
  } else if (warp == 2) {
    // --------------------------- prefix records S<_i, z<_i, one per unit
    long long issued = 0;
    for (int k = 0; (int)blockIdx.x + k * (int)gridDim.x < a.units; ++k) {
      const int x = k & 1;
      bool ok = true;
      if (lane == 0) ok = mbar_wait(stfree(x), (uint32_t)((k >> 1) & 1) ^ 1u, a.err, 0x913, abort_flag);
      if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
      const int w = (int)blockIdx.x + k * (int)gridDim.x;
      const int u = (int)fdiv((uint32_t)w, a.f_m);
      const size_t rec = (size_t)u * p.M + (size_t)(w - u * p.M);
      uint8_t* zt = gb + kOffSt + x * kStBytes + 2 * kBTile;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int kk = lane + 32 * j;
        const size_t zo = rec * a.R + 64 * 64 + kk;
        put_z(zt, kk, __bfloat162float(a.mixed_hi[zo]) + __bfloat162float(a.mixed_lo[zo]));
      }
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) {
        const uint64_t pol = policy_evict_first();
        mbar_arrive_expect_tx(stfull(x), 2 * kBTile);
        tma_load_3d(stb(x), &a.tmS_hi, stfull(x), 0, 0, (int)rec, pol);
        tma_load_3d(stb(x) + kBTile, &a.tmS_lo, stfull(x), 0, 0, (int)rec, pol);
      }
      ++issued;
    }
    if (lane == 0) drain_loads(stfull(0), 2, issued, a.err, 0x914);
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------- MMA
      // Two groups per chunk: prefix + scores (once its P, F and state are
      // in place), then numerator + state (once the scores epilogue has
      // written P~).  Whichever is ready goes first, numerator groups in
      // chunk order, so a chunk's prefix and scores can run while the
      // previous chunk's scores epilogue works.
      const uint32_t id_s64 = idesc_bf16_f32(128, 64, false, true);
      const uint32_t id_z = idesc_bf16_f32(128, 16, false, false);
      const uint32_t id_s = idesc_bf16_f32(128, 128, false, false);
      const uint32_t id_v = idesc_bf16_f32(128, 80, false, true);
      const uint32_t id_u = idesc_bf16_f32(128, 80, true, true);
      const uint32_t e0 = base + kOffE0;
      // Descriptors are formed once per group and advanced by adding to their
      // fields: the address field (byte offset / 16) and, for the operands
      // whose second atom is the ones tile e0, the leading offset field
      // (bits 16..29), which shrinks by as much as the address grows.  The
      // issue of each MMA waits for the tensor pipe, so every instruction on
      // this thread adds to the chunk's time.
      const uint64_t e_step = 128ull - (128ull << 16);  // + 2048 bytes, leading offset - 2048 bytes
      long long nupd0 = 0, nupd1 = 0, nu = 0;
      long long qn0 = 0, qn1 = 0;   // chunks waiting for their second group (oldest first)
      bool qm0 = false, qm1 = false;
      int nq = 0;
      unsigned long long idle_since = 0;
      ChunkIt nx;
      ci_begin(a, p, nx);
      while (nx.valid || nq > 0) {
        bool did = false;
        if (nq > 0 && mbar_test(ptready, (uint32_t)(qn0 & 1)) &&
            (!qm0 || nu == 0 || mbar_test(ufree, (uint32_t)((nu - 1) & 1)))) {
          // D_a += P~ [V | e0] (numerator; row sum of P~ in column 64), and
          // D_u = [F | e0]^T [V | e0] when another chunk of the unit follows
          tc_fence_after();
          const int ps = (int)(qn0 % kStages);
          const uint32_t k_s = tst(ps) + kTile, v_s = tst(ps) + 2 * kTile;
          const uint32_t DA = tmem + col_a((int)(qn0 & 1));
          const uint64_t vd0 = sdesc_sw128(v_s, e0 - v_s, 1024u);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            umma_tmem_a(DA, tmem + kColP + (uint32_t)ks * 8u, vd0 + (uint64_t)ks * e_step, id_v, 1u);
          if (qm0) {
            const uint64_t fd0 = sdesc_sw128(k_s, e0 - k_s, 1024u);
            uint64_t fd = fd0, vd = vd0;
            for (int kt = 0; kt < rows_pad / 16; ++kt) {
              umma_bf16(tmem + kColU, fd, vd, id_u, kt > 0 ? 1u : 0u);
              fd += e_step;
              vd += e_step;
            }
            ++nu;
          }
          umma_commit(tempty(ps));
          umma_commit(ptfree);
          umma_commit(afull((int)(qn0 & 1)));
          qn0 = qn1;
          qm0 = qm1;
          --nq;
          did = true;
        } else if (nx.valid && nq < 2) {
          const int s = (int)(nx.n % kStages), x = nx.k & 1, acc = (int)(nx.n & 1);
          const long long nupd = x ? nupd1 : nupd0;
          bool ready = nx.c == 0 ? mbar_test(stfull(x), (uint32_t)((nx.k >> 1) & 1))
                                 : mbar_test(stupd(x), (uint32_t)(nupd & 1));
          ready = ready && mbar_test(pready(s), (uint32_t)((nx.n / kStages) & 1)) &&
                  mbar_test(afree(acc), (uint32_t)((nx.n >> 1) & 1) ^ 1u) &&
                  mbar_test(sfree, (uint32_t)(nx.n & 1) ^ 1u);
          if (ready) {
            if (nx.c > 0) {
              if (x) ++nupd1;
              else ++nupd0;
            }
            tc_fence_after();
            // D_a = P S_hi + P S_lo | P Z (prefix), D_s = P F^T (scores)
            const uint32_t q_s = tst(s), k_s = q_s + kTile;
            const uint32_t sh = stb(x), sl = sh + kBTile, zt = sh + 2 * kBTile;
            const uint32_t DA = tmem + col_a(acc);
            // one shape at a time: scores first (the scores epilogue waits
            // for them), then the prefix parts
            const uint64_t qd = sdesc_sw128(q_s, 0u, 1024u), kd = sdesc_sw128(k_s, 0u, 1024u);
            const uint64_t shd = sdesc_sw128(sh, 0u, 1024u), sld = sdesc_sw128(sl, 0u, 1024u);
            const uint64_t zd = sdesc_sw128(zt, 0u, 1024u);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) umma_bf16(tmem + kColS, qd + 2 * ks, kd + 2 * ks, id_s, ks > 0 ? 1u : 0u);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
              umma_bf16(DA, qd + 2 * (ks & 3), (ks < 4 ? shd : sld) + 128 * (ks & 3), id_s64, ks > 0 ? 1u : 0u);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) umma_bf16(DA + 64u, qd + 2 * ks, zd + 2 * ks, id_z, ks > 0 ? 1u : 0u);
            umma_commit(sfull);
            if (nx.c + 1 == nck) umma_commit(stfree(x));   // the unit's state buffer is read for the last time
            if (nq == 0) {
              qn0 = nx.n;
              qm0 = nx.c + 1 < nck;
            } else {
              qn1 = nx.n;
              qm1 = nx.c + 1 < nck;
            }
            ++nq;
            ci_next(a, p, nx);
            did = true;
          }
        }
        if (did) {
          idle_since = 0;
          continue;
        }
        // nothing ready: bounded polling
        if (*abort_flag) break;
        const unsigned long long now = globaltimer();
        if (idle_since == 0) {
          idle_since = now;
        } else if (now - idle_since > kWaitLimitNs) {
          report_timeout(a.err, 0x915);
          *abort_flag = 1;
          break;
        }
        __nanosleep(64);
      }
      // every MMA issued has completed before TMEM is released
      umma_commit(mdone);
      mbar_wait(mdone, 0u, a.err, 0x91c);
    }
  } else if (warp >= 4 && warp < 8) {
    // --------------------------------------- P = phi(Q), F = phi(K)
    const int t = threadIdx.x - 4 * 32;
    ChunkIt it;
    for (ci_begin(a, p, it); it.valid; ci_next(a, p, it)) {
      const int s = (int)(it.n % kStages);
      const bool ok = mbar_wait(tfull(s), (uint32_t)((it.n / kStages) & 1), a.err, 0x91d, abort_flag);
      if (!named_all(9, kGrpThreads, ok)) break;
      if (t < rows) {
        // rows t of Q and of K, four 16-byte chunks at a time, visited as
        // j ^ t so that the eight rows of a quarter-warp touch eight
        // different bank groups (a rolled loop keeps this role's code small)
#pragma unroll 1
        for (int g = 0; g < 4; ++g) {
          uint4* r = reinterpret_cast<uint4*>(gb + (tst(s) - base) + (uint32_t)(g >> 1) * kTile + t * 128);
          const int j0 = 4 * (g & 1);
          uint4 xv[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) xv[j] = r[((j0 + j) ^ t) & 7];
          if (p.fmap == MHLA_FEATURE_ELU1) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              xv[j].x = phi2_elu1_bf16(xv[j].x);
              xv[j].y = phi2_elu1_bf16(xv[j].y);
              xv[j].z = phi2_elu1_bf16(xv[j].z);
              xv[j].w = phi2_elu1_bf16(xv[j].w);
            }
          } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              uint32_t* pw = &xv[j].x;
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float2 f = bf16x2_to_float2(pw[e]);
                pw[e] = pack_bf16x2(phi_map(f.x, p.fmap), phi_map(f.y, p.fmap));
              }
            }
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) r[((j0 + j) ^ t) & 7] = xv[j];
        }
      }
      fence_proxy_async();
      mbar_arrive_warp(pready(s));
    }
  } else if (warp >= 8 && warp < 12) {
    // --------------------------- P~ = w mask(D_s), j <= t, into TMEM
    const int e = warp - 8, t = threadIdx.x - 8 * 32;
    const uint32_t ta = tmem + ((uint32_t)(32 * e) << 16);
    {
      // token pairs past every row of this warp stay zero from here on
      uint32_t zero[32];
#pragma unroll
      for (int m = 0; m < 32; ++m) zero[m] = 0u;
      tmem_st32(ta + kColP, zero);
      tmem_st32(ta + kColP + 32u, zero);
      tmem_wait_st();
    }
    // scores of 32 tokens (part h of the row) -> 16 bf16 pairs of P~; only
    // the part on the diagonal (h == e) needs the mask j <= t
    auto pack_part = [&](const float (&sc)[32], int h, float wt, uint32_t* pw) {
      if (h < e) {
#pragma unroll
        for (int m = 0; m < 16; ++m) pw[m] = pack_bf16x2(wt * sc[2 * m], wt * sc[2 * m + 1]);
      } else {
        const int d = t - 32 * h;   // 0..31: last token of the part this row sees
#pragma unroll
        for (int m = 0; m < 16; ++m)
          pw[m] = pack_bf16x2(2 * m <= d ? wt * sc[2 * m] : 0.f, 2 * m + 1 <= d ? wt * sc[2 * m + 1] : 0.f);
      }
    };
    ChunkIt it;
    for (ci_begin(a, p, it); it.valid; ci_next(a, p, it)) {
      const float w = diag_weight(a, p, it);
      const float wt = t < rows ? w : 0.f;
      bool ok = mbar_wait(sfull, (uint32_t)(it.n & 1), a.err, 0x91e, abort_flag);
      ok = ok && mbar_wait(ptfree, (uint32_t)(it.n & 1) ^ 1u, a.err, 0x91f, abort_flag);
      if (!named_all(8, kGrpThreads, ok)) break;
      tc_fence_after();
      // tokens 64 hp .. 64 hp + 63 -> P~ columns 32 hp .. 32 hp + 31; the
      // tokens past every row of a warp keep their zero columns
#pragma unroll 1
      for (int hp = 0; hp < 2; ++hp) {
        if (2 * hp > e) break;
        uint32_t pw[32];
        float sc[32];
        tmem_ld32(ta + kColS + 64u * hp, sc);
        tmem_wait_ld();
        pack_part(sc, 2 * hp, wt, pw);
        if (2 * hp + 1 <= e) {
          tmem_ld32(ta + kColS + 64u * hp + 32u, sc);
          tmem_wait_ld();
          pack_part(sc, 2 * hp + 1, wt, pw + 16);
        } else {
#pragma unroll
          for (int m = 16; m < 32; ++m) pw[m] = 0u;
        }
        tmem_st32(ta + kColP + 32u * hp, pw);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive_warp(sfree);
      mbar_arrive_warp(ptready);
    }
  } else if (warp >= 12) {
    // ----------------------- state for the next chunk, then the outputs
    const int e = warp - 12, t = threadIdx.x - 12 * 32;
    const uint32_t ta = tmem + ((uint32_t)(32 * e) << 16);
    float zr0 = 0.f, zr1 = 0.f;   // z state of row t (< 64) for state buffers 0, 1
    ChunkIt it;
    for (ci_begin(a, p, it); it.valid; ci_next(a, p, it)) {
      const int acc = (int)(it.n & 1), x = it.k & 1;
      const bool upd = it.c + 1 < nck && e < 2;
      const float w = diag_weight(a, p, it);
      bool ok = true;
      float zin = 0.f;
      if (upd && it.c == 0) {
        const size_t zo = ((size_t)it.u * p.M + it.i) * a.R + 64 * 64 + t;
        zin = __bfloat162float(a.mixed_hi[zo]) + __bfloat162float(a.mixed_lo[zo]);
        ok = mbar_wait(stfull(x), (uint32_t)((it.k >> 1) & 1), a.err, 0x920, abort_flag);
      }
      ok = ok && mbar_wait(afull(acc), (uint32_t)((it.n >> 1) & 1), a.err, 0x921, abort_flag);
      if (t == 0) bulk_wait_read<1>();   // staging tile acc: the store two chunks back has been read
      if (!named_all(7, kGrpThreads, ok)) break;
      tc_fence_after();
      if (upd) {
        // S_state += w F^T V (bf16 high + low), z_state += w F^T 1
        float dv[32], zc[16];
        uint8_t* shr = gb + kOffSt + x * kStBytes + t * 128;
        uint8_t* slr = shr + kBTile;
        tmem_ld16(ta + kColU + 64u, zc);
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
            for (int m = 0; m < 4; ++m) {
              const float2 fh = bf16x2_to_float2(hp[m]), fl = bf16x2_to_float2(lp[m]);
              const float y0 = fh.x + fl.x + w * dv[8 * q + 2 * m], y1 = fh.y + fl.y + w * dv[8 * q + 2 * m + 1];
              hp[m] = pack_bf16x2(y0, y1);
              const float2 g = bf16x2_to_float2(hp[m]);
              lp[m] = pack_bf16x2(y0 - g.x, y1 - g.y);
            }
            *reinterpret_cast<uint4*>(shr + off) = hv;
            *reinterpret_cast<uint4*>(slr + off) = lv;
          }
        }
        const float zn = (it.c == 0 ? zin : (x ? zr1 : zr0)) + w * zc[0];
        if (x) zr1 = zn;
        else zr0 = zn;
        put_z(gb + kOffSt + x * kStBytes + 2 * kBTile, t, zn);
        tc_fence_before();
        fence_proxy_async();
        mbar_arrive_warp(ufree);
        mbar_arrive_warp(stupd(x));
      }
      {
        // s = P z_state + rowsum(P~) (columns 64, 65); DIVISIVE o = num / s
        float nm[32], zc[16];
        const uint32_t DA = ta + col_a(acc);
        tmem_ld16(DA + 64u, zc);
        tmem_wait_ld();
        const float s = zc[0] + zc[1];
        float scale = 1.f;
        if (p.norm == MHLA_NORM_DIVISIVE) scale = s != 0.f ? 1.f / s : 0.f;
        uint8_t* orow = gb + kOffO + acc * kTile + t * 128;
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
          tmem_ld32(DA + 32u * h, nm);
          tmem_wait_ld();
          if (t < rows) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint4 ov;
              uint32_t* op = &ov.x;
#pragma unroll
              for (int m = 0; m < 4; ++m)
                op[m] = pack_bf16x2(nm[8 * q + 2 * m] * scale, nm[8 * q + 2 * m + 1] * scale);
              *reinterpret_cast<uint4*>(orow + ((((4 * h + q) ^ t) & 7) << 4)) = ov;
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive_warp(afree(acc));
      fence_proxy_async();
      named_sync(7, kGrpThreads);
      if (t == 0) {
        int x0, y0, t0;
        chunk_origin(p, a.c, (uint32_t)it.i, (uint32_t)it.c, x0, y0, t0);
        const TileCoords g5 = token_tile_coords(p, it.u, x0, y0, t0);
        tma_store_5d(&a.tmO, obuf(acc), g5.c[0], g5.c[1], g5.c[2], g5.c[3], g5.c[4]);
        bulk_commit();
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
  a.units = p.BH * p.M;
  a.f_m = make_fastdiv((uint32_t)p.M);
  a.c = c;
  a.err = p.err;
  cudaError_t ce = (cudaError_t)set_max_dynamic_smem((const void*)tc_causal_kernel, (int)kSmemBytes);
  if (ce != cudaSuccess) return (int)ce;
  const int grid = a.units < num_sms() ? a.units : num_sms();
  tc_causal_kernel<<<grid, kThreads, kSmemBytes, s>>>(a, p);
  return (int)cudaGetLastError();
}

}  // namespace mhla
