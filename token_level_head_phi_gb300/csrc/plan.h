// Internal execution plan shared by the host dispatcher and the kernels.
//
// A Plan is a plain struct passed by value to every kernel.  It holds the
// problem shape, the block partition of the token grid, how long blocks are
// split into partial summaries, and where each intermediate lives in the
// caller's workspace.
#pragma once

#include <cstddef>
#include <cstdint>

#include "mhla.h"

#ifndef __CUDACC__
#define __host__
#define __device__
#endif

namespace mhla {

// Unsigned division by a divisor fixed when the plan is made, by one
// multiply-high, an add and a shift (T. Granlund, P. Montgomery, "Division
// by invariant integers using multiplication", PLDI 1994, section 4): for
// 1 <= d < 2^31, s = ceil(log2 d) and m = floor(2^32 (2^s - d) / d) + 1,
// n / d = (hi32(m n) + n) >> s for every 32-bit n.  Work-unit and grid
// indices are split this way once per unit on the device, where an
// integer division would otherwise cost a few dozen dependent instructions.
struct FastDiv {
  uint32_t d, m, s;
};

inline FastDiv make_fastdiv(uint32_t d) {
  FastDiv f;
  f.d = d < 1 ? 1 : d;
  f.s = 0;
  while ((1ull << f.s) < f.d) ++f.s;
  f.m = (uint32_t)((((1ull << f.s) - f.d) << 32) / f.d + 1);
  return f;
}

__host__ __device__ inline uint32_t fdiv(uint32_t n, const FastDiv& f) {
#ifdef __CUDA_ARCH__
  const uint32_t hi = __umulhi(n, f.m);
#else
  const uint32_t hi = (uint32_t)(((uint64_t)n * f.m) >> 32);
#endif
  return (uint32_t)(((uint64_t)hi + n) >> f.s);
}

// Token tile ("chunk") of the tensor-core path: a (ct, ch, cw) sub-box of a
// block with ct*ch*cw <= 128 rows that tiles the block exactly.
struct ChunkShape {
  int ct, ch, cw;
  int ncx, ncy, nct;  // chunks per block along x, y, t
  int per_block;      // ncx * ncy * nct
  int rows;           // ct * ch * cw
  int rows_pad;       // rows rounded up to 16 (MMA K granularity)
  FastDiv f_ncx, f_ncxy;  // divisions by ncx and ncx * ncy
};

struct Plan {
  // shape
  int B, H, BH, d;
  int T, Hg, Wg;  // token grid
  int bt, bh, bw; // block shape
  int Mt, Mh, Mw; // block grid
  int N, M, nb;   // tokens, blocks, tokens per block
  // options
  int dtype, fmap, norm, variant;
  int causal;         // block-ordered causal form (float32 kernels only)
  int layout;         // MHLA_LAYOUT_BHND or MHLA_LAYOUT_BNHD for q, k, v, out (and gradients)
  int mc_heads;       // mixing matrices: 1 (shared) or H (one per head, shared over the batch)
  FastDiv f_h;        // division by H (unit -> batch, head)
  // long blocks are summarised in `splits` pieces of at most `split_len`
  // tokens each; the mixing step sums the pieces (every piece of block b
  // takes the weight Mc[i, b])
  int splits, split_len;
  // tensor-core path: token chunk and chunks per piece
  ChunkShape chunk;
  int cpp;
  // one stack row per (block, piece): S_b (d*d, row-major over (k, c)),
  // z_b (d), v_b (d)
  int R;
  // number of kernel launches one forward enqueues
  int kernels;
  // workspace layout: byte offsets from the 256-aligned base
  size_t ws_total;
  size_t off_stack, off_mixed, off_rowsum, off_aux;
  size_t off_mcl;     // causal: Mc with its diagonal and upper triangle zeroed
  // tensor-core path buffers
  size_t off_stack_lo, off_mixed_lo;
  size_t off_mc_f16, off_mc_scale, off_mc_hi, off_mc_lo, off_blkinfo;
  // fp16 path: per-record exponents, per-head fp16 Mc copies, per-(head,
  // block) output scales
  size_t off_rexp, off_mcx, off_sinfo, off_mcw;
  int Qp;
  int slots;          // heads the stack and mixed buffers hold (BH, or the fused ring)
  size_t off_flow;    // fused launch: [3][BH] progress counters
  int f16_mix;        // fp16 records and mixing (DIVISIVE and NONE, multi-pass)
  // divisions by Mw and Mw * Mh (block index -> block grid coordinates)
  FastDiv f_mw, f_mwh;
  // device error word (code, detail), set by kernels whose bounded waits
  // expire
  unsigned int* err;
};

// Grid origin (x0, y0, t0) of chunk c of block b: the block's corner plus the
// chunk's offset inside it (chunks tile the block in raster order).
__host__ __device__ inline void chunk_origin(const Plan& p, const ChunkShape& ch, uint32_t b, uint32_t c, int& x0,
                                             int& y0, int& t0) {
  const uint32_t bq = fdiv(b, p.f_mw), bz = fdiv(b, p.f_mwh);
  const uint32_t bx = b - bq * (uint32_t)p.Mw, by = bq - bz * (uint32_t)p.Mh;
  const uint32_t cq = fdiv(c, ch.f_ncx), cz = fdiv(c, ch.f_ncxy);
  const uint32_t cx = c - cq * (uint32_t)ch.ncx, cy = cq - cz * (uint32_t)ch.ncy;
  x0 = (int)(bx * p.bw + cx * ch.cw);
  y0 = (int)(by * p.bh + cy * ch.ch);
  t0 = (int)(bz * p.bt + cz * ch.ct);
}

// Which mixing matrix unit u = b * H + h uses (0 when one Mc is shared).
// Matrix j occupies rows j*M .. j*M + M - 1 of every per-row array
// (Mc, its copies, row sums, block info).
__host__ __device__ inline int mc_index(const Plan& p, int u) {
  if (p.mc_heads == 1) return 0;
  return u - (int)fdiv((uint32_t)u, p.f_h) * p.H;
}

// Element offset of feature 0 of token t of unit u = b * H + h in q, k, v
// and the outputs: [B, H, N, d] (BHND) or [B, N, H, d] (BNHD, token-major as
// a fused QKV projection writes it).
__host__ __device__ inline size_t tok_off(const Plan& p, int u, int t) {
  if (p.layout == MHLA_LAYOUT_BHND) return ((size_t)u * p.N + t) * p.d;
  const int b = (int)fdiv((uint32_t)u, p.f_h), h = u - b * p.H;
  return (((size_t)b * p.N + t) * p.H + h) * p.d;
}

// Coordinates of the token tile of unit u whose corner is grid position
// (x0, y0, t0), in the 5D tensor maps encode_token_map builds:
//   BHND: axes (feature, x, y, t, unit)        -> (0, x0, y0, t0, u)
//   BNHD: axes (feature, head, x, y, batch*T+t) -> (0, h, x0, y0, b T + t0)
// (token-major: the head axis sits right after the features, and batch and
// time share one axis because a batch is N = T Hg Wg token rows).
struct TileCoords {
  int c[5];
};
__host__ __device__ inline TileCoords token_tile_coords(const Plan& p, int u, int x0, int y0, int t0) {
  TileCoords r;
  r.c[0] = 0;
  if (p.layout == MHLA_LAYOUT_BHND) {
    r.c[1] = x0;
    r.c[2] = y0;
    r.c[3] = t0;
    r.c[4] = u;
  } else {
    const int b = (int)fdiv((uint32_t)u, p.f_h);
    r.c[1] = u - b * p.H;
    r.c[2] = x0;
    r.c[3] = y0;
    r.c[4] = b * p.T + t0;
  }
  return r;
}

// Global token index (within one head) of local token l of block b.  Local
// tokens run in raster order over the (bt, bh, bw) box; blocks in raster
// order over the (Mt, Mh, Mw) block grid.
__host__ __device__ inline int block_token(const Plan& p, int b, int l) {
  int bx = b % p.Mw;
  int r = b / p.Mw;
  int by = r % p.Mh;
  int bz = r / p.Mh;
  int x = l % p.bw;
  r = l / p.bw;
  int y = r % p.bh;
  int z = r / p.bh;
  return ((bz * p.bt + z) * p.Hg + by * p.bh + y) * p.Wg + bx * p.bw + x;
}

// cudaFuncSetAttribute(kernel, MaxDynamicSharedMemorySize, bytes), done once
// per kernel and context (a launch would otherwise pay for it every time);
// returns a cudaError_t as int.
int set_max_dynamic_smem(const void* kernel, int bytes);

// Launchers implemented by the kernel translation units.  Each returns the
// cudaError_t of its launch (as int, to keep this header runtime-free).
int launch_mc_rowsum(const Plan& p, const float* mc, float* rowsum, void* stream);
int launch_simt_summary(const Plan& p, const void* k, const void* v, float* stack, void* stream);
int launch_simt_mix(const Plan& p, const float* mc, const float* stack, float* mixed, void* stream);
int launch_simt_output(const Plan& p, const void* q, const float* mixed, const float* rowsum,
                       void* out, void* stream);
// Causal form: the strict lower triangle of Mc, and the output step that walks
// each block in order (mixed = the records mixed with that triangle,
// rowsum_lower = its row sums).
int launch_mc_strict_lower(const Plan& p, const float* mc, float* mcl, void* stream);
int launch_simt_causal_output(const Plan& p, const void* q, const void* k, const void* v, const float* mixed,
                              const float* rowsum_lower, const float* mc, void* out, void* stream);

}  // namespace mhla
