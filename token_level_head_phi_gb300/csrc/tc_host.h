// Interface between the host dispatcher and the tensor-core (tcgen05) path.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "plan.h"

namespace mhla {

// Head dimension the tensor-core kernels are written for: one 128-byte row
// of bf16 per token, one 64-wide swizzle atom.
constexpr int kTcHeadDim = 64;
// Largest token tile one MMA row block holds.
constexpr int kTcTileRows = 128;
// SM count the planner assumes when it splits long blocks (the workspace
// size must not depend on the device).
constexpr int kPlanSms = 152;

// Tiled TMA tensor map with 128-byte swizzle over 2-byte elements (bf16, or
// fp16 when f16 is set); dims[0] innermost, strides_bytes[i] is the stride of
// dims[i + 1].
int encode_tmap(CUtensorMap* map, const void* base, int rank, const uint64_t* dims, const uint64_t* strides_bytes,
                const uint32_t* box, bool f16);
// Same without swizzle (row-major boxes in shared memory), bf16.
int encode_tmap_plain(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                      const uint64_t* strides_bytes, const uint32_t* box);
inline int encode_tmap_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                            const uint64_t* strides_bytes, const uint32_t* box) {
  return encode_tmap(map, base, rank, dims, strides_bytes, box, false);
}
int num_sms();
// 5D map over q, k, v, an output or a gradient tensor in the plan's layout,
// box = one token chunk (64, cw, ch, ct, 1); see unit_coords for the
// coordinates.
int encode_token_map(CUtensorMap* map, const Plan& p, const void* base, const ChunkShape& c);

ChunkShape choose_chunk(const Plan& p);

// Workspace pointers of the tensor-core path.  Stack rows are block pieces
// (Q = M * splits per head), each a record of R = d*d + 2d values: S_b
// (row-major over (k, c)), z_b, v_b.
// The stack and the mixed summaries hold `slots` heads: every head (slots =
// BH) for the multi-pass launches, a ring of heads reused in turn for the
// fused launch.
//
// Two precisions.  fp16 (DIVISIVE and NONE, multi-pass): record q holds
// S_b * 2^-eS[q] and z_b * 2^-eZ[q] in fp16 (v_b, which only MALA reads, is
// stored as zeros), the exponents chosen from the record's own largest
// entries; the mixing multiplies by per-head fp16 copies of Mc into which
// those exponents are folded (mcx), and the output step applies a per-(head,
// block) power of two (sinfo).  Split (MALA, the causal form, the fused
// launch, the backward's recomputation): every record as bf16 high + low
// parts, Mc as bf16 high + low parts.
struct TcBuffers {
  void* stack;               // [slots][Q][R]: fp16 scaled record (fp16 path) or bf16 high part (split)
  __nv_bfloat16* stack_lo;   // [slots][Q][R] low bf16 residual (split path, else nullptr)
  __nv_bfloat16* mixed_hi;   // [slots][M][R] S~_i, z~_i, v~_i high parts (fp16 path: times 2^-ES, 2^-EZ)
  __nv_bfloat16* mixed_lo;   // [slots][M][R] low residuals (S~ part for MALA only)
  __half* mc_f16;            // [M][Qp] Mc[i][q / splits] * 2^-e_i in fp16 (unused by the fp16 path)
  float* mc_scale;           // [M] 2^e_i (power of two with max_b |Mc[i][b]| <= 2^e_i)
  __nv_bfloat16* mc_hi;      // [M][Qp] bf16(Mc[i][q / splits])
  __nv_bfloat16* mc_lo;      // [M][Qp] low bf16 residual of the same
  float* rowsum;             // [M] sum_b (hi + lo)(Mc[i][b])
  float4* blkinfo;           // [M] {1, n~_i, 0, 0} (split path)
  int2* rexp;                // fp16 path: [slots][Q] record exponents {eS, eZ}
  uint32_t* mcw;             // fp16 path: [M][Qp] Mc[i][q / splits] as {fp16 bits of its mantissa in
                             //            [1, 2) (with sign), x + 8192 in the high 16 bits} with
                             //            Mc = mantissa 2^(x - 1); 0 for a zero entry
  __half* mcx;               // fp16 path: [slots][2][M][Qp] Mc[i][q / splits] 2^(eS[q] - ES[i]) (part 0),
                             //            the same with eZ, EZ (part 1)
  float4* sinfo;             // fp16 path: [slots][M] {output scale, 0, 0, 0}
  int Qp;                    // padded row pitch of the Mc copies
  bool f16;                  // fp16 records and mixing
  int slots;                 // heads the stack and mixed buffers hold
  unsigned int* flow;        // fused launch: [3][BH] progress counters, zeroed by the prep kernel
  bool no_prep;              // the summary kernel is the call's first kernel
};

// Whether the output step multiplies phi(Q) by the low residual of S~_i too
// (a second MMA per K step), which the mixing then writes.  MALA cancels its
// leading terms; exponential features let a few tokens dominate every
// feature, so the bf16 rounding of S~_i no longer averages out.
inline bool tc_out_lo(const Plan& p) { return p.norm == MHLA_NORM_MALA || p.fmap == MHLA_FEATURE_EXP; }
// Whether phi(Q) enters the output step as bf16 high + low parts
// (exponential features: the rounding of e^q to bf16 does not average out
// either, and MALA's cancellation amplifies it).
inline bool tc_q_lo(const Plan& p) { return p.fmap == MHLA_FEATURE_EXP; }

// Launch with programmatic stream serialization (the kernel's body calls
// pdl_wait before it reads its predecessor's results).
template <typename... KArgs, typename... Args>
int launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
  return e != cudaSuccess ? (int)e : (int)cudaGetLastError();
}

int launch_tc_prep(const Plan& p, const float* mc, const TcBuffers& b, cudaStream_t s);
int launch_tc_summary(const Plan& p, const ChunkShape& c, const void* k, const void* v, const TcBuffers& b,
                      cudaStream_t s);
// fp16 path, between the summaries and the mixing: the per-head Mc copies
// with the record exponents folded in, and the output scales.
int launch_tc_scale(const Plan& p, const TcBuffers& b, cudaStream_t s);
int launch_tc_mix(const Plan& p, const TcBuffers& b, cudaStream_t s);
// Mixing of few blocks on the CUDA cores (tc_mixs.cu): M <= kSmallMixMaxM query
// blocks and Q <= kSmallMixMaxQ records per head, read from the tensor-core
// records, written as launch_tc_mix writes them (fp16 records need no
// launch_tc_scale before it).
constexpr int kSmallMixMaxM = 16;
constexpr int kSmallMixMaxQ = 256;
bool small_mix_supported(const Plan& p);
int launch_tc_mix_small(const Plan& p, const float* mc, const TcBuffers& b, cudaStream_t s);
int launch_tc_output(const Plan& p, const ChunkShape& c, const void* q, const TcBuffers& b, void* out,
                     cudaStream_t s);
// Testing hooks set by mhla_set_debug: limit of the fused launch's counter
// waits (0: default) and whether the output group demands one signal more
// than will come.
unsigned long long debug_flow_wait_ns();
unsigned int debug_flow_stall();

// Summary, mixing and output in one cooperative launch (after launch_tc_prep).
int launch_tc_fused(const Plan& p, const ChunkShape& c, const void* q, const void* k, const void* v,
                    const TcBuffers& b, void* out, cudaStream_t s);

}  // namespace mhla
