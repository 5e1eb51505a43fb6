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
struct TcBuffers {
  void* stack;               // [slots][Q][R]: fp16(x * stack_scale) (DIVISIVE/NONE) or bf16 high part (MALA)
  __nv_bfloat16* stack_lo;   // [slots][Q][R] low bf16 residual (MALA only, else nullptr)
  __nv_bfloat16* mixed_hi;   // [slots][M][R] S~_i, z~_i, v~_i high parts
  __nv_bfloat16* mixed_lo;   // [slots][M][R] low residuals (S~ part for MALA only)
  __half* mc_f16;            // [M][Qp] Mc[i][q / splits] * 2^-e_i in fp16
  float* mc_scale;           // [M] 2^e_i (power of two with max_b |Mc[i][b]| <= 2^e_i)
  __nv_bfloat16* mc_hi;      // [M][Qp] bf16(Mc[i][q / splits])
  __nv_bfloat16* mc_lo;      // [M][Qp] low bf16 residual of the same
  float* rowsum;             // [M] sum_b (hi + lo)(Mc[i][b])
  float4* blkinfo;           // [M] {scale the output step applies to S~_i, n~_i, 0, 0}
  int Qp;                    // padded row pitch of the Mc copies
  bool f16;                  // fp16 stack and mixing (DIVISIVE and NONE)
  float stack_scale;         // 2^-ceil(log2(tokens per piece))
  int slots;                 // heads the stack and mixed buffers hold
  unsigned int* flow;        // fused launch: [3][BH] progress counters, zeroed by the prep kernel
};

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
int launch_tc_mix(const Plan& p, const TcBuffers& b, cudaStream_t s);
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
