// Interface between the host dispatcher and the tensor-core (tcgen05) path.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
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

int encode_tmap_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                     const uint64_t* strides_bytes, const uint32_t* box);
int num_sms();

ChunkShape choose_chunk(const Plan& p);

// Workspace pointers of the tensor-core path.
struct TcBuffers {
  __nv_bfloat16* stack_hi;  // [BH][M*splits][R]
  __nv_bfloat16* stack_lo;  // same, MALA only (else nullptr)
  __nv_bfloat16* mixed_hi;  // [BH][M][R]
  __nv_bfloat16* mixed_lo;  // [BH][M][R]
  __nv_bfloat16* mc_exp;    // [M][Qp] bf16(Mc[i][q / splits])
  __nv_bfloat16* mc_exp_lo; // [M][Qp] low bf16 residual of the same
  float* rowsum;            // [M] sum_b (hi + lo)(Mc[i][b])
  int Qp;                   // padded row pitch of mc_exp
};

int launch_tc_prep(const Plan& p, const float* mc, const TcBuffers& b, cudaStream_t s);
int launch_tc_summary(const Plan& p, const ChunkShape& c, const void* k, const void* v, const TcBuffers& b,
                      cudaStream_t s);
int launch_tc_mix(const Plan& p, const TcBuffers& b, cudaStream_t s);
int launch_tc_output(const Plan& p, const ChunkShape& c, const void* q, const TcBuffers& b, void* out,
                     cudaStream_t s);

}  // namespace mhla
