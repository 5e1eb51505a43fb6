// Interface between the host dispatcher and the tensor-core backward kernels
// (head dimension 64, bf16 tensors).  Intermediate records are kept as two
// bf16 planes, high and low parts of a float32 value (hi = bf16(x),
// lo = bf16(x - hi)), in the record layout of the forward stack: one row of
// R = d*d + 2d values per (head, block piece) or (head, block).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "tc_host.h"

namespace mhla {

// dMc from the gradient records dX~ (dx planes, [BH][Q][R]) and the forward
// records X (x planes, [BH][Q][R]), Q = M * splits piece rows; `partial`
// holds tc_bwd_mc_partial_bytes(p) bytes; dnp [BH][Q] is read for MALA only.
size_t tc_bwd_mc_partial_bytes(const Plan& p);
int launch_tc_bwd_mc(const Plan& p, const __nv_bfloat16* dx_hi, const __nv_bfloat16* dx_lo,
                     const __nv_bfloat16* x_hi, const __nv_bfloat16* x_lo, const float* dnp, float* partial,
                     float* dmc, cudaStream_t s);

// dK, dV from the gradient records dX_b = (dS_b, dz_b, dv_b) (dx planes,
// [BH][M][R]) and the K, V tensors ([B, H, N, 64] bf16).
int launch_tc_bwd_summary(const Plan& p, const void* k, const void* v, const __nv_bfloat16* dx_hi,
                          const __nv_bfloat16* dx_lo, void* dk, void* dv, cudaStream_t s);

// dq and the per-piece gradient records dX~ (dS~, dz~, dv~ as dx planes,
// [BH][Q][R]; dn~ into dnp [BH][Q] for MALA) from Q, dO and the mixed
// forward records (planes [BH][M][R], blkinfo as the forward prep writes it).
int launch_tc_bwd_output(const Plan& p, const void* q, const void* dout, const __nv_bfloat16* mixed_hi,
                         const __nv_bfloat16* mixed_lo, const float4* blkinfo, void* dq, __nv_bfloat16* dx_hi,
                         __nv_bfloat16* dx_lo, float* dnp, cudaStream_t s);

// out[j][b][i] = in[j][i][b] for `count` M x M float32 matrices.
int launch_transpose_mc(const float* in, float* out, int M, int count, cudaStream_t s);

}  // namespace mhla
