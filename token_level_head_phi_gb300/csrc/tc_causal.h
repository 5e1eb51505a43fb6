// Tensor-core output step of the block-ordered causal form.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "tc_host.h"

namespace mhla {

// Whether the tensor-core causal output step applies: DIVISIVE or NONE, and
// token chunks that are contiguous runs of their block's local order.
bool tc_causal_supported(const Plan& p);

// out for every token from Q, K, V and the records mixed with the strict
// lower triangle of Mc (bf16 high + low planes [BH][M][R]); mc supplies the
// diagonal weight of each block's own tokens.
int launch_tc_causal(const Plan& p, const void* q, const void* k, const void* v, const __nv_bfloat16* mixed_hi,
                     const __nv_bfloat16* mixed_lo, const float* mc, void* out, cudaStream_t s);

}  // namespace mhla
