// Small device helpers shared by the kernels: the feature map and element
// conversions.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "plan.h"

namespace mhla {

// phi = ELU(x) + 1 with alpha = 1 ("MHLA: Restoring Expressivity of Linear
// Attention via Token-Level Multi-Head", background: a positive feature map
// with Sim(Q_i, K_j) ~ phi(Q_i) phi(K_j)^T); ReLU and exp, the other maps of
// the kernel-function ablation of "Rectifying Magnitude Neglect in Linear
// Attention".  IDENTITY is the test-only map.
__device__ __forceinline__ float phi_apply(float x, int fmap) {
  if (fmap == MHLA_FEATURE_IDENTITY) return x;
  if (fmap == MHLA_FEATURE_RELU) return fmaxf(x, 0.f);
  if (fmap == MHLA_FEATURE_EXP) return expf(x);
  return x > 0.f ? x + 1.f : expf(x);
}

// phi'(x) given x and phi(x) (ReLU: 0 at and below zero).
__device__ __forceinline__ float phi_deriv(float x, float phi, int fmap) {
  if (fmap == MHLA_FEATURE_IDENTITY) return 1.f;
  if (fmap == MHLA_FEATURE_RELU) return x > 0.f ? 1.f : 0.f;
  if (fmap == MHLA_FEATURE_EXP) return phi;
  return x > 0.f ? 1.f : phi;
}

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

}  // namespace mhla
