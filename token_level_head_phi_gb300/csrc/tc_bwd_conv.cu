// Float32 records <-> bf16 high/low planes.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "tc_bwd.h"

namespace mhla {
namespace {

__global__ void planes_to_f32_kernel(const __nv_bfloat16* __restrict__ hi, const __nv_bfloat16* __restrict__ lo,
                                     float* __restrict__ out, size_t n) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
    out[i] = __bfloat162float(hi[i]) + __bfloat162float(lo[i]);
}

__global__ void f32_to_planes_kernel(const float* __restrict__ in, __nv_bfloat16* __restrict__ hi,
                                     __nv_bfloat16* __restrict__ lo, size_t n) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const float x = in[i];
    const __nv_bfloat16 h = __float2bfloat16_rn(x);
    hi[i] = h;
    lo[i] = __float2bfloat16_rn(x - __bfloat162float(h));
  }
}

__global__ void transpose_kernel(const float* __restrict__ in, float* __restrict__ out, int M) {
  __shared__ float t[32][33];
  const int x = blockIdx.x * 32 + threadIdx.x, y0 = blockIdx.y * 32;
  for (int j = threadIdx.y; j < 32; j += blockDim.y)
    if (x < M && y0 + j < M) t[j][threadIdx.x] = in[(size_t)(y0 + j) * M + x];
  __syncthreads();
  const int ox = y0 + threadIdx.x, oy0 = blockIdx.x * 32;
  for (int j = threadIdx.y; j < 32; j += blockDim.y)
    if (ox < M && oy0 + j < M) out[(size_t)(oy0 + j) * M + ox] = t[threadIdx.x][j];
}

int grid_for(size_t n) {
  const size_t g = (n + 255) / 256;
  return (int)(g < 4096 ? (g < 1 ? 1 : g) : 4096);
}

}  // namespace

int launch_transpose_mc(const float* in, float* out, int M, cudaStream_t s) {
  const dim3 grid((M + 31) / 32, (M + 31) / 32);
  transpose_kernel<<<grid, dim3(32, 8), 0, s>>>(in, out, M);
  return (int)cudaGetLastError();
}

int launch_planes_to_f32(const __nv_bfloat16* hi, const __nv_bfloat16* lo, float* out, size_t n, cudaStream_t s) {
  planes_to_f32_kernel<<<grid_for(n), 256, 0, s>>>(hi, lo, out, n);
  return (int)cudaGetLastError();
}

int launch_f32_to_planes(const float* in, __nv_bfloat16* hi, __nv_bfloat16* lo, size_t n, cudaStream_t s) {
  f32_to_planes_kernel<<<grid_for(n), 256, 0, s>>>(in, hi, lo, n);
  return (int)cudaGetLastError();
}

}  // namespace mhla
