// Transpose of the mixing matrix (the gradient mixing multiplies by Mc^T).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "tc_bwd.h"

namespace mhla {
namespace {

__global__ void transpose_kernel(const float* __restrict__ in, float* __restrict__ out, int M) {
  __shared__ float t[32][33];
  in += (size_t)blockIdx.z * M * M;    // matrix blockIdx.z of a stack of M x M matrices
  out += (size_t)blockIdx.z * M * M;
  const int x = blockIdx.x * 32 + threadIdx.x, y0 = blockIdx.y * 32;
  for (int j = threadIdx.y; j < 32; j += blockDim.y)
    if (x < M && y0 + j < M) t[j][threadIdx.x] = in[(size_t)(y0 + j) * M + x];
  __syncthreads();
  const int ox = y0 + threadIdx.x, oy0 = blockIdx.x * 32;
  for (int j = threadIdx.y; j < 32; j += blockDim.y)
    if (ox < M && oy0 + j < M) out[(size_t)(oy0 + j) * M + ox] = t[threadIdx.x][j];
}

}  // namespace

int launch_transpose_mc(const float* in, float* out, int M, int count, cudaStream_t s) {
  const dim3 grid((M + 31) / 32, (M + 31) / 32, count);
  transpose_kernel<<<grid, dim3(32, 8), 0, s>>>(in, out, M);
  return (int)cudaGetLastError();
}

}  // namespace mhla
