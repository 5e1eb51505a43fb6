// Standalone launch of the block-summary kernel (body in tc_summary.cuh).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstring>

#include "tc_summary.cuh"

namespace mhla {
namespace {

using namespace tc;
using sm::Layout;
using sm::SummaryArgs;
using sm::kThreads;

template <bool kLo>
__global__ void __launch_bounds__(kThreads, 1) tc_summary_kernel(const __grid_constant__ SummaryArgs a, const Plan p) {
  FlowCtl f = {};
  f.cta = blockIdx.x;
  f.ncta = gridDim.x;
  sm::summary_body<kLo>(a, p, f);
}

template <bool kLo>
int launch_variant(const SummaryArgs& a, const Plan& p, cudaStream_t s) {
  const uint32_t smem = Layout<kLo>::kSmemBytes;
  cudaError_t ce = (cudaError_t)set_max_dynamic_smem((const void*)tc_summary_kernel<kLo>, (int)smem);
  if (ce != cudaSuccess) return (int)ce;
  const int grid = a.units < num_sms() ? a.units : num_sms();
  return launch_pdl(tc_summary_kernel<kLo>, dim3(grid), dim3(kThreads), smem, s, a, p);
}

}  // namespace

int build_summary_args(const Plan& p, const ChunkShape& c, const void* k, const void* v, const TcBuffers& b,
                       int slots, sm::SummaryArgs* out) {
  SummaryArgs& a = *out;
  memset(&a, 0, sizeof(a));
  int e;
  if ((e = encode_token_map(&a.tmK, p, k, c)) != 0) return e;
  if ((e = encode_token_map(&a.tmV, p, v, c)) != 0) return e;
  // the stack holds `slots` heads: every head (standalone) or a ring (fused)
  const uint64_t stack_rows = (uint64_t)slots * p.M * p.splits * 66ull;
  const uint64_t dims2[2] = {64, stack_rows};
  const uint64_t str2[1] = {128};
  const uint32_t boxS[2] = {64, 64};
  const uint32_t boxZV[2] = {64, 2};
  const bool lo = b.stack_lo != nullptr;  // MALA: phi(K) and the stack carry low residuals
  const void* lo_base = lo ? (const void*)b.stack_lo : b.stack;
  if ((e = encode_tmap(&a.tmS, b.stack, 2, dims2, str2, boxS, b.f16)) != 0) return e;
  if ((e = encode_tmap(&a.tmZV, b.stack, 2, dims2, str2, boxZV, b.f16)) != 0) return e;
  if ((e = encode_tmap_bf16(&a.tmS_lo, lo_base, 2, dims2, str2, boxS)) != 0) return e;
  if ((e = encode_tmap_bf16(&a.tmZV_lo, lo_base, 2, dims2, str2, boxZV)) != 0) return e;
  a.rexp = b.rexp;
  a.wait_prev = b.no_prep ? 1 : 0;
  a.splits = p.splits;
  a.cpp = p.cpp;
  a.units = p.BH * p.M * p.splits;
  a.f_head = make_fastdiv((uint32_t)(p.M * p.splits));
  a.f_splits = make_fastdiv((uint32_t)p.splits);
  a.c = c;
  a.err = p.err;
  return 0;
}

uint32_t summary_smem_bytes(bool lo) { return lo ? Layout<true>::kSmemBytes : Layout<false>::kSmemBytes; }

int launch_tc_summary(const Plan& p, const ChunkShape& c, const void* k, const void* v, const TcBuffers& b,
                      cudaStream_t s) {
  SummaryArgs a;
  int e = build_summary_args(p, c, k, v, b, b.slots, &a);
  if (e != 0) return e;
  return b.stack_lo ? launch_variant<true>(a, p, s) : launch_variant<false>(a, p, s);
}

}  // namespace mhla
