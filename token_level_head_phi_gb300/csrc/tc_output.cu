// Standalone launch of the output kernel (body in tc_output.cuh).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstring>

#include "tc_output.cuh"

namespace mhla {
namespace {

using namespace tc;
using ot::OutArgs;
using ot::kThreads;

template <bool kLo, bool kQLo>
__global__ void __launch_bounds__(ot::kThreads, 1) tc_output_kernel(const __grid_constant__ ot::OutArgs a, const Plan p) {
  FlowCtl f = {};
  f.cta = blockIdx.x;
  f.ncta = gridDim.x;
  ot::output_body<kLo, kQLo>(a, p, f);
}

template <bool kLo, bool kQLo>
int launch_variant(const OutArgs& a, const Plan& p, cudaStream_t s) {
  const uint32_t smem = output_smem_bytes(kLo, kQLo);
  auto kern = tc_output_kernel<kLo, kQLo>;
  cudaError_t ce = (cudaError_t)set_max_dynamic_smem((const void*)kern, (int)smem);
  if (ce != cudaSuccess) return (int)ce;
  const int grid = a.units < num_sms() ? a.units : num_sms();
  return launch_pdl(kern, dim3(grid), dim3(kThreads), smem, s, a, p);
}

}  // namespace

int build_output_args(const Plan& p, const ChunkShape& c, const void* q, const TcBuffers& b, void* out, int slots,
                      ot::OutArgs* args) {
  OutArgs& a = *args;
  memset(&a, 0, sizeof(a));
  int e;
  if ((e = encode_token_map(&a.tmQ, p, q, c)) != 0) return e;
  if ((e = encode_token_map(&a.tmO, p, out, c)) != 0) return e;
  const uint64_t dims3[3] = {64, (uint64_t)(p.R / 64), (uint64_t)slots * p.M};
  const uint64_t str3[2] = {128, 2ull * p.R};
  const uint32_t box3[3] = {64, 64, 1};
  if ((e = encode_tmap_bf16(&a.tmB_hi, b.mixed_hi, 3, dims3, str3, box3)) != 0) return e;
  if ((e = encode_tmap_bf16(&a.tmB_lo, b.mixed_lo, 3, dims3, str3, box3)) != 0) return e;
  a.blkinfo = b.f16 ? b.sinfo : b.blkinfo;
  a.info_per_slot = b.f16 ? 1 : 0;
  a.mixed_hi = b.mixed_hi;
  a.mixed_lo = b.mixed_lo;
  a.R = p.R;
  a.units = p.BH * p.M * c.per_block;
  a.f_head = make_fastdiv((uint32_t)(p.M * c.per_block));
  a.f_nck = make_fastdiv((uint32_t)c.per_block);
  a.c = c;
  a.err = p.err;
  return 0;
}

int launch_tc_output(const Plan& p, const ChunkShape& c, const void* q, const TcBuffers& b, void* out,
                     cudaStream_t s) {
  OutArgs a;
  int e = build_output_args(p, c, q, b, out, b.slots, &a);
  if (e != 0) return e;
  if (tc_q_lo(p)) return tc_out_lo(p) ? launch_variant<true, true>(a, p, s) : launch_variant<false, true>(a, p, s);
  return tc_out_lo(p) ? launch_variant<true, false>(a, p, s) : launch_variant<false, false>(a, p, s);
}

}  // namespace mhla
