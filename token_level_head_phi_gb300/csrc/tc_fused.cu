// Fused MHLA forward ("MHLA: Restoring Expressivity of Linear Attention via
// Token-Level Multi-Head", the three steps of Multi-Head Mixing): block
// summaries, mixing and output run as three CTA groups of ONE cooperative
// launch instead of three launches in sequence.
//
// Why: in the multi-pass path the stack of block summaries and the mixed
// summaries make a full round trip through HBM, and the mixing GEMM runs
// while no Q/K/V bytes stream.  Here the groups work through the heads in
// order, concurrently:
//   summary group: K, V of head u   -> stack slot u % ring
//   mixing group:  stack slot        -> mixed slot u % ring
//   output group:  Q of head u, mixed slot -> O
// The ring holds a few heads, so both intermediates stay in L2, and the
// streaming groups keep HBM busy while the mixing group uses the tensor
// cores.  Per-head counters in global memory order the groups:
//   s_done[u]  summary units of head u whose stack rows are stored
//   x_done[u]  mixing epilogue groups of head u whose rows are stored
//   o_done[u]  output units of head u that have read their S~_i
// The summary of head u waits for x_done[u - ring] (its slot is free), the
// mixing of head u for s_done[u] and o_done[u - ring], the output of head u
// for x_done[u].  Every dependency points to an earlier head or an earlier
// step of the same head, each group takes its units in head order, and a
// cooperative launch keeps every CTA resident, so the waits always end; each
// one is also bounded in time and reports MHLA_ERR_DEVICE_TIMEOUT.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <cstdlib>
#include <cstring>

#include "tc_mix.cuh"
#include "tc_output.cuh"
#include "tc_summary.cuh"

namespace mhla {
namespace {

using namespace tc;

constexpr int kThreads = sm::kThreads;
static_assert(ot::kThreads == kThreads && mx::kThreads <= kThreads, "bodies must fit one block shape");

struct FusedArgs {
  sm::SummaryArgs s;
  mx::MixArgs x;
  ot::OutArgs o;
  int n_s, n_x, n_o;  // CTAs of the summary, mixing and output groups (in that order)
  int ring;
  int BH;
  unsigned int* flow;  // s_done [BH] | x_done [BH] | o_done [BH]
  unsigned int need_s, need_x, need_o;
  unsigned long long wait_ns;  // limit of each counter wait (0: default)
  unsigned int stall;          // testing: the output waits for a signal that never comes
};

// Every norm mixes split (bf16 high + low) records here: the fp16 records'
// exponents are folded into Mc by a pass between the summaries and the
// mixing, which the concurrent groups do not have.
template <bool kOutLo, bool kQLo>
__global__ void __launch_bounds__(kThreads, 1) tc_fused_kernel(const __grid_constant__ FusedArgs a, const Plan p) {
  FlowCtl f;
  f.ring = a.ring;
  f.s_done = a.flow;
  f.x_done = a.flow + a.BH;
  f.o_done = a.flow + 2 * a.BH;
  f.need_s = a.need_s;
  f.need_x = a.need_x;
  f.need_o = a.need_o;
  f.wait_ns = a.wait_ns;
  f.stall = a.stall;
  const int cta = blockIdx.x;
  if (cta < a.n_s) {
    f.cta = cta;
    f.ncta = a.n_s;
    sm::summary_body<true>(a.s, p, f);
  } else if (cta < a.n_s + a.n_x) {
    f.cta = cta - a.n_s;
    f.ncta = a.n_x;
    mx::mix_body<false>(a.x, p, f);
  } else {
    f.cta = cta - a.n_s - a.n_x;
    f.ncta = a.n_o;
    ot::output_body<kOutLo, kQLo>(a.o, p, f);
  }
}

// Costs the group split assumes: a streaming CTA moves about 40 GB/s of
// Q/K/V/O; a mixing unit (128 r x NT query blocks) takes a fixed ~1.3 us
// (barriers, epilogue, stores) plus ~1.1 us per 64-deep K step of a
// 256-wide tile (the three bf16 products of the split records).
constexpr double kStreamBytesPerSmUs = 40.0e3;
constexpr double kMixUnitUs = 1.3;
constexpr double kMixStepUs = 0.45;

// Splits `total` CTAs over the three groups in proportion to their work;
// every group gets at least one CTA and none more than it has units.
// MHLA_FUSED_GROUPS="s,x,o" overrides the split (benchmark tuning).
void split_groups(const Plan& p, const FusedArgs& a, int total, int* n) {
  const char* env = getenv("MHLA_FUSED_GROUPS");
  if (env) {
    int s = 0, x = 0, o = 0;
    if (sscanf(env, "%d,%d,%d", &s, &x, &o) == 3 && s > 0 && x > 0 && o > 0 && s + x + o <= total) {
      n[0] = s;
      n[1] = x;
      n[2] = o;
      return;
    }
  }
  const double stream = (double)p.BH * p.N * p.d * 4.0;  // bytes of K+V, and of Q+O
  const double step = kMixStepUs * 2.5 * a.x.kchunks * a.x.NT / 256.0;
  const double mix = (double)a.x.units * (kMixUnitUs + step);
  const double w[3] = {stream / kStreamBytesPerSmUs, mix, stream / kStreamBytesPerSmUs};
  const int cap[3] = {a.s.units, a.x.units, a.o.units};
  const double sum = w[0] + w[1] + w[2];
  int used = 0;
  for (int g = 0; g < 3; ++g) {
    n[g] = (int)(total * w[g] / sum + 0.5);
    if (n[g] < 1) n[g] = 1;
    if (n[g] > cap[g]) n[g] = cap[g];
    used += n[g];
  }
  // trim or fill to the total, largest streaming group first
  while (used > total) {
    int g = n[0] >= n[2] ? 0 : 2;
    if (n[g] <= 1) g = 1;
    if (n[g] <= 1) break;
    --n[g];
    --used;
  }
  while (used < total) {
    int g = n[0] <= n[2] ? 0 : 2;
    if (n[g] >= cap[g]) g = 2 - g;
    if (n[g] >= cap[g]) break;
    ++n[g];
    ++used;
  }
}

template <bool kOutLo, bool kQLo>
int launch_variant(FusedArgs& a, const Plan& p, cudaStream_t s) {
  auto kern = tc_fused_kernel<kOutLo, kQLo>;
  uint32_t smem = summary_smem_bytes(true);
  if (mix_smem_bytes() > smem) smem = mix_smem_bytes();
  if (output_smem_bytes(kOutLo, kQLo) > smem) smem = output_smem_bytes(kOutLo, kQLo);
  cudaError_t ce = (cudaError_t)set_max_dynamic_smem((const void*)kern, (int)smem);
  if (ce != cudaSuccess) return (int)ce;
  int dev = 0, coop = 0, per_sm = 0;
  if ((ce = cudaGetDevice(&dev)) != cudaSuccess) return (int)ce;
  if ((ce = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev)) != cudaSuccess) return (int)ce;
  if (!coop) return (int)cudaErrorNotSupported;
  if ((ce = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem)) != cudaSuccess)
    return (int)ce;
  if (per_sm < 1) return (int)cudaErrorNotSupported;
  const int total = num_sms() * per_sm;
  if (total < 3) return (int)cudaErrorNotSupported;
  int n[3];
  split_groups(p, a, total, n);
  a.n_s = n[0];
  a.n_x = n[1];
  a.n_o = n[2];

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(n[0] + n[1] + n[2]));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  ce = cudaLaunchKernelEx(&cfg, kern, a, p);
  if (ce != cudaSuccess) return (int)ce;
  return (int)cudaGetLastError();
}

}  // namespace

int launch_tc_fused(const Plan& p, const ChunkShape& c, const void* q, const void* k, const void* v,
                    const TcBuffers& b, void* out, cudaStream_t s) {
  if (!b.flow || b.slots < 1) return (int)cudaErrorInvalidValue;
  FusedArgs a;
  memset(&a, 0, sizeof(a));
  int e;
  if ((e = build_summary_args(p, c, k, v, b, b.slots, &a.s)) != 0) return e;
  if ((e = build_mix_args(p, b, b.slots, &a.x)) != 0) return e;
  if ((e = build_output_args(p, c, q, b, out, b.slots, &a.o)) != 0) return e;
  a.ring = b.slots < p.BH ? b.slots : 0;
  a.BH = p.BH;
  a.flow = b.flow;
  a.need_s = (unsigned)(p.M * p.splits);
  a.need_x = (unsigned)(mx::kEpiGroups * a.x.rtiles * a.x.itiles);
  a.need_o = (unsigned)(p.M * c.per_block);
  a.wait_ns = debug_flow_wait_ns();
  a.stall = debug_flow_stall();
  if (tc_q_lo(p)) return tc_out_lo(p) ? launch_variant<true, true>(a, p, s) : launch_variant<false, true>(a, p, s);
  return tc_out_lo(p) ? launch_variant<true, false>(a, p, s) : launch_variant<false, false>(a, p, s);
}

}  // namespace mhla
