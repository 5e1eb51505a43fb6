// C ABI of libmhla.so (declared in include/mhla.h): argument validation,
// planning, workspace layout and dispatch to the kernels.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <atomic>
#include <mutex>
#include <string>

#include "mhla.h"
#include "plan.h"
#include "backward.h"
#include "tc_bwd.h"
#include "tc_causal.h"
#include "tc_host.h"

namespace mhla {

// Testing hooks of the fused launch (mhla_set_debug).
std::atomic<unsigned long long> g_debug_flow_wait_ns{0};
std::atomic<unsigned int> g_debug_flow_stall{0};
unsigned long long debug_flow_wait_ns() { return g_debug_flow_wait_ns.load(); }
unsigned int debug_flow_stall() { return g_debug_flow_stall.load(); }

namespace {

thread_local std::string g_last_error;

std::mutex g_events_mu;
cudaEvent_t g_events[MHLA_NUM_PHASE_EVENTS];
int g_num_events = 0;
cudaEvent_t g_bwd_events[MHLA_NUM_BWD_PHASE_EVENTS];
int g_num_bwd_events = 0;

// Device error word: [0] status code, [1] location detail.  Kernels with
// bounded waits write it when a wait expires.
__device__ unsigned int g_device_error[2];

constexpr int kMaxDevices = 64;
std::mutex g_err_mu;
unsigned int* g_err_ptr[kMaxDevices] = {};

constexpr size_t kAlign = 256;
constexpr int kSimtSplitLen = 1024;
// Fused launch: the stack and mixed-summary rings take at most this many
// bytes (well inside the 126 MB L2, which also carries the Q/K/V/O streams)
// and hold at most kFusedMaxRing heads.
constexpr size_t kFusedRingBytes = 48ull << 20;
constexpr size_t kFusedMaxRing = 16;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

mhla_status cuda_fail(cudaError_t e) {
  g_last_error = cudaGetErrorString(e);
  return MHLA_ERR_CUDA;
}

size_t elem_bytes(int dtype) { return dtype == MHLA_DTYPE_BF16 ? 2 : 4; }

mhla_status device_error_ptr(unsigned int** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return MHLA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_err_mu);
  if (!g_err_ptr[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_device_error);
    if (e != cudaSuccess) return cuda_fail(e);
    g_err_ptr[dev] = static_cast<unsigned int*>(ptr);
  }
  *out = g_err_ptr[dev];
  return MHLA_OK;
}

// Shape and option checks; fills the plan without touching the device.
// split_units: the number of (batch, head) units the split of long blocks is
// sized for (0: this problem's own); a group of a larger problem passes the
// whole problem's count so that it sums the same pieces in the same order.
mhla_status make_plan(const mhla_params* prm, Plan* p, int split_units = 0) {
  if (!prm || !p) return MHLA_ERR_INVALID_ARG;
  std::memset(p, 0, sizeof(*p));
  const int d = prm->head_dim;
  if (prm->batch < 0 || prm->heads < 0) return MHLA_ERR_INVALID_ARG;
  if (d != 16 && d != 32 && d != 64 && d != 128) return MHLA_ERR_INVALID_ARG;
  for (int i = 0; i < 3; ++i) {
    if (prm->grid[i] < 1 || prm->block[i] < 1) return MHLA_ERR_INVALID_ARG;
    if (prm->grid[i] % prm->block[i] != 0) return MHLA_ERR_INVALID_ARG;
  }
  if (prm->dtype != MHLA_DTYPE_BF16 && prm->dtype != MHLA_DTYPE_F32) return MHLA_ERR_INVALID_ARG;
  if (prm->feature_map < MHLA_FEATURE_ELU1 || prm->feature_map > MHLA_FEATURE_EXP)
    return MHLA_ERR_INVALID_ARG;
  if (prm->norm != MHLA_NORM_DIVISIVE && prm->norm != MHLA_NORM_MALA && prm->norm != MHLA_NORM_NONE)
    return MHLA_ERR_INVALID_ARG;
  if (prm->variant != MHLA_VARIANT_AUTO && prm->variant != MHLA_VARIANT_SIMT &&
      prm->variant != MHLA_VARIANT_MULTIPASS && prm->variant != MHLA_VARIANT_FUSED)
    return MHLA_ERR_INVALID_ARG;
  if (prm->causal != 0 && prm->causal != 1) return MHLA_ERR_INVALID_ARG;
  if (prm->layout != MHLA_LAYOUT_BHND && prm->layout != MHLA_LAYOUT_BNHD) return MHLA_ERR_INVALID_ARG;
  if (prm->mc_per_head != 0 && prm->mc_per_head != 1) return MHLA_ERR_INVALID_ARG;
  // the fused launch keeps one Mc resident per CTA group
  if (prm->mc_per_head && prm->variant == MHLA_VARIANT_FUSED) return MHLA_ERR_UNSUPPORTED;

  const int64_t N64 = (int64_t)prm->grid[0] * prm->grid[1] * prm->grid[2];
  const int64_t BH64 = (int64_t)prm->batch * prm->heads;
  if (N64 > (1LL << 30) || BH64 > 65535) return MHLA_ERR_UNSUPPORTED;
  if (BH64 * N64 * d > (1LL << 40)) return MHLA_ERR_UNSUPPORTED;

  p->B = prm->batch;
  p->H = prm->heads;
  p->BH = (int)BH64;
  p->d = d;
  p->T = prm->grid[0];
  p->Hg = prm->grid[1];
  p->Wg = prm->grid[2];
  p->bt = prm->block[0];
  p->bh = prm->block[1];
  p->bw = prm->block[2];
  p->Mt = p->T / p->bt;
  p->Mh = p->Hg / p->bh;
  p->Mw = p->Wg / p->bw;
  p->N = (int)N64;
  const int64_t M64 = (int64_t)p->Mt * p->Mh * p->Mw;
  if (M64 > 65536) return MHLA_ERR_UNSUPPORTED;
  p->M = (int)M64;
  p->f_mw = make_fastdiv((uint32_t)p->Mw);
  p->f_mwh = make_fastdiv((uint32_t)(p->Mw * p->Mh));
  p->nb = p->bt * p->bh * p->bw;
  p->dtype = prm->dtype;
  p->fmap = prm->feature_map;
  p->norm = prm->norm;
  p->causal = prm->causal;
  p->layout = prm->layout;
  p->mc_heads = prm->mc_per_head ? (p->H > 0 ? p->H : 1) : 1;
  p->f_h = make_fastdiv((uint32_t)(p->H > 0 ? p->H : 1));

  bool tc_ok = prm->dtype == MHLA_DTYPE_BF16 && d == kTcHeadDim;
  if (tc_ok && prm->causal) {
    // the tensor-core causal output step: DIVISIVE / NONE with token chunks
    // that are contiguous runs of the block's local order; never fused
    Plan probe = *p;
    probe.chunk = choose_chunk(probe);
    tc_ok = tc_causal_supported(probe) && prm->variant != MHLA_VARIANT_FUSED;
  }
  int variant = prm->variant;
  if (variant == MHLA_VARIANT_AUTO) variant = tc_ok ? MHLA_VARIANT_MULTIPASS : MHLA_VARIANT_SIMT;
  if ((variant == MHLA_VARIANT_MULTIPASS || variant == MHLA_VARIANT_FUSED) && !tc_ok) return MHLA_ERR_UNSUPPORTED;
  p->variant = variant;
  p->R = d * d + 2 * d;
  p->kernels = 4;

  if (variant == MHLA_VARIANT_SIMT) {
    // pieces of at most kSimtSplitLen tokens
    p->splits = (p->nb + kSimtSplitLen - 1) / kSimtSplitLen;
    p->split_len = (p->nb + p->splits - 1) / p->splits;
  } else {
    // token chunks of <= 128 rows; blocks are cut into pieces only when there
    // are too few blocks to keep every SM busy for several waves
    p->chunk = choose_chunk(*p);
    const int nck = p->chunk.per_block;
    const int64_t blocks = (int64_t)(split_units > 0 ? split_units : p->BH) * p->M;
    int splits = 1;
    if (blocks > 0 && blocks < 8LL * kPlanSms)
      splits = (int)((8LL * kPlanSms + blocks - 1) / blocks);
    if (splits > nck) splits = nck;
    if (splits < 1) splits = 1;
    p->cpp = (nck + splits - 1) / splits;
    p->splits = (nck + p->cpp - 1) / p->cpp;
    p->split_len = p->cpp * p->chunk.rows;
    p->Qp = (p->M * p->splits + 7) / 8 * 8;
    // fp16 records and mixing for DIVISIVE and NONE in the multi-pass launch.
    // MALA cancels its leading terms and needs the split (bf16 high + low)
    // records and phi(K); so do exponential features, where a few tokens
    // dominate each feature and the bf16 rounding of phi(K) no longer
    // averages out; so does the causal output step, which adds its in-block
    // terms in float32 to the mixed prefix records; the fused launch has no
    // pass between its summary and mixing groups to fold the records'
    // exponents into Mc, so it takes the split records too.
    p->f16_mix = p->norm != MHLA_NORM_MALA && p->fmap != MHLA_FEATURE_EXP && !p->causal &&
                 variant == MHLA_VARIANT_MULTIPASS;
  }

  if (p->BH == 0) {
    p->ws_total = 0;
    p->kernels = 0;
    return MHLA_OK;
  }
  size_t off = 0;
  if (variant == MHLA_VARIANT_SIMT) {
    p->off_stack = off;
    off = align_up(off + sizeof(float) * (size_t)p->BH * p->M * p->splits * p->R);
    p->off_mixed = off;
    off = align_up(off + sizeof(float) * (size_t)p->BH * p->M * p->R);
    p->off_rowsum = off;
    off = align_up(off + sizeof(float) * (size_t)p->M * p->mc_heads);
    if (p->causal) {
      p->off_mcl = off;
      off = align_up(off + sizeof(float) * (size_t)p->M * p->M * p->mc_heads);
      p->kernels = 5;
    }
  } else {
    // fused: a ring of heads small enough to stay in L2 (at least two, so
    // that consecutive heads overlap)
    const size_t per_head = 2 * (size_t)p->M * p->splits * p->R * (p->f16_mix ? 1 : 2) +
                            4 * (size_t)p->M * p->R;
    p->slots = p->BH;
    if (variant == MHLA_VARIANT_FUSED) {
      size_t ring = kFusedRingBytes / per_head;
      if (ring < 2) ring = 2;
      if (ring > kFusedMaxRing) ring = kFusedMaxRing;
      if (ring < (size_t)p->slots) p->slots = (int)ring;
    }
    const size_t rows = (size_t)p->slots * p->M * p->splits;
    const size_t stack = 2 * rows * p->R;
    const size_t mixed = 2 * (size_t)p->slots * p->M * p->R;
    const size_t mcq = 2 * (size_t)p->M * p->mc_heads * p->Qp;
    p->off_stack = off;
    off = align_up(off + stack);
    p->off_stack_lo = off;
    if (!p->f16_mix) off = align_up(off + stack);
    p->off_mixed = off;
    off = align_up(off + mixed);
    p->off_mixed_lo = off;
    off = align_up(off + mixed);
    p->off_mc_f16 = off;
    off = align_up(off + mcq);
    p->off_mc_hi = off;
    off = align_up(off + mcq);
    p->off_mc_lo = off;
    off = align_up(off + mcq);
    p->off_mc_scale = off;
    off = align_up(off + sizeof(float) * (size_t)p->M * p->mc_heads);
    p->off_rowsum = off;
    off = align_up(off + sizeof(float) * (size_t)p->M * p->mc_heads);
    p->off_blkinfo = off;
    off = align_up(off + 16 * (size_t)p->M * p->mc_heads);
    p->kernels = 4;
    if (p->f16_mix) {
      p->off_rexp = off;
      off = align_up(off + 8 * rows);
      p->off_mcx = off;
      off = align_up(off + 2 * 2 * (size_t)p->slots * p->M * p->Qp);
      p->off_sinfo = off;
      off = align_up(off + 16 * (size_t)p->slots * p->M);
      p->off_mcw = off;
      off = align_up(off + 4 * (size_t)p->M * p->mc_heads * p->Qp);
      // few blocks: the CUDA-core mixing reads the record exponents itself
      // few blocks: no prep kernel, no exponent folding
      p->kernels = small_mix_supported(*p) ? 3 : 5;
    }
    if (variant == MHLA_VARIANT_FUSED) {
      p->off_flow = off;
      off = align_up(off + 3 * sizeof(unsigned int) * (size_t)p->BH);
      p->kernels = 2;
    }
    if (p->causal) {
      p->off_mcl = off;
      off = align_up(off + sizeof(float) * (size_t)p->M * p->M * p->mc_heads);
      p->kernels = 5;
    }
  }
  p->off_aux = off;
  p->ws_total = off;
  return MHLA_OK;
}

bool misaligned(const void* ptr, size_t a) { return ((uintptr_t)ptr) % a != 0; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  if (!a || !b || na == 0 || nb == 0) return false;
  const uintptr_t a0 = (uintptr_t)a, b0 = (uintptr_t)b;
  return a0 < b0 + nb && b0 < a0 + na;
}

void record_event(int idx, cudaStream_t s) {
  std::lock_guard<std::mutex> lock(g_events_mu);
  if (g_num_events == MHLA_NUM_PHASE_EVENTS) cudaEventRecord(g_events[idx], s);
}

void record_bwd_event(int idx, void* stream) {
  std::lock_guard<std::mutex> lock(g_events_mu);
  if (g_num_bwd_events == MHLA_NUM_BWD_PHASE_EVENTS)
    cudaEventRecord(g_bwd_events[idx], static_cast<cudaStream_t>(stream));
}

mhla_status run_plan(const Plan& plan, const void* q, const void* k, const void* v, const float* mc,
                     void* out, char* ws, cudaStream_t s) {
  Plan p = plan;
  mhla_status st = device_error_ptr(&p.err);
  if (st != MHLA_OK) return st;
  int e;
  if (p.variant == MHLA_VARIANT_MULTIPASS || p.variant == MHLA_VARIANT_FUSED) {
    const bool fused = p.variant == MHLA_VARIANT_FUSED;
    TcBuffers b;
    b.stack = ws + p.off_stack;
    b.stack_lo = p.f16_mix ? nullptr : reinterpret_cast<__nv_bfloat16*>(ws + p.off_stack_lo);
    b.mixed_hi = reinterpret_cast<__nv_bfloat16*>(ws + p.off_mixed);
    b.mixed_lo = reinterpret_cast<__nv_bfloat16*>(ws + p.off_mixed_lo);
    b.mc_f16 = reinterpret_cast<__half*>(ws + p.off_mc_f16);
    b.mc_scale = reinterpret_cast<float*>(ws + p.off_mc_scale);
    b.mc_hi = reinterpret_cast<__nv_bfloat16*>(ws + p.off_mc_hi);
    b.mc_lo = reinterpret_cast<__nv_bfloat16*>(ws + p.off_mc_lo);
    b.rowsum = reinterpret_cast<float*>(ws + p.off_rowsum);
    b.blkinfo = reinterpret_cast<float4*>(ws + p.off_blkinfo);
    b.rexp = p.f16_mix ? reinterpret_cast<int2*>(ws + p.off_rexp) : nullptr;
    b.mcx = p.f16_mix ? reinterpret_cast<__half*>(ws + p.off_mcx) : nullptr;
    b.sinfo = p.f16_mix ? reinterpret_cast<float4*>(ws + p.off_sinfo) : nullptr;
    b.mcw = p.f16_mix ? reinterpret_cast<uint32_t*>(ws + p.off_mcw) : nullptr;
    b.Qp = p.Qp;
    b.f16 = p.f16_mix != 0;
    b.slots = p.slots;
    b.flow = fused ? reinterpret_cast<unsigned int*>(ws + p.off_flow) : nullptr;
    record_event(0, s);
    if (fused) {
      if ((e = launch_tc_prep(p, mc, b, s)) != 0) return cuda_fail((cudaError_t)e);
      record_event(1, s);
      record_event(2, s);
      record_event(3, s);
      record_event(4, s);
      if ((e = launch_tc_fused(p, p.chunk, q, k, v, b, out, s)) != 0) return cuda_fail((cudaError_t)e);
      record_event(5, s);
      return MHLA_OK;
    }
    if (p.causal) {
      // records mixed with the strict lower triangle of Mc, every part in
      // high + low planes (the MALA precision settings of the forward kernels)
      Plan pr = p;
      pr.norm = MHLA_NORM_MALA;
      float* mcl = reinterpret_cast<float*>(ws + p.off_mcl);
      if ((e = launch_mc_strict_lower(p, mc, mcl, s)) != 0) return cuda_fail((cudaError_t)e);
      if ((e = launch_tc_prep(pr, mcl, b, s)) != 0) return cuda_fail((cudaError_t)e);
      record_event(1, s);
      if ((e = launch_tc_summary(pr, pr.chunk, k, v, b, s)) != 0) return cuda_fail((cudaError_t)e);
      record_event(2, s);
      record_event(3, s);
      if ((e = launch_tc_mix(pr, b, s)) != 0) return cuda_fail((cudaError_t)e);
      record_event(4, s);
      if ((e = launch_tc_causal(p, q, k, v, b.mixed_hi, b.mixed_lo, mc, out, s)) != 0)
        return cuda_fail((cudaError_t)e);
      record_event(5, s);
      return MHLA_OK;
    }
    // few blocks: the mixing runs on the CUDA cores (a tensor-core tile would
    // be almost all padding) and decodes the fp16 records' exponents itself
    const bool small = small_mix_supported(p);
    // the fp16 records with few blocks need nothing the prep kernel makes
    // (the small mixing reads Mc itself and writes the output scales)
    b.no_prep = b.f16 && small;
    if (!b.no_prep && (e = launch_tc_prep(p, mc, b, s)) != 0) return cuda_fail((cudaError_t)e);
    record_event(1, s);
    if ((e = launch_tc_summary(p, p.chunk, k, v, b, s)) != 0) return cuda_fail((cudaError_t)e);
    record_event(2, s);
    if (b.f16 && !small && (e = launch_tc_scale(p, b, s)) != 0) return cuda_fail((cudaError_t)e);
    record_event(3, s);
    if ((e = small ? launch_tc_mix_small(p, mc, b, s) : launch_tc_mix(p, b, s)) != 0) return cuda_fail((cudaError_t)e);
    record_event(4, s);
    if ((e = launch_tc_output(p, p.chunk, q, b, out, s)) != 0) return cuda_fail((cudaError_t)e);
    record_event(5, s);
    return MHLA_OK;
  }
  float* stack = reinterpret_cast<float*>(ws + p.off_stack);
  float* mixed = reinterpret_cast<float*>(ws + p.off_mixed);
  float* rowsum = reinterpret_cast<float*>(ws + p.off_rowsum);
  record_event(0, s);
  if (p.causal) {
    float* mcl = reinterpret_cast<float*>(ws + p.off_mcl);
    if ((e = launch_mc_strict_lower(p, mc, mcl, s)) != 0) return cuda_fail((cudaError_t)e);
    if ((e = launch_mc_rowsum(p, mcl, rowsum, s)) != 0) return cuda_fail((cudaError_t)e);
    record_event(1, s);
    if ((e = launch_simt_summary(p, k, v, stack, s)) != 0) return cuda_fail((cudaError_t)e);
    record_event(2, s);
    record_event(3, s);
    if ((e = launch_simt_mix(p, mcl, stack, mixed, s)) != 0) return cuda_fail((cudaError_t)e);
    record_event(4, s);
    if ((e = launch_simt_causal_output(p, q, k, v, mixed, rowsum, mc, out, s)) != 0)
      return cuda_fail((cudaError_t)e);
    record_event(5, s);
    return MHLA_OK;
  }
  if ((e = launch_mc_rowsum(p, mc, rowsum, s)) != 0) return cuda_fail((cudaError_t)e);
  record_event(1, s);
  if ((e = launch_simt_summary(p, k, v, stack, s)) != 0) return cuda_fail((cudaError_t)e);
  record_event(2, s);
  record_event(3, s);
  if ((e = launch_simt_mix(p, mc, stack, mixed, s)) != 0) return cuda_fail((cudaError_t)e);
  record_event(4, s);
  if ((e = launch_simt_output(p, q, mixed, rowsum, out, s)) != 0) return cuda_fail((cudaError_t)e);
  record_event(5, s);
  return MHLA_OK;
}

}  // namespace
}  // namespace mhla

namespace mhla {

// Head groups of mhla_forward_host: at least ~32 MB of each input tensor per
// group so the copies stay efficient, at most kMaxHostGroups groups.
constexpr int kMaxHostGroups = 8;
struct HostGroups {
  int n, per;  // groups, units per group (the last group may have fewer)
};

HostGroups host_groups(const Plan& plan) {
  const size_t io = (size_t)plan.BH * plan.N * plan.d * elem_bytes(plan.dtype);
  int n = (int)(io / (32ull << 20));
  if (n > kMaxHostGroups) n = kMaxHostGroups;
  if (n > plan.BH) n = plan.BH;
  if (n < 1) n = 1;
  HostGroups g;
  g.per = (plan.BH + n - 1) / n;
  // token-major tensors are contiguous per batch only, and per-head mixing
  // matrices index heads within a batch: whole batches per group
  if ((plan.layout == MHLA_LAYOUT_BNHD || plan.mc_heads > 1) && plan.H > 0)
    g.per = (g.per + plan.H - 1) / plan.H * plan.H;
  g.n = (plan.BH + g.per - 1) / g.per;
  return g;
}

// The parameters of a group of `units` (batch, head) pairs: one batch of
// `units` heads (the kernels see only the flattened unit index), or for
// token-major tensors units / H batches of H heads.
mhla_params group_params(const mhla_params* p, int units) {
  mhla_params g = *p;
  if ((p->layout == MHLA_LAYOUT_BNHD || p->mc_per_head) && p->heads > 0) {
    g.batch = units / p->heads;
  } else {
    g.batch = 1;
    g.heads = units;
  }
  return g;
}

// Largest workspace any group's plan needs.
mhla_status host_group_workspace(const mhla_params* p, const Plan& plan, size_t* ws) {
  const HostGroups hg = host_groups(plan);
  *ws = 0;
  const int sizes[2] = {hg.per, plan.BH - (hg.n - 1) * hg.per};
  for (int i = 0; i < 2; ++i) {
    Plan gp;
    mhla_params g = group_params(p, sizes[i]);
    mhla_status st = make_plan(&g, &gp, plan.BH);
    if (st != MHLA_OK) return st;
    if (gp.ws_total > *ws) *ws = gp.ws_total;
  }
  return MHLA_OK;
}

struct HostPipe {
  bool ready = false;
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t ev[3 * kMaxHostGroups + 1] = {};
};
HostPipe g_pipe[kMaxDevices];
std::mutex g_pipe_mu[kMaxDevices];

}  // namespace mhla

namespace mhla {

// Backward plan and its workspace layout.  The tensor-core backward (bf16,
// d = 64) recomputes the forward records with the forward kernels in split
// precision (bf16 high + low planes for every part) and keeps its gradient
// records as planes too; the float32 CUDA-core backward keeps float32
// records.
struct BwdLayout {
  bool tc;
  size_t stack, mixed, rowsum, dmixp, dnp, dstack;   // float32 records
  size_t stack_hi, stack_lo, mixed_hi, mixed_lo;     // planes (tensor cores)
  size_t dmixp_hi, dmixp_lo;
  size_t mc_f16, mc_hi, mc_lo, mc_scale, blkinfo, partial;
  size_t mct, mct_f16, mct_hi, mct_lo, mct_scale, mct_rowsum, mct_blkinfo;  // Mc transposed
  size_t dx_hi, dx_lo;                                                      // dS_b, dz_b, dv_b planes
  size_t mcl, tokbuf, xk, xv, diag;                                         // causal form (CUDA cores)
  size_t mc_partial;                                                        // dMc partial sums (CUDA cores)
  size_t total;
};

mhla_status make_bwd_plan(const mhla_params* prm, Plan* plan, BwdLayout* lay) {
  if (!prm) return MHLA_ERR_INVALID_ARG;
  mhla_params p = *prm;
  const bool tc_ok = p.dtype == MHLA_DTYPE_BF16 && p.head_dim == kTcHeadDim;
  if (p.causal == 1) {
    // the causal form's gradients run on the CUDA cores only
    if (p.variant != MHLA_VARIANT_AUTO && p.variant != MHLA_VARIANT_SIMT) return MHLA_ERR_UNSUPPORTED;
    p.variant = MHLA_VARIANT_SIMT;
  }
  if (p.variant == MHLA_VARIANT_AUTO) p.variant = tc_ok ? MHLA_VARIANT_MULTIPASS : MHLA_VARIANT_SIMT;
  if (p.variant == MHLA_VARIANT_FUSED) p.variant = MHLA_VARIANT_MULTIPASS;
  mhla_status st = make_plan(&p, plan);
  if (st != MHLA_OK) return st;
  memset(lay, 0, sizeof(*lay));
  lay->tc = plan->variant == MHLA_VARIANT_MULTIPASS;
  const size_t rows = (size_t)plan->BH * plan->M * plan->splits;
  const size_t mrows = (size_t)plan->BH * plan->M;
  const size_t R = (size_t)plan->R;
  size_t off = 0;
  auto take = [&](size_t& field, size_t bytes) {
    field = off;
    off = align_up(off + bytes);
  };
  const size_t mh = (size_t)plan->mc_heads;
  take(lay->rowsum, sizeof(float) * plan->M * mh);
  take(lay->dnp, sizeof(float) * rows);
  if (!lay->tc) {
    take(lay->stack, sizeof(float) * rows * R);
    take(lay->mixed, sizeof(float) * mrows * R);
    take(lay->dmixp, sizeof(float) * rows * R);
    take(lay->dstack, sizeof(float) * mrows * R);
    take(lay->mc_partial, bwd_mc_partial_bytes(*plan));
    if (plan->causal) {
      const size_t toks = (size_t)plan->BH * plan->N;
      take(lay->mcl, sizeof(float) * (size_t)plan->M * plan->M * mh);
      take(lay->tokbuf, sizeof(float) * toks * (plan->d + 4));
      take(lay->xk, sizeof(float) * toks * plan->d);
      take(lay->xv, sizeof(float) * toks * plan->d);
      take(lay->diag, sizeof(float) * mrows);
    }
  } else {
    take(lay->stack_hi, 2 * rows * R);
    take(lay->stack_lo, 2 * rows * R);
    take(lay->mixed_hi, 2 * mrows * R);
    take(lay->mixed_lo, 2 * mrows * R);
    take(lay->dmixp_hi, 2 * rows * R);
    take(lay->dmixp_lo, 2 * rows * R);
    const size_t mcq = 2 * (size_t)plan->M * mh * plan->Qp;
    take(lay->mc_f16, mcq);
    take(lay->mc_hi, mcq);
    take(lay->mc_lo, mcq);
    take(lay->mc_scale, sizeof(float) * plan->M * mh);
    take(lay->blkinfo, 16 * (size_t)plan->M * mh);
    take(lay->partial, tc_bwd_mc_partial_bytes(*plan));
    take(lay->mct, sizeof(float) * (size_t)plan->M * plan->M * mh);
    take(lay->mct_f16, mcq);
    take(lay->mct_hi, mcq);
    take(lay->mct_lo, mcq);
    take(lay->mct_scale, sizeof(float) * plan->M * mh);
    take(lay->mct_rowsum, sizeof(float) * plan->M * mh);
    take(lay->mct_blkinfo, 16 * (size_t)plan->M * mh);
    take(lay->dx_hi, 2 * mrows * R);
    take(lay->dx_lo, 2 * mrows * R);
  }
  lay->total = plan->BH == 0 ? 0 : off;
  return MHLA_OK;
}

int run_backward(const Plan& plan, const BwdLayout& lay, const void* q, const void* k, const void* v,
                 const float* mc, const void* dout, void* dq, void* dk, void* dv, float* dmc, char* ws,
                 cudaStream_t s) {
  Plan p = plan;
  if (device_error_ptr(&p.err) != MHLA_OK) return (int)cudaErrorUnknown;
  auto F = [&](size_t off) { return reinterpret_cast<float*>(ws + off); };
  auto H = [&](size_t off) { return reinterpret_cast<__nv_bfloat16*>(ws + off); };
  BwdBuffers w;
  w.mc = mc;
  w.stack = F(lay.stack);
  w.mixed = F(lay.mixed);
  w.rowsum = F(lay.rowsum);
  w.dmixp = F(lay.dmixp);
  w.dnp = F(lay.dnp);
  w.dstack = F(lay.dstack);
  w.dmc = dmc;
  w.diag = nullptr;
  w.xk = nullptr;
  w.xv = nullptr;
  w.mc_partial = lay.tc ? nullptr : F(lay.mc_partial);
  int e;
  record_bwd_event(0, s);
  if (lay.tc) {
    // forward records in split precision: the forward kernels with the MALA
    // precision settings (bf16 high + low planes for every part)
    Plan pr = p;
    pr.norm = MHLA_NORM_MALA;
    pr.f16_mix = 0;
    TcBuffers b;
    b.stack = H(lay.stack_hi);
    b.stack_lo = H(lay.stack_lo);
    b.mixed_hi = H(lay.mixed_hi);
    b.mixed_lo = H(lay.mixed_lo);
    b.mc_f16 = reinterpret_cast<__half*>(ws + lay.mc_f16);
    b.mc_scale = F(lay.mc_scale);
    b.mc_hi = H(lay.mc_hi);
    b.mc_lo = H(lay.mc_lo);
    b.rowsum = F(lay.rowsum);
    b.blkinfo = reinterpret_cast<float4*>(ws + lay.blkinfo);
    b.rexp = nullptr;
    b.mcx = nullptr;
    b.sinfo = nullptr;
    b.mcw = nullptr;
    b.Qp = p.Qp;
    b.f16 = false;
    b.slots = p.BH;
    b.flow = nullptr;
    if ((e = launch_tc_prep(pr, mc, b, s)) != 0) return e;
    if ((e = launch_tc_summary(pr, pr.chunk, k, v, b, s)) != 0) return e;
    if ((e = launch_tc_mix(pr, b, s)) != 0) return e;
    record_bwd_event(1, s);
    if ((e = launch_tc_bwd_output(p, q, dout, b.mixed_hi, b.mixed_lo, b.blkinfo, dq, H(lay.dmixp_hi),
                                  H(lay.dmixp_lo), w.dnp, s)) != 0)
      return e;
    record_bwd_event(2, s);
    // gradient mixing dX_b = sum_q Mc[i(q), b] dX~_q: the forward mixing
    // kernel with Mc transposed
    TcBuffers bt = b;
    bt.stack = H(lay.dmixp_hi);
    bt.stack_lo = H(lay.dmixp_lo);
    bt.mixed_hi = H(lay.dx_hi);
    bt.mixed_lo = H(lay.dx_lo);
    bt.mc_f16 = reinterpret_cast<__half*>(ws + lay.mct_f16);
    bt.mc_scale = F(lay.mct_scale);
    bt.mc_hi = H(lay.mct_hi);
    bt.mc_lo = H(lay.mct_lo);
    bt.rowsum = F(lay.mct_rowsum);
    bt.blkinfo = reinterpret_cast<float4*>(ws + lay.mct_blkinfo);
    if ((e = launch_transpose_mc(mc, F(lay.mct), p.M, p.mc_heads, s)) != 0) return e;
    if ((e = launch_tc_prep(pr, F(lay.mct), bt, s)) != 0) return e;
    if ((e = launch_tc_mix(pr, bt, s)) != 0) return e;
    record_bwd_event(3, s);
    if ((e = launch_tc_bwd_mc(p, H(lay.dmixp_hi), H(lay.dmixp_lo), H(lay.stack_hi), b.stack_lo, w.dnp, F(lay.partial), dmc,
                              s)) != 0)
      return e;
    record_bwd_event(4, s);
    if ((e = launch_tc_bwd_summary(p, k, v, H(lay.dx_hi), H(lay.dx_lo), dk, dv, s)) != 0) return e;
    record_bwd_event(5, s);
    return 0;
  }
  if (p.causal) {
    // earlier blocks through Mc's strict lower triangle, the own block token
    // by token through its diagonal
    float* mcl = F(lay.mcl);
    if ((e = launch_mc_strict_lower(p, mc, mcl, s)) != 0) return e;
    if ((e = launch_mc_rowsum(p, mcl, w.rowsum, s)) != 0) return e;
    if ((e = launch_simt_summary(p, k, v, w.stack, s)) != 0) return e;
    if ((e = launch_simt_mix(p, mcl, w.stack, w.mixed, s)) != 0) return e;
    record_bwd_event(1, s);
    CausalBwdBuffers c;
    c.mc = mc;
    c.mixed = w.mixed;
    c.rowsum_lower = w.rowsum;
    c.dmixp = w.dmixp;
    c.dnp = w.dnp;
    c.diag = F(lay.diag);
    c.tokbuf = F(lay.tokbuf);
    c.xk = F(lay.xk);
    c.xv = F(lay.xv);
    if ((e = launch_bwd_causal_block(p, c, q, k, v, dout, dq, s)) != 0) return e;
    record_bwd_event(2, s);
    w.mc = mcl;
    w.diag = c.diag;
    w.xk = c.xk;
    w.xv = c.xv;
    if ((e = launch_bwd_mix(p, w, s)) != 0) return e;
    record_bwd_event(3, s);
    if ((e = launch_bwd_mc(p, w, s)) != 0) return e;
    record_bwd_event(4, s);
    if ((e = launch_bwd_summary(p, w, k, v, dk, dv, s)) != 0) return e;
    record_bwd_event(5, s);
    return 0;
  }
  if ((e = launch_mc_rowsum(p, mc, w.rowsum, s)) != 0) return e;
  if ((e = launch_simt_summary(p, k, v, w.stack, s)) != 0) return e;
  if ((e = launch_simt_mix(p, mc, w.stack, w.mixed, s)) != 0) return e;
  record_bwd_event(1, s);
  if ((e = launch_bwd_output(p, w, q, dout, dq, s)) != 0) return e;
  record_bwd_event(2, s);
  if ((e = launch_bwd_mix(p, w, s)) != 0) return e;
  record_bwd_event(3, s);
  if ((e = launch_bwd_mc(p, w, s)) != 0) return e;
  record_bwd_event(4, s);
  if ((e = launch_bwd_summary(p, w, k, v, dk, dv, s)) != 0) return e;
  record_bwd_event(5, s);
  return 0;
}

}  // namespace mhla

using mhla::Plan;

extern "C" {

mhla_status mhla_backward_workspace_bytes(const mhla_params* p, size_t* bytes) {
  if (!bytes) return MHLA_ERR_INVALID_ARG;
  Plan plan;
  mhla::BwdLayout lay;
  mhla_status st = mhla::make_bwd_plan(p, &plan, &lay);
  if (st != MHLA_OK) return st;
  *bytes = lay.total;
  return MHLA_OK;
}

mhla_status mhla_backward(const void* q, const void* k, const void* v, const float* mc, const void* dout,
                          const mhla_params* p, void* dq, void* dk, void* dv, float* dmc, void* workspace,
                          size_t workspace_bytes, void* stream) {
  Plan plan;
  mhla::BwdLayout lay;
  mhla_status st = mhla::make_bwd_plan(p, &plan, &lay);
  if (st != MHLA_OK) return st;
  if (plan.BH == 0) return MHLA_OK;
  if (!q || !k || !v || !mc || !dout || !dq || !dk || !dv || !dmc) return MHLA_ERR_INVALID_ARG;
  const void* io_in[4] = {q, k, v, dout};
  void* io_out[3] = {dq, dk, dv};
  for (const void* x : io_in)
    if (mhla::misaligned(x, 16)) return MHLA_ERR_INVALID_ARG;
  for (const void* x : io_out)
    if (mhla::misaligned(x, 16)) return MHLA_ERR_INVALID_ARG;
  if (mhla::misaligned(mc, 4) || mhla::misaligned(dmc, 4)) return MHLA_ERR_INVALID_ARG;
  const size_t io = (size_t)plan.BH * plan.N * plan.d * mhla::elem_bytes(plan.dtype);
  const size_t mcb = sizeof(float) * (size_t)plan.M * plan.M * plan.mc_heads;
  for (int a = 0; a < 3; ++a) {
    for (const void* x : io_in)
      if (mhla::overlaps(io_out[a], io, x, io)) return MHLA_ERR_INVALID_ARG;
    if (mhla::overlaps(io_out[a], io, mc, mcb) || mhla::overlaps(io_out[a], io, dmc, mcb)) return MHLA_ERR_INVALID_ARG;
    for (int b = a + 1; b < 3; ++b)
      if (mhla::overlaps(io_out[a], io, io_out[b], io)) return MHLA_ERR_INVALID_ARG;
  }
  for (const void* x : io_in)
    if (mhla::overlaps(dmc, mcb, x, io)) return MHLA_ERR_INVALID_ARG;
  if (mhla::overlaps(dmc, mcb, mc, mcb)) return MHLA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  bool owned = false;
  if (!workspace) {
    if (workspace_bytes != 0) return MHLA_ERR_INVALID_ARG;
    cudaError_t e = cudaMallocAsync(&workspace, lay.total, s);
    if (e != cudaSuccess) return mhla::cuda_fail(e);
    owned = true;
  } else {
    if (workspace_bytes < lay.total) return MHLA_ERR_WORKSPACE;
    if (mhla::misaligned(workspace, 256)) return MHLA_ERR_INVALID_ARG;
  }
  char* ws = static_cast<char*>(workspace);
  const int e = mhla::run_backward(plan, lay, q, k, v, mc, dout, dq, dk, dv, dmc, ws, s);
  if (e != 0) st = mhla::cuda_fail((cudaError_t)e);
  if (owned) {
    cudaError_t fe = cudaFreeAsync(workspace, s);
    if (st == MHLA_OK && fe != cudaSuccess) st = mhla::cuda_fail(fe);
  }
  return st;
}


mhla_status mhla_plan(const mhla_params* p, mhla_plan_info* info) {
  Plan plan;
  mhla_status st = mhla::make_plan(p, &plan);
  if (st != MHLA_OK) return st;
  if (info) {
    info->n_tokens = plan.N;
    info->n_blocks = plan.M;
    info->block_tokens = plan.nb;
    info->variant = plan.variant;
    info->kernels_per_call = plan.kernels;
    info->summary_splits = plan.splits;
    info->workspace_bytes = plan.ws_total;
  }
  return MHLA_OK;
}

mhla_status mhla_workspace_bytes(const mhla_params* p, size_t* bytes) {
  if (!bytes) return MHLA_ERR_INVALID_ARG;
  Plan plan;
  mhla_status st = mhla::make_plan(p, &plan);
  if (st != MHLA_OK) return st;
  *bytes = plan.ws_total;
  return MHLA_OK;
}

mhla_status mhla_forward(const void* q, const void* k, const void* v, const float* mc,
                         const mhla_params* p, void* out, void* workspace, size_t workspace_bytes,
                         void* stream) {
  Plan plan;
  mhla_status st = mhla::make_plan(p, &plan);
  if (st != MHLA_OK) return st;
  if (plan.BH == 0) return MHLA_OK;
  if (!q || !k || !v || !mc || !out) return MHLA_ERR_INVALID_ARG;
  if (mhla::misaligned(q, 16) || mhla::misaligned(k, 16) || mhla::misaligned(v, 16) ||
      mhla::misaligned(out, 16) || mhla::misaligned(mc, 4))
    return MHLA_ERR_INVALID_ARG;
  const size_t io_bytes = (size_t)plan.BH * plan.N * plan.d * mhla::elem_bytes(plan.dtype);
  const size_t mc_bytes = sizeof(float) * (size_t)plan.M * plan.M * plan.mc_heads;
  if (mhla::overlaps(out, io_bytes, q, io_bytes) || mhla::overlaps(out, io_bytes, k, io_bytes) ||
      mhla::overlaps(out, io_bytes, v, io_bytes) || mhla::overlaps(out, io_bytes, mc, mc_bytes))
    return MHLA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  bool owned = false;
  if (!workspace) {
    if (workspace_bytes != 0) return MHLA_ERR_INVALID_ARG;
    cudaError_t e = cudaMallocAsync(&workspace, plan.ws_total, s);
    if (e != cudaSuccess) return mhla::cuda_fail(e);
    owned = true;
  } else {
    if (workspace_bytes < plan.ws_total) return MHLA_ERR_WORKSPACE;
    if (mhla::misaligned(workspace, 256)) return MHLA_ERR_INVALID_ARG;
    if (mhla::overlaps(out, io_bytes, workspace, plan.ws_total)) return MHLA_ERR_INVALID_ARG;
  }
  st = mhla::run_plan(plan, q, k, v, mc, out, static_cast<char*>(workspace), s);
  if (owned) {
    cudaError_t e = cudaFreeAsync(workspace, s);
    if (st == MHLA_OK && e != cudaSuccess) st = mhla::cuda_fail(e);
  }
  return st;
}

mhla_status mhla_host_buffer_bytes(const mhla_params* p, size_t* bytes) {
  if (!bytes) return MHLA_ERR_INVALID_ARG;
  Plan plan;
  mhla_status st = mhla::make_plan(p, &plan);
  if (st != MHLA_OK) return st;
  if (plan.BH == 0) {
    *bytes = 0;
    return MHLA_OK;
  }
  size_t ws = 0;
  st = mhla::host_group_workspace(p, plan, &ws);
  if (st != MHLA_OK) return st;
  const size_t io = mhla::align_up((size_t)plan.BH * plan.N * plan.d * mhla::elem_bytes(plan.dtype));
  const size_t mcb = mhla::align_up(sizeof(float) * (size_t)plan.M * plan.M * plan.mc_heads);
  *bytes = 4 * io + mcb + ws;
  return MHLA_OK;
}

mhla_status mhla_forward_host(const void* q, const void* k, const void* v, const float* mc,
                              const mhla_params* p, void* out, void* dev_buffer,
                              size_t dev_buffer_bytes, void* stream) {
  Plan plan;
  mhla_status st = mhla::make_plan(p, &plan);
  if (st != MHLA_OK) return st;
  if (plan.BH == 0) return MHLA_OK;
  if (!q || !k || !v || !mc || !out || !dev_buffer) return MHLA_ERR_INVALID_ARG;
  if (mhla::misaligned(dev_buffer, 256)) return MHLA_ERR_INVALID_ARG;
  size_t need = 0;
  if ((st = mhla_host_buffer_bytes(p, &need)) != MHLA_OK) return st;
  if (dev_buffer_bytes < need) return MHLA_ERR_WORKSPACE;
  const size_t unit_bytes = (size_t)plan.N * plan.d * mhla::elem_bytes(plan.dtype);
  const size_t io_raw = (size_t)plan.BH * unit_bytes;
  const size_t io = mhla::align_up(io_raw);
  const size_t mc_raw = sizeof(float) * (size_t)plan.M * plan.M * plan.mc_heads;
  const size_t mcb = mhla::align_up(mc_raw);
  char* base = static_cast<char*>(dev_buffer);
  char* dq = base;
  char* dk = dq + io;
  char* dv = dk + io;
  char* dmc = dv + io;
  char* dout = dmc + mcb;
  char* ws = dout + io;
  const mhla::HostGroups hg = mhla::host_groups(plan);
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  // One pipeline per device: group g's copies in run on `in` while group
  // g-1's kernels run on the caller's stream and group g-2's result goes
  // back on `out` (the two copy directions use separate engines).
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return mhla::cuda_fail(e);
  if (dev < 0 || dev >= mhla::kMaxDevices) return MHLA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(mhla::g_pipe_mu[dev]);
  mhla::HostPipe& hp = mhla::g_pipe[dev];
  if (!hp.ready) {
    if ((e = cudaStreamCreateWithFlags(&hp.in, cudaStreamNonBlocking)) != cudaSuccess) return mhla::cuda_fail(e);
    if ((e = cudaStreamCreateWithFlags(&hp.out, cudaStreamNonBlocking)) != cudaSuccess) return mhla::cuda_fail(e);
    for (int i = 0; i < 3 * mhla::kMaxHostGroups + 1; ++i)
      if ((e = cudaEventCreateWithFlags(&hp.ev[i], cudaEventDisableTiming)) != cudaSuccess) return mhla::cuda_fail(e);
    hp.ready = true;
  }
  cudaEvent_t ev_start = hp.ev[3 * mhla::kMaxHostGroups];
  auto fail = [&](cudaError_t err) {
    cudaStreamSynchronize(hp.in);
    cudaStreamSynchronize(s);
    cudaStreamSynchronize(hp.out);
    return mhla::cuda_fail(err);
  };
  // the copies start after the caller's earlier work on its stream
  if ((e = cudaEventRecord(ev_start, s)) != cudaSuccess) return fail(e);
  if ((e = cudaStreamWaitEvent(hp.in, ev_start, 0)) != cudaSuccess) return fail(e);
  if ((e = cudaStreamWaitEvent(hp.out, ev_start, 0)) != cudaSuccess) return fail(e);
  if ((e = cudaMemcpyAsync(dmc, mc, mc_raw, cudaMemcpyHostToDevice, hp.in)) != cudaSuccess) return fail(e);
  for (int g = 0; g < hg.n; ++g) {
    const int u0 = g * hg.per;
    const int nu = plan.BH - u0 < hg.per ? plan.BH - u0 : hg.per;
    const size_t off = (size_t)u0 * unit_bytes, len = (size_t)nu * unit_bytes;
    cudaEvent_t ev_in = hp.ev[3 * g], ev_run = hp.ev[3 * g + 1], ev_out = hp.ev[3 * g + 2];
    // K and V first: the summaries need them before the output step needs Q
    if ((e = cudaMemcpyAsync(dk + off, static_cast<const char*>(k) + off, len, cudaMemcpyHostToDevice, hp.in)) != cudaSuccess)
      return fail(e);
    if ((e = cudaMemcpyAsync(dv + off, static_cast<const char*>(v) + off, len, cudaMemcpyHostToDevice, hp.in)) != cudaSuccess)
      return fail(e);
    if ((e = cudaMemcpyAsync(dq + off, static_cast<const char*>(q) + off, len, cudaMemcpyHostToDevice, hp.in)) != cudaSuccess)
      return fail(e);
    if ((e = cudaEventRecord(ev_in, hp.in)) != cudaSuccess) return fail(e);
    if ((e = cudaStreamWaitEvent(s, ev_in, 0)) != cudaSuccess) return fail(e);
    Plan gp;
    mhla_params gprm = mhla::group_params(p, nu);
    if ((st = mhla::make_plan(&gprm, &gp, plan.BH)) != MHLA_OK) {
      fail(cudaSuccess);
      return st;
    }
    st = mhla::run_plan(gp, dq + off, dk + off, dv + off, reinterpret_cast<const float*>(dmc), dout + off, ws, s);
    if (st != MHLA_OK) {
      fail(cudaSuccess);
      return st;
    }
    if ((e = cudaEventRecord(ev_run, s)) != cudaSuccess) return fail(e);
    if ((e = cudaStreamWaitEvent(hp.out, ev_run, 0)) != cudaSuccess) return fail(e);
    if ((e = cudaMemcpyAsync(static_cast<char*>(out) + off, dout + off, len, cudaMemcpyDeviceToHost, hp.out)) != cudaSuccess)
      return fail(e);
    if ((e = cudaEventRecord(ev_out, hp.out)) != cudaSuccess) return fail(e);
  }
  // the caller's stream ends after the last copy back
  if ((e = cudaStreamWaitEvent(s, hp.ev[3 * (hg.n - 1) + 2], 0)) != cudaSuccess) return fail(e);
  if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return mhla::cuda_fail(e);
  return MHLA_OK;
}

mhla_status mhla_device_status(int* code, int* detail) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return mhla::cuda_fail(e);
  unsigned int h[2] = {0, 0};
  e = cudaMemcpyFromSymbol(h, mhla::g_device_error, sizeof(h));
  if (e != cudaSuccess) return mhla::cuda_fail(e);
  const unsigned int zero[2] = {0, 0};
  e = cudaMemcpyToSymbol(mhla::g_device_error, zero, sizeof(zero));
  if (e != cudaSuccess) return mhla::cuda_fail(e);
  if (code) *code = (int)h[0];
  if (detail) *detail = (int)h[1];
  return MHLA_OK;
}

mhla_status mhla_set_debug(int option, long long value) {
  switch (option) {
    case MHLA_DEBUG_FLOW_WAIT_NS:
      mhla::g_debug_flow_wait_ns.store(value > 0 ? (unsigned long long)value : 0ull);
      return MHLA_OK;
    case MHLA_DEBUG_FLOW_STALL:
      mhla::g_debug_flow_stall.store(value != 0 ? 1u : 0u);
      return MHLA_OK;
    default:
      return MHLA_ERR_INVALID_ARG;
  }
}

mhla_status mhla_set_phase_events(void* const* events, int n) {
  if (n != 0 && n != MHLA_NUM_PHASE_EVENTS) return MHLA_ERR_INVALID_ARG;
  if (n && !events) return MHLA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(mhla::g_events_mu);
  for (int i = 0; i < n; ++i) {
    if (!events[i]) return MHLA_ERR_INVALID_ARG;
  }
  for (int i = 0; i < n; ++i) mhla::g_events[i] = static_cast<cudaEvent_t>(events[i]);
  mhla::g_num_events = n;
  return MHLA_OK;
}

mhla_status mhla_set_backward_phase_events(void* const* events, int n) {
  if (n != 0 && n != MHLA_NUM_BWD_PHASE_EVENTS) return MHLA_ERR_INVALID_ARG;
  if (n && !events) return MHLA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(mhla::g_events_mu);
  for (int i = 0; i < n; ++i) {
    if (!events[i]) return MHLA_ERR_INVALID_ARG;
  }
  for (int i = 0; i < n; ++i) mhla::g_bwd_events[i] = static_cast<cudaEvent_t>(events[i]);
  mhla::g_num_bwd_events = n;
  return MHLA_OK;
}

const char* mhla_status_string(mhla_status s) {
  switch (s) {
    case MHLA_OK: return "MHLA_OK";
    case MHLA_ERR_INVALID_ARG: return "MHLA_ERR_INVALID_ARG: invalid pointer, shape, option or alignment";
    case MHLA_ERR_UNSUPPORTED: return "MHLA_ERR_UNSUPPORTED: valid request the library does not support";
    case MHLA_ERR_WORKSPACE: return "MHLA_ERR_WORKSPACE: workspace missing or too small";
    case MHLA_ERR_CUDA: return "MHLA_ERR_CUDA: a CUDA runtime call failed";
    case MHLA_ERR_DEVICE_TIMEOUT: return "MHLA_ERR_DEVICE_TIMEOUT: a kernel's bounded wait expired";
    case MHLA_ERR_OVERFLOW: return "MHLA_ERR_OVERFLOW: an intermediate left the fp16 range";
  }
  return "MHLA: unknown status";
}

const char* mhla_last_error_string(void) { return mhla::g_last_error.c_str(); }

int mhla_abi_version(void) { return MHLA_ABI_VERSION; }

}  // extern "C"
