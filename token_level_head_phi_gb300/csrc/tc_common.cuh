// Blackwell (sm_103a) building blocks written as inline PTX: mbarriers with
// bounded waits, TMA tensor copies, bulk copies, tcgen05 MMA / TMEM access
// and the shared-memory matrix descriptors the tensor cores read.
//
// Conventions used by every tensor-core kernel of this library:
//  * Operand tiles live in shared memory in the 128-byte-swizzle layout that
//    TMA writes for a box whose inner extent is 64 bf16 (128 bytes): row r of
//    a tile occupies bytes [r*128, r*128+128) and its 16-byte chunk j sits at
//    chunk position j ^ (r % 8).  Tile bases are 1024-byte aligned.
//  * K-major operand (contraction index contiguous): rows are M (or N)
//    indices, 64 K-elements per row; 8-row groups are 1024 bytes apart (SBO);
//    one MMA step of K = 16 advances the start address by 32 bytes.
//  * MN-major operand (M or N index contiguous): rows are K indices, each row
//    holds 64 M/N-elements (one "atom" column); 8-row K groups are 1024 bytes
//    apart (SBO) and further 64-wide atom columns sit LBO bytes apart; one
//    MMA step of K = 16 advances the start address by 16 rows = 2048 bytes.
//  * Accumulators are float32 in TMEM; for M = 128 row i of D is TMEM lane i.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "mhla.h"

namespace mhla {
namespace tc {

constexpr unsigned int kErrTimeout = MHLA_ERR_DEVICE_TIMEOUT;
// Upper bound on any single wait on the device.
constexpr unsigned long long kWaitLimitNs = 1000ull * 1000ull * 1000ull;
// Longest a waiting thread stays suspended before it re-checks the abort
// flag and the time limit.
constexpr uint32_t kSleepHintNs = 200000u;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------- mbarriers

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar);

// One arrival for the whole (converged) warp, after every lane's earlier
// shared-memory writes and fences: barriers that wait for warps count
// warps, not threads.
__device__ __forceinline__ void mbar_arrive_warp(uint32_t bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// try_wait that lets the hardware suspend the thread for up to `hint_ns`
// nanoseconds (it resumes as soon as the phase completes), so waiting roles
// do not spin on the issue slots the working roles need.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Records a status in the device error word (first writer wins).
__device__ __forceinline__ void report_error(unsigned int* err, unsigned int code, unsigned int where) {
  if (err && atomicCAS(err, 0u, code) == 0u) atomicExch(err + 1, where);
}

__device__ __forceinline__ void report_timeout(unsigned int* err, unsigned int where) {
  report_error(err, kErrTimeout, where);
}

// Waits until the phase of `bar` with parity `parity` has completed.  Gives
// up after kWaitLimitNs, records the timeout (with `where`), raises the CTA's
// abort flag and returns false.  Also returns false as soon as another role
// of the CTA has raised the abort flag.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, unsigned int* err, unsigned int where,
                                          volatile int* abort_flag = nullptr) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity, kSleepHintNs)) return true;
    if (abort_flag && *abort_flag) return false;
    if (globaltimer() - t0 > kWaitLimitNs) {
      report_timeout(err, where);
      if (abort_flag) *abort_flag = 1;
      return false;
    }
  }
}

// Before a producer's CTA exits (normally or after an abort): waits, bounded
// and regardless of the abort flag, for the last loads it issued (the i-th
// load went to stage i % stages with parity (i / stages) & 1; the stage's
// full barrier sits at full0 + 8 * stage), so that no copy into shared
// memory is still in flight when the CTA's memory is released.
__device__ __forceinline__ void drain_loads(uint32_t full0, int stages, long long issued, unsigned int* err,
                                            unsigned int where) {
  const long long first = issued > stages ? issued - stages : 0;
  for (long long i = first; i < issued; ++i) {
    const uint32_t bar = full0 + 8u * (uint32_t)(i % stages);
    const uint32_t parity = (uint32_t)((i / stages) & 1);
    if (mbar_try_wait(bar, parity)) continue;
    const unsigned long long t0 = globaltimer();
    while (!mbar_try_wait_sleep(bar, parity, 20000u)) {
      if (globaltimer() - t0 > kWaitLimitNs) {
        report_timeout(err, where);
        return;
      }
    }
  }
}

// ------------------------------------------- programmatic dependent launch

// The multi-pass kernels are launched with programmatic stream
// serialization: a kernel may start while its predecessor in the stream
// drains, does its own set-up (barriers, TMEM, tensor-map prefetch) and its
// independent loads, and calls pdl_wait() before it reads anything the
// predecessor writes.  Both are no-ops for a normal launch.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ------------------------------------------------ cross-CTA work flow

// Where a CTA sits in a (possibly fused) launch and how it hands work to
// other CTAs.  A standalone launch uses cta = blockIdx.x, ncta = gridDim.x,
// one intermediate slot per head and no counters.  The fused launch gives
// each CTA group its own range, keeps the intermediates of `ring` heads in
// reused slots, and orders producer and consumer groups through per-head
// counters in global memory.
struct FlowCtl {
  int cta, ncta;              // index of this CTA in its group, group size
  int ring;                   // slots of the stack / mixed rings (0: one slot per head)
  unsigned int* s_done;       // per head: summary units whose stack rows are written
  unsigned int* x_done;       // per head: mixing epilogue groups whose rows are written
  unsigned int* o_done;       // per head: output units that have read their S~_i
  unsigned int need_s, need_x, need_o;
  unsigned long long wait_ns;  // limit of each counter wait (0: kWaitLimitNs)
  unsigned int stall;          // testing: extra count the output's waits demand (never reached)
};

__device__ __forceinline__ int flow_slot(const FlowCtl& f, int u) { return f.ring ? u % f.ring : u; }

// Waits (bounded) until *ctr >= need, then orders the caller's later TMA
// reads after the writes the counter publishes.
__device__ __forceinline__ bool flow_wait(const unsigned int* ctr, unsigned int need, unsigned int* err,
                                          unsigned int where, volatile int* abort_flag,
                                          unsigned long long limit_ns) {
  if (limit_ns == 0) limit_ns = kWaitLimitNs;
  const unsigned long long t0 = globaltimer();
  unsigned int ns = 64;
  for (;;) {
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
    if (v >= need) {
      asm volatile("fence.proxy.async.global;" ::: "memory");
      return true;
    }
    if (abort_flag && *abort_flag) return false;
    if (globaltimer() - t0 > limit_ns) {
      report_timeout(err, where);
      if (abort_flag) *abort_flag = 1;
      return false;
    }
    __nanosleep(ns);
    if (ns < 2048) ns <<= 1;
  }
}

// Publishes the caller's completed TMA stores (waited for with bulk_wait)
// and counts n more finished pieces of work.
__device__ __forceinline__ void flow_signal(unsigned int* ctr, unsigned int n) {
  asm volatile("fence.proxy.async.global;" ::: "memory");
  __threadfence();
  atomicAdd(ctr, n);
}

// Whether unit w is the last one of its head that this CTA takes (units are
// numbered head-major, per_head to a head, and a CTA takes every ncta-th).
// Counters are bumped once per head and CTA, at that unit, and waits are
// done once per head: a global-memory round trip per unit would throttle
// the producers.
__device__ __forceinline__ bool flow_head_ends(const FlowCtl& f, int w, int units, int per_head) {
  const int wn = w + f.ncta;
  return wn >= units || wn / per_head != w / per_head;
}

// Named barrier over `nthreads` threads (a multiple of 32) with id 1..15.
__device__ __forceinline__ void named_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("barrier.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Named barrier that also ANDs `pred` over the participating threads, so a
// group of threads leaves a loop together when any of them gave up a wait.
__device__ __forceinline__ bool named_all(uint32_t id, uint32_t nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "barrier.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

// Makes this thread's generic-proxy shared-memory writes visible to the
// async proxy (TMA stores, tensor-core operand reads).
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------- TMA

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1,
                                            int c2, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1,
                                            int c2, int c3, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5, %6}], [%2], %7;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_load_5d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1,
                                            int c2, int c3, int c4, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5, %6, %7}], [%2], %8;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_store_5d(const CUtensorMap* map, uint32_t src, int c0, int c1, int c2, int c3,
                                             int c4) {
  asm volatile("cp.async.bulk.tensor.5d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5, %6}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
               : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}

__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int c0, int c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(c0), "r"(c1)
               : "memory");
}

// Plain (untiled) bulk copy global -> shared completing on an mbarrier;
// 16-byte aligned addresses, size % 16 == 0.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

// Plain (untiled) bulk copy shared -> global; 16-byte aligned, size % 16 == 0.
__device__ __forceinline__ void bulk_store(void* gdst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(src), "r"(bytes)
               : "memory");
}

// 16-byte asynchronous copy global -> shared (L2 only), and an arrival on
// `bar` once this thread's earlier copies have landed (the barrier's
// expected count is raised by one when the arrival is registered, so it
// needs no extra count at init).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

template <int N>
__device__ __forceinline__ void bulk_wait() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// ------------------------------------------------------------ tcgen05

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem] with kind::f16: bf16 or fp16 inputs (as the
// instruction descriptor says; A and B of one MMA share the type), float32
// accumulate.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Same with the A operand in tensor memory: a_tmem addresses its first
// column (lane = row of A, each 32-bit column two consecutive K entries).
__device__ __forceinline__ void umma_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives once on `bar` when every MMA this thread issued before has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 32 consecutive 32-bit columns into this warp's 32 TMEM lanes (one lane per thread).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// 32 consecutive float32 columns of this warp's 32 TMEM lanes (one lane per thread).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 2 consecutive float32 columns of this warp's 32 TMEM lanes.
__device__ __forceinline__ void tmem_ld2(uint32_t taddr, float& a, float& b) {
  uint32_t r0, r1;
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x2.b32 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(taddr));
  a = __uint_as_float(r0);
  b = __uint_as_float(r1);
}

// 16 consecutive float32 columns of this warp's 32 TMEM lanes.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// phi = ELU(x) + 1 written as max(x, 0) + exp(min(x, 0)): x + 1 above zero,
// exp(x) at and below it, with no branch or select.
__device__ __forceinline__ float phi_elu1_fast(float x) {
  return fmaxf(x, 0.f) + __expf(fminf(x, 0.f));
}

__device__ __forceinline__ float phi_map(float x, int fmap) {
  if (fmap == MHLA_FEATURE_IDENTITY) return x;
  if (fmap == MHLA_FEATURE_RELU) return fmaxf(x, 0.f);
  if (fmap == MHLA_FEATURE_EXP) return __expf(x);
  return phi_elu1_fast(x);
}

// phi' from the bf16 high and low parts of phi(x) (x itself is not kept):
// ELU+1 gives phi > 1 exactly where x > 0 and phi' = min(phi, 1); ReLU gives
// phi > 0 exactly where x > 0; exp gives phi' = phi.
__device__ __forceinline__ float phi_deriv_from_phi(float hi, float lo, int fmap) {
  if (fmap == MHLA_FEATURE_ELU1) return fminf(hi + lo, 1.f);
  if (fmap == MHLA_FEATURE_RELU) return hi > 0.f ? 1.f : 0.f;
  if (fmap == MHLA_FEATURE_EXP) return hi + lo;
  return 1.f;
}

// phi = ELU+1 of two bf16 values, returned as bf16x2 rounded to nearest:
// max(x, 0) and min(x, 0) are exact in bf16x2 arithmetic, exp runs in
// float32 on the min part and is rounded once, and the final bf16x2 add is
// exact because one of its two terms is zero (x <= 0) or exp(0) = 1 (x > 0,
// where x + 1 is rounded once) -- the same result as rounding the float32
// value max(x, 0) + exp(min(x, 0)).
__device__ __forceinline__ uint32_t phi2_elu1_bf16(uint32_t w) {
  const __nv_bfloat162 x = *reinterpret_cast<const __nv_bfloat162*>(&w);
  const __nv_bfloat162 zero = __float2bfloat162_rn(0.f);
  const __nv_bfloat162 mx = __hmax2(x, zero);
  const float2 mn = __bfloat1622float2(__hmin2(x, zero));
  const __nv_bfloat162 e = __floats2bfloat162_rn(__expf(mn.x), __expf(mn.y));
  const __nv_bfloat162 r = __hadd2(mx, e);
  return *reinterpret_cast<const uint32_t*>(&r);
}

// Two bf16 (one 32-bit word) -> float2, exact.
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// Shared-memory matrix descriptor, 128-byte swizzle (layout type 2),
// descriptor version 1 (bits 46-47), base offset 0 (tile bases 1024-aligned).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor of kind::f16 with bf16 A/B and float32 D.
// a_mn / b_mn select MN-major operands; N % 16 == 0 (M = 128), 16 <= N <= 256.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Same for fp16 A/B (format 0).
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

// Byte offset of element (row, col) (col < 64, bf16) inside a 128-byte
// swizzled tile whose base is 1024-byte aligned.
__host__ __device__ constexpr uint32_t sw128_offset(uint32_t row, uint32_t col) {
  return row * 128u + ((((col >> 3) ^ (row & 7u)) & 7u) << 4) + ((col & 7u) << 1);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

}  // namespace tc
}  // namespace mhla
