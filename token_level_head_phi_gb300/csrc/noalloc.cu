// Allocation-free entry point: the MHLA forward pass with its scratch memory
// taken from a fixed device array inside this library.
//
// Some callers cannot allocate device memory at the time they call us: code
// running inside an allocator callback or an out-of-memory handler, plugin
// hosts and embedded runtimes that forbid cudaMalloc after start-up, and
// real-time loops that must not touch the allocator (cudaMalloc can
// synchronise the device and its latency is unbounded).  mhla_forward_noalloc
// serves them: the caller still passes Q, K, V, Mc and the output, and the
// intermediate summaries live in kNoallocScratchBytes of static device
// memory that every GPU loading this library holds until the process exits.
//
// The scratch array is an ordinary __device__ symbol.  Host code only sees a
// host-side stand-in for it, so its device address is looked up with
// cudaGetSymbolAddress on every call (for the device current at that call,
// in the context current there; once the library's code is loaded on that
// device the lookup is a table read and allocates nothing) and handed to the
// kernels as a plain pointer.
//
// First call on a device: with CUDA's lazy module loading (the default since
// CUDA 12.2) the part of the library that holds the array may be loaded only
// by that call's lookup, and loading it commits the array's 32 MiB of device
// memory then.  A caller that will need this entry point where it cannot
// allocate (an out-of-memory handler, say) should make one small call at
// start-up, before any stream capture.
#include <cuda_runtime.h>

#include "mhla.h"

namespace {

// 32 MiB: room for the summaries of problems up to a few hundred thousand
// token-heads at d = 64 (e.g. B = 64, H = 3 on a 14 x 14 grid).
constexpr size_t kNoallocScratchBytes = 32ull << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

// Device address of the scratch array on the current device.
mhla_status scratch_address(void** out) {
  void* ptr = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
  if (e != cudaSuccess || !ptr) return MHLA_ERR_CUDA;
  *out = ptr;
  return MHLA_OK;
}

}  // namespace

extern "C" {

mhla_status mhla_forward_noalloc(const void* q, const void* k, const void* v, const float* mc,
                                 const mhla_params* p, void* out, void* stream) {
  size_t need = 0;
  mhla_status st = mhla_workspace_bytes(p, &need);
  if (st != MHLA_OK) return st;
  // larger problems do not fit the static area: refuse before enqueuing anything
  if (need > kNoallocScratchBytes) return MHLA_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (need > 0) {
    st = scratch_address(&scratch);
    if (st != MHLA_OK) return st;
  }
  // Every kernel of the forward pass writes each scratch byte it later
  // reads, so nothing has to be cleared between calls.
  return mhla_forward(q, k, v, mc, p, out, scratch, need > 0 ? kNoallocScratchBytes : 0, stream);
}

}  // extern "C"
