// Host helpers of the tensor-core path: TMA tensor-map encoding (through the
// driver entry point, so the library does not link libcuda directly) with a
// cache of encoded maps, and the SM count of the current device.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "tc_host.h"

namespace mhla {
namespace {

std::once_flag g_enc_once;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

constexpr int kMaxDevices = 64;
std::mutex g_sm_mu;
int g_sms[kMaxDevices] = {};

// Encoded maps keyed by everything the encoding reads (base address, rank,
// extents, strides, box, element type, swizzle): a map is a pure function of
// its key, so a hit is always valid, whatever happened to the memory in
// between.  A call encodes up to a dozen maps; a repeated call with the same
// buffers finds them here instead of re-encoding them.  Direct-mapped.
struct MapKey {
  const void* base;
  uint64_t dims[5], strides[4];
  uint32_t box[5];
  int rank, f16, swizzle;
};
struct MapEntry {
  bool used;
  MapKey key;
  CUtensorMap map;
};
constexpr int kMapCache = 512;
std::mutex g_map_mu;
MapEntry g_maps[kMapCache];

uint64_t key_hash(const MapKey& k) {
  // FNV-1a over the key's bytes
  const unsigned char* b = reinterpret_cast<const unsigned char*>(&k);
  uint64_t h = 1469598103934665603ull;
  for (size_t i = 0; i < sizeof(MapKey); ++i) h = (h ^ b[i]) * 1099511628211ull;
  return h;
}

}  // namespace

namespace {
int encode_impl(CUtensorMap* map, const void* base, int rank, const uint64_t* dims, const uint64_t* strides_bytes,
                const uint32_t* box, bool f16, bool swizzle);
}  // namespace

int encode_tmap(CUtensorMap* map, const void* base, int rank, const uint64_t* dims, const uint64_t* strides_bytes,
                const uint32_t* box, bool f16) {
  return encode_impl(map, base, rank, dims, strides_bytes, box, f16, true);
}

int encode_tmap_plain(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                      const uint64_t* strides_bytes, const uint32_t* box) {
  return encode_impl(map, base, rank, dims, strides_bytes, box, false, false);
}

namespace {
int encode_impl(CUtensorMap* map, const void* base, int rank, const uint64_t* dims, const uint64_t* strides_bytes,
                const uint32_t* box, bool f16, bool swizzle) {
  std::call_once(g_enc_once, [] {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode) return (int)cudaErrorNotSupported;
  MapKey key;
  std::memset(&key, 0, sizeof(key));  // padding bytes take part in the hash and the comparison
  key.base = base;
  key.rank = rank;
  key.f16 = f16 ? 1 : 0;
  key.swizzle = swizzle ? 1 : 0;
  for (int i = 0; i < rank; ++i) {
    key.dims[i] = dims[i];
    key.box[i] = box[i];
    if (i + 1 < rank) key.strides[i] = strides_bytes[i];
  }
  MapEntry& slot = g_maps[key_hash(key) % kMapCache];
  {
    std::lock_guard<std::mutex> lock(g_map_mu);
    if (slot.used && std::memcmp(&slot.key, &key, sizeof(key)) == 0) {
      *map = slot.map;
      return 0;
    }
  }
  cuuint64_t gdim[5];
  cuuint64_t gstride[4];
  cuuint32_t bdim[5];
  cuuint32_t estride[5];
  for (int i = 0; i < rank; ++i) {
    gdim[i] = dims[i];
    bdim[i] = box[i];
    estride[i] = 1;
    if (i + 1 < rank) gstride[i] = strides_bytes[i];
  }
  CUresult r = g_encode(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void*>(base), gdim,
                        gstride, bdim, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return (int)cudaErrorInvalidValue;
  std::lock_guard<std::mutex> lock(g_map_mu);
  slot.used = true;
  slot.key = key;
  slot.map = *map;
  return 0;
}
}  // namespace

int encode_token_map(CUtensorMap* map, const Plan& p, const void* base, const ChunkShape& c) {
  const uint32_t box[5] = {64, (uint32_t)c.cw, (uint32_t)c.ch, (uint32_t)c.ct, 1};
  if (p.layout == MHLA_LAYOUT_BHND) {
    const uint64_t dims[5] = {64, (uint64_t)p.Wg, (uint64_t)p.Hg, (uint64_t)p.T, (uint64_t)p.BH};
    const uint64_t str[4] = {128, 128ull * p.Wg, 128ull * p.Wg * p.Hg, 128ull * p.N};
    return encode_tmap_bf16(map, base, 5, dims, str, box);
  }
  // token-major: the head axis (128 bytes) comes right after the features, a
  // token row is H * 128 bytes, (batch, time) share one axis of Hg * Wg rows
  const uint32_t box_t[5] = {64, 1, (uint32_t)c.cw, (uint32_t)c.ch, (uint32_t)c.ct};
  const uint64_t row = 128ull * p.H;
  const uint64_t dims[5] = {64, (uint64_t)p.H, (uint64_t)p.Wg, (uint64_t)p.Hg, (uint64_t)p.T * p.B};
  const uint64_t str[4] = {128, row, row * p.Wg, row * p.Wg * p.Hg};
  return encode_tmap_bf16(map, base, 5, dims, str, box_t);
}

ChunkShape choose_chunk(const Plan& p) {
  auto largest_divisor = [](int n, int limit) {
    for (int d = limit < n ? limit : n; d >= 1; --d)
      if (n % d == 0) return d;
    return 1;
  };
  ChunkShape c;
  c.cw = largest_divisor(p.bw, kTcTileRows);
  c.ch = largest_divisor(p.bh, kTcTileRows / c.cw);
  c.ct = largest_divisor(p.bt, kTcTileRows / (c.cw * c.ch));
  c.ncx = p.bw / c.cw;
  c.ncy = p.bh / c.ch;
  c.nct = p.bt / c.ct;
  c.per_block = c.ncx * c.ncy * c.nct;
  c.f_ncx = make_fastdiv((uint32_t)c.ncx);
  c.f_ncxy = make_fastdiv((uint32_t)(c.ncx * c.ncy));
  c.rows = c.ct * c.ch * c.cw;
  c.rows_pad = (c.rows + 15) / 16 * 16;
  return c;
}

// Kernels whose shared-memory limit has been raised, per current context
// (a device reset or another context starts afresh).  The context is read
// through the driver entry point, like the tensor-map encoder.
int set_max_dynamic_smem(const void* kernel, int bytes) {
  struct Done {
    const void* kernel;
    CUcontext ctx;
    int bytes;
  };
  static std::once_flag once;
  static PFN_cuCtxGetCurrent_v4000 get_ctx = nullptr;
  static std::mutex mu;
  static Done done[256];
  static int n_done = 0;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_ctx = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
  });
  // no current context yet: the runtime call creates the primary one
  CUcontext ctx = nullptr;
  if (!get_ctx || get_ctx(&ctx) != CUDA_SUCCESS || !ctx)
    return (int)cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  std::lock_guard<std::mutex> lock(mu);
  int slot = -1;
  for (int i = 0; i < n_done; ++i) {
    if (done[i].kernel == kernel && done[i].ctx == ctx) {
      if (done[i].bytes >= bytes) return 0;
      slot = i;
      break;
    }
  }
  const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return (int)e;
  if (slot < 0) slot = n_done < 256 ? n_done++ : (int)(((uintptr_t)kernel >> 4) % 256);
  done[slot] = Done{kernel, ctx, bytes};
  return 0;
}

int num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
  std::lock_guard<std::mutex> lock(g_sm_mu);
  if (!g_sms[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    g_sms[dev] = n;
  }
  return g_sms[dev];
}

}  // namespace mhla
