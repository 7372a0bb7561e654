// host_common.cu -- shared host helpers and the library-wide C ABI entry points
// (status, timeouts, version).
#include "host_common.h"

#include <atomic>
#include <cstring>
#include <mutex>

#include "tmap_cache.h"

namespace attn_internal {

namespace {
std::atomic<uint64_t> g_timeout_ns{kDefaultWaitTimeoutNs};
std::atomic<int> g_schedule{ATTN_SCHEDULE_PINGPONG};
std::atomic<int> g_last_cuda_error{0};

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}
}  // namespace

uint64_t wait_timeout_ns() { return g_timeout_ns.load(std::memory_order_relaxed); }
int schedule_mode() { return g_schedule.load(std::memory_order_relaxed); }

void record_cuda_error(cudaError_t e) {
  if (e != cudaSuccess) g_last_cuda_error.store(static_cast<int>(e));
}

attn_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return ATTN_OK;
  record_cuda_error(e);
  return ATTN_ERR_CUDA;
}

int sm_count() {
  static std::mutex mu;
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (dev < 64 && cached[dev] > 0) return cached[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev < 64) cached[dev] = n;
  return n;
}

namespace {
// 32 recent maps (a launch encodes four).
TmapCache<CUtensorMap, 32> g_tmaps;
}  // namespace

bool encode_tmap_4d(CUtensorMap* out, CUtensorMapDataType dtype, const void* base,
                    const uint64_t (&dims)[4], const uint64_t (&strides)[3], const uint32_t (&box)[4],
                    CUtensorMapSwizzle swizzle) {
  TmapKey key;
  std::memset(&key, 0, sizeof(key));
  key.base = reinterpret_cast<uint64_t>(base);
  for (int i = 0; i < 4; ++i) key.dims[i] = dims[i], key.box[i] = box[i];
  for (int i = 0; i < 3; ++i) key.strides[i] = strides[i];
  key.dtype = static_cast<uint32_t>(dtype);
  key.swizzle = static_cast<uint32_t>(swizzle);
  if (g_tmaps.find(key, out)) return true;
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t gdims[4] = {dims[0], dims[1], dims[2], dims[3]};
  const cuuint64_t gstrides[3] = {strides[0], strides[1], strides[2]};
  const cuuint32_t gbox[4] = {box[0], box[1], box[2], box[3]};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(out, dtype, 4, const_cast<void*>(base), gdims, gstrides, gbox, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  g_tmaps.insert(key, *out);
  return true;
}

}  // namespace attn_internal

using namespace attn_internal;

ATTN_EXPORT attn_status attn_get_device_status(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_status(e);
  unsigned int a = 0, b = 0, c = 0;
  if ((e = fwd_status_exchange(&a)) != cudaSuccess) return cuda_status(e);
  if ((e = fp8_status_exchange(&b)) != cudaSuccess) return cuda_status(e);
  if ((e = bwd_status_exchange(&c)) != cudaSuccess) return cuda_status(e);
  return (a | b | c) ? ATTN_ERR_TIMEOUT : ATTN_OK;
}

ATTN_EXPORT void attn_set_wait_timeout_ns(uint64_t timeout_ns) {
  g_timeout_ns.store(timeout_ns ? timeout_ns : kDefaultWaitTimeoutNs);
}

ATTN_EXPORT attn_status attn_set_schedule(int mode) {
  if (mode != ATTN_SCHEDULE_PINGPONG && mode != ATTN_SCHEDULE_ONE_TILE && mode != ATTN_SCHEDULE_BALANCED)
    return ATTN_ERR_INVALID_ARG;
  g_schedule.store(mode);
  return ATTN_OK;
}

ATTN_EXPORT int attn_last_cuda_error(void) { return g_last_cuda_error.load(); }

ATTN_EXPORT const char* attn_status_string(attn_status s) {
  switch (s) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG";
    case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED";
    case ATTN_ERR_MISALIGNED: return "ATTN_ERR_MISALIGNED";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
    case ATTN_ERR_TIMEOUT: return "ATTN_ERR_TIMEOUT";
  }
  return "ATTN_ERR_UNKNOWN";
}

ATTN_EXPORT const char* attn_version(void) { return "0.1.0"; }
