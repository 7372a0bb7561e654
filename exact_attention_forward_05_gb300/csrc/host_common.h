// host_common.h -- host-side helpers shared by the kernel modules of the
// library (argument checks, TMA descriptor encoding, device properties,
// process-wide settings).  Internal: not part of the C ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "attn.h"

#define ATTN_EXPORT extern "C" __attribute__((visibility("default")))

namespace attn_internal {

// Device status word bits (any bit set reads back as ATTN_ERR_TIMEOUT).
enum : unsigned int {
  kStatusTimeoutLoad = 1u << 0,
  kStatusTimeoutMma = 1u << 1,
  kStatusTimeoutSoftmax = 1u << 2,
  kStatusTimeoutDebug = 1u << 3,
  kStatusTimeoutPrep = 1u << 4,
};

constexpr uint64_t kDefaultWaitTimeoutNs = 1000000000ull;

uint64_t wait_timeout_ns();
int schedule_mode();  // ATTN_SCHEDULE_* of later launches
void record_cuda_error(cudaError_t e);
attn_status cuda_status(cudaError_t e);  // records and maps to ATTN_OK / ATTN_ERR_CUDA

// Multiprocessor count of the current device (cached per device).
int sm_count();

// Encode a 4-D tiled TMA descriptor: dims[0] is contiguous, strides[i] is the
// byte stride of dims[i + 1] (a multiple of 16).  Out-of-bounds elements of a
// load read as zero; a store skips them.  Returns false on failure.
bool encode_tmap_4d(CUtensorMap* out, CUtensorMapDataType dtype, const void* base,
                    const uint64_t (&dims)[4], const uint64_t (&strides)[3], const uint32_t (&box)[4],
                    CUtensorMapSwizzle swizzle);

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Per-module status exchange: read the module's device status word and clear it.
cudaError_t fwd_status_exchange(unsigned int* out);
cudaError_t fp8_status_exchange(unsigned int* out);
cudaError_t bwd_status_exchange(unsigned int* out);

}  // namespace attn_internal
