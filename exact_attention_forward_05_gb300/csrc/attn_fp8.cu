// attn_fp8.cu -- FP8 (E4M3) path: pre-pass and attention kernel.
#include "host_common.h"

namespace {
__device__ unsigned int g_status_fp8 = 0;
}  // namespace

namespace attn_internal {
cudaError_t fp8_status_exchange(unsigned int* out) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_status_fp8, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_status_fp8, &zero, sizeof(unsigned int));
}
}  // namespace attn_internal
