// attn_fwd.cu -- C ABI of the 16-bit (fp16 / bf16) exact attention forward:
// argument checks and dispatch to attn_kernel::attn_fwd_kernel<D, kind>
// (attn_kernel.cuh), the host-buffer entry point, and the bounded-wait probe.
#include <atomic>
#include <cmath>
#include <mutex>

#include "attn_kernel.cuh"

using namespace sm103;
using attn_kernel::FwdParams;
using attn_kernel::KIND_BF16;
using attn_kernel::KIND_F16;

namespace {

template <int D, int KIND>
attn_status launch(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                   int Nq, int Nk, int causal, float scale, int layout, cudaStream_t stream,
                   void* ws = nullptr, size_t ws_bytes = 0) {
  FwdParams prm{};
  prm.o = o;
  prm.lse = lse;
  prm.causal = causal != ATTN_CAUSAL_NONE;
  prm.causal_off = causal == ATTN_CAUSAL_BOTTOM_RIGHT ? Nk - Nq : 0;
  prm.layout = layout;
  return attn_kernel::launch_fwd<D, KIND>(q, k, v, prm, B, H, Nq, Nk, scale, stream, ws, ws_bytes);
}

__global__ void debug_wait_kernel(uint64_t timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const WaitCtx wc{&abort_flag, &attn_kernel::g_status_word, timeout_ns};
    mbar_wait(smem_u32(&bar), 0, wc, attn_internal::kStatusTimeoutDebug);  // nothing arrives
  }
  __syncthreads();
}

// Evaluates exp2_poly2 (the FMA-pipe 2^x of the FP8 weights) and, beside it,
// CUDA's exp2f, on n values: thread i takes elements 2i and 2i + 1.
__global__ void debug_exp2_kernel(const float* x, float* y_poly, float* y_ref, int n) {
  const int i = 2 * (blockIdx.x * blockDim.x + threadIdx.x);
  if (i >= n) return;
  const bool two = i + 1 < n;
  const float2 v = make_float2(x[i], two ? x[i + 1] : x[i]);
  const float2 r = exp2_poly2(v);
  y_poly[i] = r.x;
  y_ref[i] = exp2f(v.x);
  if (two) {
    y_poly[i + 1] = r.y;
    y_ref[i + 1] = exp2f(v.y);
  }
}

attn_status check_args(const void* q, const void* k, const void* v, const void* o, const float* lse,
                       int B, int H, int N, int d, float scale, int dtype) {
  if (B < 0 || H < 0 || N < 0) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_FP16 && dtype != ATTN_BF16) return ATTN_ERR_UNSUPPORTED;
  if (d != 64 && d != 128 && d != 256) return ATTN_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(B) * H > 0x7fffffff) return ATTN_ERR_INVALID_ARG;
  if (static_cast<int64_t>(B) * H * N == 0) return ATTN_OK;
  if (!q || !k || !v || !o) return ATTN_ERR_INVALID_ARG;
  using attn_internal::aligned;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16)) return ATTN_ERR_MISALIGNED;
  if (lse && !aligned(lse, 4)) return ATTN_ERR_MISALIGNED;
  return ATTN_OK;
}

using attn_kernel::align256;

// Longest query or key sequence attn_fwd_ex takes: row and key indices plus a
// tile stay inside int arithmetic in the kernel.
constexpr int kMaxRows = 1 << 30;

}  // namespace

namespace attn_internal {
cudaError_t fwd_status_exchange(unsigned int* out) { return attn_kernel::status_exchange(out); }
}  // namespace attn_internal

ATTN_EXPORT attn_status attn_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                                    int H, int Nq, int Nk, int d, int causal, float scale,
                                    attn_dtype dtype, int layout, void* stream) {
  if (layout != ATTN_LAYOUT_BHND && layout != ATTN_LAYOUT_BNHD) return ATTN_ERR_INVALID_ARG;
  if (causal != ATTN_CAUSAL_NONE && causal != ATTN_CAUSAL_TOP_LEFT && causal != ATTN_CAUSAL_BOTTOM_RIGHT)
    return ATTN_ERR_INVALID_ARG;
  if (Nk < 0) return ATTN_ERR_INVALID_ARG;
  if (Nq > kMaxRows || Nk > kMaxRows) return ATTN_ERR_UNSUPPORTED;
  attn_status st = check_args(q, k, v, o, lse, B, H, Nq, d, scale, dtype);
  if (st != ATTN_OK || static_cast<int64_t>(B) * H * Nq == 0) return st;
  // Every query row must see at least one key.
  if (Nk == 0 || (causal == ATTN_CAUSAL_BOTTOM_RIGHT && Nq > Nk)) return ATTN_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool bf = dtype == ATTN_BF16;
  switch (d) {
    case 64: return bf ? launch<64, KIND_BF16>(q, k, v, o, lse, B, H, Nq, Nk, causal, scale, layout, s)
                       : launch<64, KIND_F16>(q, k, v, o, lse, B, H, Nq, Nk, causal, scale, layout, s);
    case 128: return bf ? launch<128, KIND_BF16>(q, k, v, o, lse, B, H, Nq, Nk, causal, scale, layout, s)
                        : launch<128, KIND_F16>(q, k, v, o, lse, B, H, Nq, Nk, causal, scale, layout, s);
    default: return bf ? launch<256, KIND_BF16>(q, k, v, o, lse, B, H, Nq, Nk, causal, scale, layout, s)
                       : launch<256, KIND_F16>(q, k, v, o, lse, B, H, Nq, Nk, causal, scale, layout, s);
  }
}

ATTN_EXPORT size_t attn_fwd_workspace_bytes(int d) {
  if (d != 64 && d != 128 && d != 256) return 0;
  return attn_kernel::stream_k_ws_bytes(d, attn_internal::sm_count());
}

ATTN_EXPORT attn_status attn_fwd_ws(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                                    int H, int N, int d, int causal, float scale, attn_dtype dtype,
                                    void* workspace, size_t workspace_bytes, void* stream) {
  attn_status st = check_args(q, k, v, o, lse, B, H, N, d, scale, dtype);
  if (st != ATTN_OK || static_cast<int64_t>(B) * H * N == 0) return st;
  if (N > kMaxRows) return ATTN_ERR_UNSUPPORTED;
  if (workspace != nullptr && !attn_internal::aligned(workspace, 256)) return ATTN_ERR_MISALIGNED;
  const int cm = causal ? ATTN_CAUSAL_TOP_LEFT : ATTN_CAUSAL_NONE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool bf = dtype == ATTN_BF16;
  void* w = workspace;
  const size_t wb = workspace_bytes;
  switch (d) {
    case 64: return bf ? launch<64, KIND_BF16>(q, k, v, o, lse, B, H, N, N, cm, scale, ATTN_LAYOUT_BHND, s, w, wb)
                       : launch<64, KIND_F16>(q, k, v, o, lse, B, H, N, N, cm, scale, ATTN_LAYOUT_BHND, s, w, wb);
    case 128: return bf ? launch<128, KIND_BF16>(q, k, v, o, lse, B, H, N, N, cm, scale, ATTN_LAYOUT_BHND, s, w, wb)
                        : launch<128, KIND_F16>(q, k, v, o, lse, B, H, N, N, cm, scale, ATTN_LAYOUT_BHND, s, w, wb);
    default: return bf ? launch<256, KIND_BF16>(q, k, v, o, lse, B, H, N, N, cm, scale, ATTN_LAYOUT_BHND, s, w, wb)
                       : launch<256, KIND_F16>(q, k, v, o, lse, B, H, N, N, cm, scale, ATTN_LAYOUT_BHND, s, w, wb);
  }
}

ATTN_EXPORT attn_status attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                                 int H, int N, int d, int causal, float scale, attn_dtype dtype,
                                 void* stream) {
  return attn_fwd_ex(q, k, v, o, lse, B, H, N, N, d, causal ? ATTN_CAUSAL_TOP_LEFT : ATTN_CAUSAL_NONE,
                     scale, dtype, ATTN_LAYOUT_BHND, stream);
}

namespace {

// Test hook (attn_debug_fail_host_chunk): chunk index at which the next
// attn_fwd_host call stops as if that chunk's launch had failed; -1 = off.
std::atomic<int> g_fail_chunk{-1};

// Streams and events of the host-buffer pipeline, created once per device.
constexpr int kHostChunks = 8;
struct HostPipe {
  std::mutex mu;
  cudaStream_t st[3];  // copies in, kernels, copies out
  cudaEvent_t start;
  cudaEvent_t in[kHostChunks], done[kHostChunks];
};

attn_status host_pipe(HostPipe** out) {
  static std::mutex mu;
  static HostPipe* pipes[64] = {nullptr};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return attn_internal::cuda_status(e);
  if (dev < 0 || dev >= 64) return ATTN_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(mu);
  if (pipes[dev] == nullptr) {
    HostPipe* hp = new HostPipe();
    bool good = true;
    for (int i = 0; i < 3 && good; ++i) good = cudaStreamCreateWithFlags(&hp->st[i], cudaStreamNonBlocking) == cudaSuccess;
    good = good && cudaEventCreateWithFlags(&hp->start, cudaEventDisableTiming) == cudaSuccess;
    for (int c = 0; c < kHostChunks && good; ++c)
      good = cudaEventCreateWithFlags(&hp->in[c], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&hp->done[c], cudaEventDisableTiming) == cudaSuccess;
    if (!good) return attn_internal::cuda_status(cudaGetLastError());  // kept for the process (not freed)
    pipes[dev] = hp;
  }
  *out = pipes[dev];
  return ATTN_OK;
}

}  // namespace

ATTN_EXPORT size_t attn_fwd_host_workspace_bytes(int B, int H, int N, int d, attn_dtype dtype) {
  (void)dtype;
  if (B < 0 || H < 0 || N < 0 || d <= 0) return 0;
  const size_t elems = static_cast<size_t>(B) * H * N * d;
  return 4 * align256(elems * 2) + align256(static_cast<size_t>(B) * H * N * 4);
}

ATTN_EXPORT attn_status attn_fwd_host(const void* q_host, const void* k_host, const void* v_host,
                                      void* o_host, float* lse_host, int B, int H, int N, int d,
                                      int causal, float scale, attn_dtype dtype, void* workspace,
                                      size_t workspace_bytes, void* stream) {
  if (!workspace && static_cast<int64_t>(B) * H * N > 0) return ATTN_ERR_INVALID_ARG;
  attn_status st = check_args(q_host, k_host, v_host, o_host, lse_host, B, H, N, d, scale, dtype);
  if (st != ATTN_OK || static_cast<int64_t>(B) * H * N == 0) return st;
  if (workspace_bytes < attn_fwd_host_workspace_bytes(B, H, N, d, dtype)) return ATTN_ERR_INVALID_ARG;
  if (!attn_internal::aligned(workspace, 256)) return ATTN_ERR_MISALIGNED;
  const size_t bytes = static_cast<size_t>(B) * H * N * d * 2;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint8_t* dq = ws;
  uint8_t* dk = ws + align256(bytes);
  uint8_t* dv = ws + 2 * align256(bytes);
  uint8_t* dout = ws + 3 * align256(bytes);
  float* dlse = reinterpret_cast<float*>(ws + 4 * align256(bytes));
  const uint8_t* hq = static_cast<const uint8_t*>(q_host);
  const uint8_t* hk = static_cast<const uint8_t*>(k_host);
  const uint8_t* hv = static_cast<const uint8_t*>(v_host);
  uint8_t* ho = static_cast<uint8_t*>(o_host);

  // Pipeline over chunks of consecutive (batch, head) pairs, contiguous in
  // every tensor: chunk c's inputs are copied in on one stream while the
  // kernel runs on chunk c - 1 on a second and chunk c - 2's output is copied
  // out on a third, so copies in both directions overlap the compute.
  HostPipe* hp = nullptr;
  st = host_pipe(&hp);
  if (st != ATTN_OK) return st;
  std::lock_guard<std::mutex> lock(hp->mu);  // the streams and events serve one call at a time
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int BH = B * H;
  const int nchunk = BH < kHostChunks ? BH : kHostChunks;
  const size_t row_bytes = static_cast<size_t>(N) * d * 2;  // one (batch, head) of Q/K/V/O
  const int fail_at = g_fail_chunk.exchange(-1);
  cudaError_t e;
  // On any failure, whatever was already enqueued on the pipeline streams
  // (copies into the caller's workspace and host buffers, kernels) finishes
  // before the call returns and the streams are handed to the next call.
  auto drain = [&](attn_status failed) {
    for (int i = 0; i < 3; ++i) cudaStreamSynchronize(hp->st[i]);
    return failed;
  };
  // Work already queued on the caller's stream comes first.
  if ((e = cudaEventRecord(hp->start, s)) != cudaSuccess) return drain(attn_internal::cuda_status(e));
  for (int i = 0; i < 3; ++i)
    if ((e = cudaStreamWaitEvent(hp->st[i], hp->start, 0)) != cudaSuccess) return drain(attn_internal::cuda_status(e));
  for (int c = 0; c < nchunk; ++c) {
    const int bh0 = static_cast<int>(static_cast<int64_t>(BH) * c / nchunk);
    const int bh1 = static_cast<int>(static_cast<int64_t>(BH) * (c + 1) / nchunk);
    const size_t off = row_bytes * bh0, len = row_bytes * (bh1 - bh0);
    if ((e = cudaMemcpyAsync(dq + off, hq + off, len, cudaMemcpyHostToDevice, hp->st[0])) != cudaSuccess ||
        (e = cudaMemcpyAsync(dk + off, hk + off, len, cudaMemcpyHostToDevice, hp->st[0])) != cudaSuccess ||
        (e = cudaMemcpyAsync(dv + off, hv + off, len, cudaMemcpyHostToDevice, hp->st[0])) != cudaSuccess ||
        (e = cudaEventRecord(hp->in[c], hp->st[0])) != cudaSuccess ||
        (e = cudaStreamWaitEvent(hp->st[1], hp->in[c], 0)) != cudaSuccess)
      return drain(attn_internal::cuda_status(e));
    if (c == fail_at) return drain(ATTN_ERR_CUDA);  // test hook: this chunk's launch "fails"
    st = attn_fwd(dq + off, dk + off, dv + off, dout + off,
                  lse_host ? dlse + static_cast<size_t>(N) * bh0 : nullptr, 1, bh1 - bh0, N, d, causal,
                  scale, dtype, hp->st[1]);
    if (st != ATTN_OK) return drain(st);
    if ((e = cudaEventRecord(hp->done[c], hp->st[1])) != cudaSuccess ||
        (e = cudaStreamWaitEvent(hp->st[2], hp->done[c], 0)) != cudaSuccess ||
        (e = cudaMemcpyAsync(ho + off, dout + off, len, cudaMemcpyDeviceToHost, hp->st[2])) != cudaSuccess)
      return drain(attn_internal::cuda_status(e));
    if (lse_host &&
        (e = cudaMemcpyAsync(lse_host + static_cast<size_t>(N) * bh0, dlse + static_cast<size_t>(N) * bh0,
                             static_cast<size_t>(N) * (bh1 - bh0) * 4, cudaMemcpyDeviceToHost, hp->st[2])) !=
            cudaSuccess)
      return drain(attn_internal::cuda_status(e));
  }
  for (int i = 0; i < 3; ++i)
    if ((e = cudaStreamSynchronize(hp->st[i])) != cudaSuccess) return drain(attn_internal::cuda_status(e));
  return attn_internal::cuda_status(cudaStreamSynchronize(s));
}

ATTN_EXPORT attn_status attn_debug_exp2_poly(const float* x, float* y_poly, float* y_ref, int n, void* stream) {
  if (n < 0) return ATTN_ERR_INVALID_ARG;
  if (n == 0) return ATTN_OK;
  if (!x || !y_poly || !y_ref) return ATTN_ERR_INVALID_ARG;
  const int pairs = (n + 1) / 2;
  debug_exp2_kernel<<<(pairs + 255) / 256, 256, 0, static_cast<cudaStream_t>(stream)>>>(x, y_poly, y_ref, n);
  return attn_internal::cuda_status(cudaGetLastError());
}

ATTN_EXPORT void attn_debug_fail_host_chunk(int chunk) { g_fail_chunk.store(chunk < 0 ? -1 : chunk); }

ATTN_EXPORT attn_status attn_debug_bounded_wait(uint64_t timeout_ns, void* stream) {
  debug_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(timeout_ns);
  return attn_internal::cuda_status(cudaGetLastError());
}

// ---------------------------------------------------------------------------
// Host-buffer entry point that allocates nothing.
//
// Some callers cannot allocate device memory: plugins whose host framework owns
// every device allocation through its own pool and forbids allocating inside a
// plugin call; processes whose device memory is already reserved in full by
// another allocator, where a cudaMalloc would fail; and latency-critical code,
// where cudaMalloc / cudaFree may synchronise the device and stall other work.
// For them the device copies that attn_fwd_host keeps in a caller-provided
// workspace live instead in one fixed array in this module's device memory.
// Every GPU that loads the library holds the array until the process exits.
namespace {

constexpr size_t kNoAllocScratchBytes = static_cast<size_t>(ATTN_NOALLOC_SCRATCH_BYTES);
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the array, looked up once per device (with that device
// current).  In host code the symbol itself is only a host-side stand-in.
attn_status noalloc_scratch_address(void** out) {
  static std::mutex mu;
  static void* addr[64] = {nullptr};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return attn_internal::cuda_status(e);
  if (dev < 0 || dev >= 64) return ATTN_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return attn_internal::cuda_status(e);
    addr[dev] = p;
  }
  *out = addr[dev];
  return ATTN_OK;
}

}  // namespace

ATTN_EXPORT attn_status attn_fwd_host_noalloc(const void* q_host, const void* k_host,
                                              const void* v_host, void* o_host, float* lse_host,
                                              int B, int H, int N, int d, int causal, float scale,
                                              attn_dtype dtype, void* stream) {
  attn_status st = check_args(q_host, k_host, v_host, o_host, lse_host, B, H, N, d, scale, dtype);
  if (st != ATTN_OK || static_cast<int64_t>(B) * H * N == 0) return st;
  if (attn_fwd_host_workspace_bytes(B, H, N, d, dtype) > kNoAllocScratchBytes) return ATTN_ERR_INVALID_ARG;
  void* scratch = nullptr;
  if ((st = noalloc_scratch_address(&scratch)) != ATTN_OK) return st;
  return attn_fwd_host(q_host, k_host, v_host, o_host, lse_host, B, H, N, d, causal, scale, dtype,
                       scratch, kNoAllocScratchBytes, stream);
}
