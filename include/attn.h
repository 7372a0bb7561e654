/*
 * attn.h -- C ABI of the GB300 (sm_103a) exact attention forward library.
 *
 * The operation is exact softmax attention, computed by one fused tiled kernel
 * that never writes the N x N score matrix to memory:
 *
 *   O   = softmax(scale * Q K^T  [+ causal mask]) V
 *   lse = per-row log-sum-exp of the scaled (masked) logits, natural log
 *
 * Definition: "FlashAttention -- one, two, three!", section "Standard
 * Attention" (the three-pass computation whose result is reproduced exactly),
 * and sections "FlashAttention v1." (tiling, running denominator, a few
 * per-row constants kept in global memory) and "FlashAttention v2." (deferred
 * normalisation, parallelism over batch, heads and sequence).  The FP8 entry
 * points follow "Incoherent Processing for FP8 Accuracy" (FlashAttention-3
 * podcast page) and item 3 of "Метод" in the comrad404 review (block
 * quantisation plus a random-sign Hadamard rotation of Q and K).
 *
 * Conventions shared by every entry point:
 *  - Layout: Q, K, V, O are contiguous [B, H, N, d] (row-major, d innermost);
 *    self-attention, so queries and keys share N.  lse is contiguous [B, H, N].
 *    attn_fwd_ex also takes Q, K, V, O as contiguous [B, N, H, d], and
 *    queries and keys of different lengths (Nq, Nk).
 *  - Device pointers are CUDA device addresses on the current device; every
 *    tensor base must be 16-byte aligned (lse: 4-byte aligned).
 *  - Ownership: the caller owns every buffer.  The library allocates no device
 *    memory per call.  It keeps one device status word per kernel module and,
 *    as the one exception, a fixed 64 MiB array in its own device memory that
 *    serves only attn_fwd_host_noalloc (resident on every device that loads
 *    the library, until the process exits).
 *  - Streams: `stream` is a cudaStream_t (NULL = legacy default stream).  All
 *    device-pointer entry points are asynchronous on that stream.
 *  - Errors: arguments are validated before anything is launched; a bad
 *    argument returns a status code and launches nothing.  Nothing throws
 *    across this boundary.  A kernel whose internal wait runs past its time
 *    limit stops cleanly and records ATTN_ERR_TIMEOUT in the device status
 *    word, read with attn_get_device_status().
 *  - Causal mask: query i sees keys j <= i (queries and keys aligned at 0;
 *    attn_fwd_ex can align them at the end instead).  Keys beyond N never
 *    contribute; rows beyond N are never written.
 */
#ifndef GB300_ATTN_H
#define GB300_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1, /* NULL pointer, non-positive size, non-finite scale, ... */
  ATTN_ERR_UNSUPPORTED = 2, /* head dim or dtype this build has no kernel for */
  ATTN_ERR_MISALIGNED = 3,  /* a base pointer breaks the alignment rule above */
  ATTN_ERR_CUDA = 4,        /* a CUDA runtime / driver call failed (see attn_last_cuda_error) */
  ATTN_ERR_TIMEOUT = 5      /* a kernel wait ran past its limit (device status word) */
} attn_status;

typedef enum { ATTN_FP16 = 0, ATTN_BF16 = 1 } attn_dtype;

/* Memory layout of Q, K, V and O (lse is [B, H, N] in both). */
#define ATTN_LAYOUT_BHND 0 /* [B, H, N, d]: each head's rows contiguous */
#define ATTN_LAYOUT_BNHD 1 /* [B, N, H, d]: each token's heads contiguous */

/* Causal mask of attn_fwd_ex over Nq queries and Nk keys (the two coincide when
 * Nq = Nk, where they are the causal mask of self-attention). */
#define ATTN_CAUSAL_NONE 0         /* every key visible */
#define ATTN_CAUSAL_TOP_LEFT 1     /* query i sees keys j <= i */
#define ATTN_CAUSAL_BOTTOM_RIGHT 2 /* query i sees keys j <= i + Nk - Nq (requires Nq <= Nk) */

/*
 * attn_fwd -- exact attention forward, 16-bit inputs and output.
 *
 *   q, k, v : [B, H, N, d] device, dtype `dtype` (fp16 or bf16), read only.
 *   o       : [B, H, N, d] device, same dtype, written (rounded to nearest even).
 *   lse     : [B, H, N] device float32, written; may be NULL (not written).
 *   B, H, N : >= 0 each; when B*H*N == 0 nothing is launched and ATTN_OK returned.
 *   d       : head dimension, one of 64, 128, 256.
 *   causal  : 0 = full attention, 1 = causal mask.
 *   scale   : multiplies Q K^T before the softmax; any finite value (0 allowed).
 *   stream  : cudaStream_t.
 *
 * Accumulation is float32 on the tensor cores; the softmax weights P are
 * rounded to the input dtype before the P V product, and O is normalised once
 * at the end.  Returns ATTN_OK once the kernel is enqueued.
 */
attn_status attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                     int N, int d, int causal, float scale, attn_dtype dtype, void* stream);

/*
 * attn_fwd_workspace_bytes -- workspace (bytes) that lets attn_fwd_ws and
 * attn_fwd_fp8_ws balance full attention over the GPU's SMs, for head
 * dimension d on the current device; 0 when d has no balanced schedule
 * (d = 256, or a d this build does not take).  It depends only on d and the
 * device's SM count (about 40 MiB at d = 128 on 152 SMs).
 */
size_t attn_fwd_workspace_bytes(int d);

/*
 * attn_fwd_ws -- attn_fwd with a caller-provided device workspace, used to
 * balance the work over the SMs when it does not divide evenly.
 *
 * Work is scheduled per CTA (one per SM) in units of two 128-row query tiles
 * of one head.  When the units do not divide evenly over the SMs, the last
 * round leaves SMs idle while it costs a full unit.  With a workspace, full
 * attention (causal = 0, d <= 128, at least one unit per SM) instead runs the
 * whole rounds as before and cuts the (unit, key block) steps of the last
 * units (at least half a round of them) into equal contiguous ranges, one
 * per CTA (a stream-K tail): a unit cut between CTAs is computed in parts
 * over disjoint key ranges, each writes its unnormalised O and its running
 * maximum and sum to the workspace, and the part that finishes last merges
 * them with the online-softmax rescaling and writes O and lse.  Every
 * operand type takes the tail (not under ATTN_SCHEDULE_ONE_TILE); results
 * equal attn_fwd's up to the float32 summation order (FP8: up to the E4M3
 * rounding of each part's weights).  Causal attention and other shapes run exactly
 * as attn_fwd.
 *
 *   workspace       : device buffer, 256-byte aligned (else ATTN_ERR_MISALIGNED),
 *                     owned by the caller; NULL or fewer than
 *                     attn_fwd_workspace_bytes(d) bytes = attn_fwd's schedule.
 *                     The call zeroes the arrival counters in it on `stream`
 *                     before the launch.  Calls whose GPU work overlaps must
 *                     use different workspaces.
 * Other arguments, rules and errors: attn_fwd.
 */
attn_status attn_fwd_ws(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                        int N, int d, int causal, float scale, attn_dtype dtype, void* workspace,
                        size_t workspace_bytes, void* stream);

/*
 * attn_fwd_ex -- attn_fwd generalised to Nq queries over Nk keys and to a
 * second memory layout.
 *
 *   q, o   : Nq rows per head; k, v : Nk rows per head.
 *   layout : ATTN_LAYOUT_BHND (q, o [B, H, Nq, d]; k, v [B, H, Nk, d]) or
 *            ATTN_LAYOUT_BNHD (q, o [B, Nq, H, d]; k, v [B, Nk, H, d], the
 *            layout a projection of [B, N, H*d] activations gives, so that no
 *            transpose is needed).  lse is [B, H, Nq] either way.
 *   causal : ATTN_CAUSAL_NONE, ATTN_CAUSAL_TOP_LEFT or ATTN_CAUSAL_BOTTOM_RIGHT
 *            (the queries are the last Nq of Nk positions: cross-attention
 *            over a key prefix, chunked prefill).
 *
 * The FlashAttention pages define the causal mask for self-attention only;
 * for Nq != Nk both alignments above are readings of it.  With Nq = Nk and
 * layout BHND this is attn_fwd, bit for bit; BNHD gives the same values,
 * element for element, as BHND on the transposed inputs.
 * Errors (ATTN_ERR_INVALID_ARG, nothing launched): a `layout` or `causal`
 * value not listed; Nk < 0; when B*H*Nq > 0, Nk == 0 or BOTTOM_RIGHT with
 * Nq > Nk (a query row would see no key).  ATTN_ERR_UNSUPPORTED: Nq or Nk
 * above 2^30.  Otherwise attn_fwd's rules and errors, with N read as Nq.
 */
attn_status attn_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                        int Nq, int Nk, int d, int causal, float scale, attn_dtype dtype, int layout,
                        void* stream);

/*
 * attn_fwd_host_workspace_bytes -- device workspace (bytes) attn_fwd_host needs
 * for these sizes: room for Q, K, V, O and lse, each 256-byte aligned.
 */
size_t attn_fwd_host_workspace_bytes(int B, int H, int N, int d, attn_dtype dtype);

/*
 * attn_fwd_host -- the same operation on HOST buffers.
 *
 *   q_host, k_host, v_host : [B, H, N, d] host memory (pinned memory makes the
 *                            copies asynchronous and fast), read only.
 *   o_host                 : [B, H, N, d] host, written.
 *   lse_host               : [B, H, N] host float32, written; may be NULL.
 *   workspace              : device buffer of at least
 *                            attn_fwd_host_workspace_bytes(...) bytes, 256-byte
 *                            aligned, owned by the caller.
 * Copies the inputs host->device on `stream`, runs attn_fwd, copies O (and lse)
 * back, and synchronises `stream` before returning.
 */
attn_status attn_fwd_host(const void* q_host, const void* k_host, const void* v_host, void* o_host,
                          float* lse_host, int B, int H, int N, int d, int causal, float scale,
                          attn_dtype dtype, void* workspace, size_t workspace_bytes, void* stream);

/*
 * attn_fwd_host_noalloc -- attn_fwd_host for callers that cannot allocate device
 * memory, with no workspace argument.  The paper has no counterpart: this is a
 * deployment variant of the host-buffer entry point.
 *
 * Who needs it: plugins whose host framework owns all device memory and forbids
 * allocating inside a call, processes whose device memory is fully reserved by
 * another allocator (a cudaMalloc would fail), and latency-critical callers
 * (cudaMalloc / cudaFree may synchronise the device).
 *
 * The device copies of Q, K, V, O and lse live in one fixed array of
 * ATTN_NOALLOC_SCRATCH_BYTES inside the library's device memory, held by every
 * GPU that loads the library until the process exits.  The call allocates
 * nothing (no cudaMalloc, cudaFree or allocating library routine).
 *  - Size limit: returns ATTN_ERR_INVALID_ARG, launching nothing, when
 *    attn_fwd_host_workspace_bytes(B, H, N, d, dtype) exceeds
 *    ATTN_NOALLOC_SCRATCH_BYTES.
 *  - Set-up: the first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current); make that first call
 *    before any stream capture.
 *  - Sharing: every call uses the same array, which keeps the last call's
 *    contents; nothing in it has to start at zero (each call writes every byte
 *    it reads).  Calls whose GPU work overlaps (other host threads or streams
 *    at the same time) race on the array and must not be issued.
 * Other arguments, copies and synchronisation as for attn_fwd_host.  As there,
 * ATTN_OK means the copies and the kernel ran to completion on the GPU, but a
 * kernel whose internal wait ran past its limit stops early and leaves O and
 * lse unfinished while the call still returns ATTN_OK: follow a successful
 * call with attn_get_device_status() to rule that out.
 */
#define ATTN_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)
attn_status attn_fwd_host_noalloc(const void* q_host, const void* k_host, const void* v_host,
                                  void* o_host, float* lse_host, int B, int H, int N, int d,
                                  int causal, float scale, attn_dtype dtype, void* stream);

/*
 * attn_fp8_prepare -- FP8 pre-pass: incoherent processing and block quantisation
 * ("Incoherent Processing for FP8 Accuracy", FlashAttention-3 podcast page;
 * comrad404 review, "Метод", item 3).
 *
 *   q, k, v     : [B, H, N, d] device, dtype `in_dtype` (fp16 or bf16), read only.
 *   q8, k8, v8  : [B, H, N, d] device, E4M3 codes (one byte each), written.
 *   q_scale, k_scale, v_scale : device float32, written.  Per-block mode:
 *                 [B, H, ceil(N/128)], one scale per 128 rows of a head.
 *                 Per-tensor mode: one float each.
 *   signs       : [H, d] device int8, +1 / -1, 16-byte aligned (else
 *                 ATTN_ERR_MISALIGNED); NULL = no rotation.  With signs,
 *                 every row x of Q and K (head h) is replaced by
 *                 (x * signs[h]) H_d / sqrt(d), H_d the Sylvester Hadamard
 *                 matrix (an orthogonal map shared by Q and K, so Q K^T is
 *                 unchanged); V is never rotated.
 *   per_tensor  : 0 = per-block scales (the FP8 method); 1 = one scale per
 *                 tensor (the naive FP8 baseline the pages compare against).
 *   d           : 64, 128 or 256.
 * Quantisation: s = amax / 448 over the block (or tensor), 1 if amax = 0;
 * code = E4M3(x / s), division and rounding (nearest even, saturating to
 * +-448) in float32.  Asynchronous on `stream`.
 */
attn_status attn_fp8_prepare(const void* q, const void* k, const void* v, attn_dtype in_dtype,
                             void* q8, void* k8, void* v8, float* q_scale, float* k_scale,
                             float* v_scale, const int8_t* signs, int per_tensor, int B, int H,
                             int N, int d, void* stream);

/*
 * attn_fp8_prepare_rotary -- attn_fp8_prepare with the rotary position
 * embedding of Q and K fused in front of the rotation ("Incoherent Processing
 * for FP8 Accuracy", FlashAttention-3 podcast page: the Hadamard transform is
 * fused into the memory-bound rotary step).  The pages do not define the
 * embedding; it is RoFormer's: pair i of the row at position n, a feature pair
 * (a, b), becomes (a cos - b sin, a sin + b cos) with cos, sin the table
 * entries (n, i).
 *
 *   rope_cos, rope_sin : [N, d/2] device float32, row n for query / key row n
 *                        (the caller's rotary cache, position offset and
 *                        frequencies included), 16-byte aligned (else
 *                        ATTN_ERR_MISALIGNED); both NULL = no embedding, exactly
 *                        attn_fp8_prepare; one NULL = ATTN_ERR_INVALID_ARG.
 *   rope_interleaved   : nonzero = pairs (2i, 2i+1), 0 = pairs (i, i + d/2).
 * Order per row of Q and K: rotary embedding, sign flip, Hadamard transform,
 * quantisation, all in float32 registers in one pass.  V is untouched by
 * both rotations.  Other arguments, rules and errors: attn_fp8_prepare.
 */
attn_status attn_fp8_prepare_rotary(const void* q, const void* k, const void* v, attn_dtype in_dtype,
                                    void* q8, void* k8, void* v8, float* q_scale, float* k_scale,
                                    float* v_scale, const int8_t* signs, int per_tensor,
                                    const float* rope_cos, const float* rope_sin, int rope_interleaved,
                                    int B, int H, int N, int d, void* stream);

/*
 * attn_fwd_fp8 -- exact attention forward on E4M3 operands with float32 scales
 * (as written by attn_fp8_prepare), bf16 output.  The FP8 tensor-core path of
 * "New GPU Features on Hopper: WGMMA, TMA, FP8" (FlashAttention-3 podcast
 * page), on the block-quantised operands of item 3 of "Метод" in the
 * comrad404 review.
 *
 *   q8, k8, v8 : [B, H, N, d] device E4M3 codes, read only; the true values are
 *                code * scale of their 128-row block (or of the tensor).
 *   q_scale, k_scale, v_scale : device float32, layout as for attn_fp8_prepare.
 *   per_tensor : 1 if the scales are single per-tensor values.  This argument
 *                widens the planned interface: it lets the same kernel run
 *                the naive per-tensor FP8 baseline the pages compare against.
 *   o          : [B, H, N, d] device bf16, written.
 *   lse        : [B, H, N] device float32 or NULL.
 *   d          : 64, 128 or 256.  Other arguments as for attn_fwd.
 * Both products run on the FP8 tensor cores with float32 accumulation; the
 * softmax runs in float32 and P is rounded to E4M3 before P V.  When the
 * queries and keys were rotated by attn_fp8_prepare, O and lse are those of
 * the unrotated inputs (up to quantisation).
 */
attn_status attn_fwd_fp8(const void* q8, const void* k8, const void* v8, const float* q_scale,
                         const float* k_scale, const float* v_scale, int per_tensor, void* o,
                         float* lse, int B, int H, int N, int d, int causal, float scale,
                         void* stream);

/*
 * attn_fwd_fp8_ws -- attn_fwd_fp8 with the balanced schedule of attn_fwd_ws
 * (same workspace rules; the FP8 kernel's per-part O includes its V scale).
 */
attn_status attn_fwd_fp8_ws(const void* q8, const void* k8, const void* v8, const float* q_scale,
                            const float* k_scale, const float* v_scale, int per_tensor, void* o,
                            float* lse, int B, int H, int N, int d, int causal, float scale,
                            void* workspace, size_t workspace_bytes, void* stream);

/*
 * attn_bwd_workspace_bytes -- device workspace (bytes) attn_bwd needs: a float32
 * dQ accumulator [B, H, N, d] and the row dot products D [B, H, N], each
 * 256-byte aligned.  0 for a head dimension attn_bwd does not take.
 */
size_t attn_bwd_workspace_bytes(int B, int H, int N, int d);

/*
 * attn_bwd -- backward pass of attn_fwd: dQ, dK, dV for a given dO = dL/dO.
 * The softmax weights are recomputed block by block from Q, K and the
 * forward's lse instead of being stored ("FlashAttention -- one, two,
 * three!", section "FlashAttention v1.", the recomputation in the backward
 * pass); lse is an auxiliary output, no gradient flows through it.  With
 * P = exp(scale Q K^T - lse) (masked entries 0) and D = rowsum(dO o O):
 *   dV = P^T dO,   dS = P o (dO V^T - D),   dQ = scale dS K,   dK = scale dS^T Q.
 *
 *   q, k, v, o, dout : [B, H, N, d] device, dtype `dtype`, read only; o and lse
 *                      are attn_fwd's outputs for q, k, v (same causal, scale).
 *   lse              : [B, H, N] device float32.
 *   dq, dk, dv       : [B, H, N, d] device, dtype `dtype`, written (rounded to
 *                      nearest even once, from float32 accumulation).
 *   d                : 64 or 128 (else ATTN_ERR_UNSUPPORTED).
 *   causal, scale    : as for attn_fwd.
 *   workspace        : device, 256-byte aligned, at least
 *                      attn_bwd_workspace_bytes(B, H, N, d) bytes, owned by the
 *                      caller; the call clears what it uses.
 * The products run on tcgen05 with float32 accumulation in tensor memory; P
 * and dS are rounded to the input dtype before the products that take them.
 * Asynchronous on `stream` (three kernels and one memset).  Errors as for
 * attn_fwd; a NULL workspace or one that is too small: ATTN_ERR_INVALID_ARG.
 */
attn_status attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                     const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                     int causal, float scale, attn_dtype dtype, void* workspace,
                     size_t workspace_bytes, void* stream);

/*
 * attn_get_device_status -- synchronises `stream`, then returns and clears the
 * device status word of every kernel module: ATTN_ERR_TIMEOUT if any kernel
 * recorded a timed-out wait since the last call, else ATTN_OK (ATTN_ERR_CUDA if
 * the synchronisation itself failed).
 */
attn_status attn_get_device_status(void* stream);

/*
 * attn_set_wait_timeout_ns -- limit for every internal wait of later launches
 * (default 1e9 ns).  0 restores the default.  Process-wide.
 */
void attn_set_wait_timeout_ns(uint64_t timeout_ns);

/*
 * attn_set_schedule -- work schedule of later launches with two Q tiles per
 * CTA (d <= 128), process-wide; an ablation switch in the spirit of the
 * FlashAttention-3 page's overlap ablation ("Overlapping GEMM and Softmax").
 *   ATTN_SCHEDULE_PINGPONG (default): each CTA holds two 128-row Q tiles and
 *       the softmax of one overlaps the matrix products of the other.
 *   ATTN_SCHEDULE_ONE_TILE: each CTA works on one Q tile at a time (the same
 *       kernel with the second tile idle), so softmax and products of a tile
 *       alternate without overlap.  Same results, bit for bit.
 *   ATTN_SCHEDULE_BALANCED: the same as ATTN_SCHEDULE_PINGPONG (under both,
 *       calls given a workspace, attn_fwd_ws and attn_fwd_fp8_ws, take the
 *       stream-K tail for every operand type); kept for callers that set it.
 * Returns ATTN_ERR_INVALID_ARG for any other value (the mode is unchanged).
 */
#define ATTN_SCHEDULE_PINGPONG 0
#define ATTN_SCHEDULE_ONE_TILE 1
#define ATTN_SCHEDULE_BALANCED 2
attn_status attn_set_schedule(int mode);

/*
 * attn_debug_bounded_wait -- launches one tiny kernel that waits on a barrier
 * nothing ever signals, using the same bounded wait as the attention kernels,
 * with limit `timeout_ns`.  It exists so that the timeout path can be tested
 * without hanging a GPU: afterwards attn_get_device_status() reports
 * ATTN_ERR_TIMEOUT.  Asynchronous on `stream`.
 */
attn_status attn_debug_bounded_wait(uint64_t timeout_ns, void* stream);

/*
 * attn_debug_fail_host_chunk -- test hook for the error path of the host-buffer
 * entry points.  Arms a one-shot failure: the next attn_fwd_host (or
 * attn_fwd_host_noalloc) call enqueues the copies of its pipeline chunk
 * `chunk` and then, in place of that chunk's kernel launch, returns
 * ATTN_ERR_CUDA as if the launch had failed, after waiting for everything it
 * had already enqueued.  Nothing faults on the device.  A negative `chunk`
 * disarms the hook; a chunk index past the call's last chunk never fires and
 * is cleared by that call.
 */
void attn_debug_fail_host_chunk(int chunk);

/*
 * attn_debug_exp2_poly -- test hook for the polynomial 2^x that part of the FP8
 * softmax weights use on the FMA pipe instead of ex2.approx (a cubic after
 * rounding the argument to the nearest integer, with the argument clamped to
 * >= -125; relative error below 7.6e-5 for -125 <= x <= 127).  For n float32
 * values x (device), writes that function to y_poly and CUDA's exp2f to y_ref
 * (device, n floats each).  Asynchronous on `stream`.  ATTN_ERR_INVALID_ARG
 * for n < 0 or a NULL pointer when n > 0.
 */
attn_status attn_debug_exp2_poly(const float* x, float* y_poly, float* y_ref, int n, void* stream);

/*
 * attn_debug_tmem_ld_red -- test hook for the reducing tensor-memory load
 * (tcgen05.ld.red, sm_103a) from which the attention softmax takes the row
 * maximum of S (the minimum when the scale is negative), in its 32-column
 * (16-bit kernels) and 128-column (E4M3 kernel) forms.  x: 128 x cols float32
 * (device, row-major; cols = 32 or 128); row r goes into TMEM lane r and is
 * read back by that load, which writes the values to vals[r] (device, 128 x
 * cols floats) and their maximum (use_min = 0) or minimum (use_min != 0) to
 * ext[r] (device, 128 floats).  One CTA, cols TMEM columns; asynchronous on
 * `stream`.  ATTN_ERR_INVALID_ARG for a NULL pointer or another cols.
 */
attn_status attn_debug_tmem_ld_red(const float* x, float* vals, float* ext, int cols, int use_min,
                                   void* stream);

/* Last CUDA error code seen by the library (cudaError_t as int; 0 = none). */
int attn_last_cuda_error(void);

/* Human-readable name of a status code (static storage). */
const char* attn_status_string(attn_status status);

/* Library version, e.g. "0.1.0". */
const char* attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GB300_ATTN_H */
