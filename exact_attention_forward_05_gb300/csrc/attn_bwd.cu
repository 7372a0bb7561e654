// attn_bwd.cu -- backward pass of the exact attention: dQ, dK, dV from Q, K, V,
// O, dO and the forward's per-row logsumexp, recomputing the softmax weights
// block by block from Q, K and the saved statistics instead of storing the
// N x N matrix ("FlashAttention -- one, two, three!", section "FlashAttention
// v1.": the backward pass recomputes the attention matrix from blocks of Q, K,
// V brought on chip, using the softmax statistics kept from the forward).
//
// Gradients, by the chain rule through O = softmax(scale S) V with S = Q K^T
// (lse is an auxiliary output: no gradient flows through it):
//   P = exp(scale S - lse),  D_i = sum_c dO_ic O_ic  (= sum_j P_ij dP_ij),
//   dV = P^T dO,  dP = dO V^T,  dS = P o (dP - D),
//   dQ = scale dS K,  dK = scale dS^T Q.
//
// Three kernels:
//   bwd_rowdot_kernel   D = rowsum(dO o O) in float32;
//   attn_bwd_kernel     one persistent CTA per SM over (head, 128-key block)
//                       units.  K_j, V_j stay in shared memory while the CTA
//                       walks the query blocks that see them (causal: from the
//                       diagonal on).  Per query block: S^T = K Q^T and
//                       dP^T = V dO^T on tcgen05 into TMEM; four warps (thread
//                       = key row = TMEM lane) form P^T = 2^(c S^T - lse log2 e)
//                       and dS^T = P^T o (dP^T - D), write both back into TMEM
//                       as 16-bit operands and dS into shared memory;
//                       dV += P^T dO and dK += dS^T Q accumulate in TMEM;
//                       dQ_i = dS K (queries on the TMEM lanes, so dS is read
//                       from shared memory as an M-major operand) lands in
//                       the S^T columns and is reduce-added (bulk tensor
//                       reduce from shared memory) into a float32 dQ
//                       accumulator; Q_i and dO_i are double-buffered so the
//                       next block loads during this one; at the end of the
//                       unit dV and scale dK
//                       are rounded and stored;
//   bwd_dq_kernel       dQ = scale * accumulator, rounded to the input type.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>
#include <mutex>
#include <type_traits>

#include "host_common.h"
#include "sm103.cuh"

namespace bwd {

using namespace sm103;

namespace {
__device__ unsigned int g_status_word = 0;
}

constexpr int kB = 128;  // keys per unit = queries per block = TMEM lanes

// Instruction descriptor (kind::f16, dense, float32 accumulator) with the
// transpose bits of both operands: a_mn / b_mn select an M-major A / N-major B.
__host__ __device__ constexpr uint32_t idesc(uint32_t fmt, int M, int N, uint32_t a_mn, uint32_t b_mn) {
  return (1u << 4) | (fmt << 7) | (fmt << 10) | (a_mn << 15) | (b_mn << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// 4-D tiled reduce-add (float32 add into global memory) from shared memory,
// bulk-group completion; elements of the box outside the tensor are skipped.
__device__ __forceinline__ void tma_reduce_add_4d(const CUtensorMap* map, uint32_t src, int x, int y, int z, int w) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.4d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(src), "r"(x), "r"(y), "r"(z), "r"(w)
      : "memory");
}

template <int D>
struct BCfg {
  static constexpr int CHUNK_BYTES = kB * 128;  // 128 rows x one 128-byte swizzle span (64 elements)
  static constexpr int CHUNKS = D * 2 / 128;
  static constexpr int TILE_BYTES = CHUNKS * CHUNK_BYTES;
  static constexpr int QD_STAGES = 2;               // Q_i, dO_i double-buffered
  // dS: 128 key rows x 128 queries, two 64-query spans; after the dQ product
  // has read it, the same bytes stage 64 float32 columns of the dQ partial
  // (two 32-column, 128-byte swizzled boxes) for the reduce-add into dQ.
  static constexpr int DS_BYTES = 2 * CHUNK_BYTES;
  static constexpr int OFF_K = 0, OFF_V = TILE_BYTES;
  static constexpr int OFF_Q = 2 * TILE_BYTES;                        // + stage * 2 * TILE_BYTES
  static constexpr int OFF_DO = 3 * TILE_BYTES;                       // + stage * 2 * TILE_BYTES
  static constexpr int OFF_DS = (2 + 2 * QD_STAGES) * TILE_BYTES;
  static constexpr int OFF_LSE = OFF_DS + DS_BYTES;  // 128 floats: lse * log2(e) of the query block
  static constexpr int OFF_D = OFF_LSE + 512;        // 128 floats: D of the query block
  static constexpr int OFF_BAR = OFF_D + 512;
  enum : int { B_KV_FULL = 0, B_KV_EMPTY, B_QD_FULL, B_QD_EMPTY = B_QD_FULL + QD_STAGES,
               B_SP_FULL = B_QD_EMPTY + QD_STAGES, B_P_READY, B_DQ_FULL, B_DQ_READ, B_EPI_DONE, B_ACC_FULL,
               B_MMA_DONE, NBARS };
  static constexpr int USED = OFF_BAR + 8 * NBARS + 16 + 1024;
  // One CTA per SM (TMEM is allocated whole): at least 115 KiB of shared memory.
  static constexpr int SMEM_BYTES = USED > 115 * 1024 ? USED : 115 * 1024;
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
  // TMEM columns: S^T (later P^T in its columns 0-31 and 96-127), dP^T (later
  // dS^T in the same columns of its own), dV, dK.  The dQ partial goes into
  // the columns the products do not read: d columns 0-63 at S^T + 32, 64-127
  // at dP^T + 32.
  static constexpr uint32_t TM_S = 0, TM_DP = 128, TM_DV = 256, TM_DK = 256 + D, TMEM_COLS = 512;
  static_assert(256 + 2 * D <= 512, "S^T, dP^T, dV and dK fit in TMEM");
  // Warps 0-7 compute (warp w: TMEM lanes 32 (w mod 4) .. + 31, column half
  // w / 4 of every 128-column pass), 8 load, 9 MMA.
  static constexpr int COMPUTE = 256;
  // Launched as 384 threads x 168 registers; the third warpgroup (load, MMA
  // and two idle warps) gives registers to the two compute warpgroups with
  // setmaxnreg: 2 x 128 x 200 + 128 x 88 = 62464 <= 384 x 168 = 64512.
  static constexpr int THREADS = COMPUTE + 128;
  static constexpr int LOAD_WARP = 8, MMA_WARP = 9;
  static constexpr int COMPUTE_REGS = 200, OTHER_REGS = 88;
};

struct BwdParams {
  const float* lse;   // [BH][N], natural log
  const float* dvec;  // [BH][N], D = rowsum(dO o O)
  float* dq_acc;      // [BH][N][d] float32, zero at launch
  void* dk;           // [BH][N][d], input type
  void* dv;
  int BH, N, causal;
  int nkb;            // 128-row blocks per head
  int num_units;      // BH * nkb
  float sl2;          // scale * log2(e)
  float scale;
  uint64_t timeout_ns;
};

// Unit u -> (head, key block).  Causal: key block 0 of every head first (it
// has the most query blocks), longest first; full: head-major.
__device__ __forceinline__ void decode(int u, const BwdParams& p, int& bh, int& j) {
  if (p.causal) {
    j = u / p.BH;
    bh = u - j * p.BH;
  } else {
    bh = u / p.nkb;
    j = u - bh * p.nkb;
  }
}

__device__ __forceinline__ int unit_of(int r) {
  const int G = gridDim.x, c = blockIdx.x;
  return r * G + ((r & 1) ? (G - 1 - c) : c);  // snake order over rounds
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack16(float lo, float hi) {
  if constexpr (BF16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

__device__ __forceinline__ bool drain(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > limit_ns) return false;
  return true;
}

template <int D, bool BF16>
__global__ void __launch_bounds__(BCfg<D>::THREADS, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                    const __grid_constant__ CUtensorMap tmDQ, const BwdParams p) {
  using C = BCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sK = smem_u32(smem + C::OFF_K), sV = smem_u32(smem + C::OFF_V);
  auto sQ = [&](uint32_t st) { return smem_u32(smem + C::OFF_Q + st * 2 * C::TILE_BYTES); };
  auto sDO = [&](uint32_t st) { return smem_u32(smem + C::OFF_DO + st * 2 * C::TILE_BYTES); };
  const uint32_t sDS = smem_u32(smem + C::OFF_DS);
  float* lse_s = reinterpret_cast<float*>(smem + C::OFF_LSE);
  float* d_s = reinterpret_cast<float*>(smem + C::OFF_D);
  const uint32_t bar0 = smem_u32(smem + C::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + 8 * C::NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  auto BAR = [&](int i) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(i); };
  const int warp = static_cast<int>(warp_id()), lane = static_cast<int>(lane_id());
  const int G = static_cast<int>(gridDim.x);

  if (threadIdx.x == 0) {
    for (int b = 0; b < C::NBARS; ++b)
      mbar_init(BAR(b), (b == C::B_P_READY || b == C::B_DQ_READ || b == C::B_EPI_DONE) ? C::COMPUTE / 32 : 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == C::MMA_WARP) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == C::LOAD_WARP && lane == 0) {
    tma_prefetch(&tmQ);
    tma_prefetch(&tmK);
    tma_prefetch(&tmV);
    tma_prefetch(&tmDO);
    tma_prefetch(&tmDQ);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtx wc{abort_flag, &g_status_word, p.timeout_ns};

  // The register budget changes inside each warpgroup's own branch, so that
  // the compiler allocates every role's code against its own budget.
  if (warp >= C::LOAD_WARP) {
  setmaxnreg_dec<C::OTHER_REGS>();
  if (warp == C::LOAD_WARP) {
    // ---------------------------------------------------------------- loads
    if (lane == 0) {
      uint32_t kv_it = 0, qd_it = 0;
      bool ok = true;
      // Tensor maps over [BH, N, d] (batch folded into heads): coordinates
      // (column, row, head, 0), 64 columns per 128-byte swizzle span.
      auto load_tile = [&](uint32_t dst, const CUtensorMap* map, uint32_t bar, int row, int bh) {
#pragma unroll
        for (int c = 0; c < C::CHUNKS; ++c) tma_load_4d(dst + c * C::CHUNK_BYTES, map, bar, c * 64, row, bh, 0);
      };
      for (int r = 0; ok && r * G < p.num_units; ++r) {
        const int u = unit_of(r);
        if (u >= p.num_units) continue;
        int bh, j;
        decode(u, p, bh, j);
        if (!(ok = mbar_wait(BAR(C::B_KV_EMPTY), (kv_it & 1u) ^ 1u, wc, attn_internal::kStatusTimeoutLoad))) break;
        ++kv_it;
        mbar_arrive_expect_tx(BAR(C::B_KV_FULL), 2 * C::TILE_BYTES);
        load_tile(sK, &tmK, BAR(C::B_KV_FULL), j * kB, bh);
        load_tile(sV, &tmV, BAR(C::B_KV_FULL), j * kB, bh);
        for (int i = p.causal ? j : 0; ok && i < p.nkb; ++i) {
          const uint32_t st = qd_it % C::QD_STAGES, ph = (qd_it / C::QD_STAGES) & 1u;
          if (!(ok = mbar_wait(BAR(C::B_QD_EMPTY + st), ph ^ 1u, wc, attn_internal::kStatusTimeoutLoad))) break;
          ++qd_it;
          mbar_arrive_expect_tx(BAR(C::B_QD_FULL + st), 2 * C::TILE_BYTES);
          load_tile(sQ(st), &tmQ, BAR(C::B_QD_FULL + st), i * kB, bh);
          load_tile(sDO(st), &tmDO, BAR(C::B_QD_FULL + st), i * kB, bh);
        }
      }
      // No copies in flight when the CTA leaves.
      if (kv_it > 0) drain(BAR(C::B_KV_FULL), (kv_it - 1) & 1u, 100000000ull);
      for (uint32_t k2 = 0; k2 < C::QD_STAGES && k2 < qd_it; ++k2) {
        const uint32_t f = qd_it - 1 - k2;
        drain(BAR(C::B_QD_FULL + f % C::QD_STAGES), (f / C::QD_STAGES) & 1u, 100000000ull);
      }
    }
  } else if (warp == C::MMA_WARP) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t fmt = BF16 ? 1u : 0u;
      constexpr uint32_t ID_T = idesc(fmt, kB, kB, 0, 0);   // S^T, dP^T: both operands K-major
      constexpr uint32_t ID_ACC = idesc(fmt, kB, D, 0, 1);  // dV, dK: A from TMEM, B N-major
      constexpr uint32_t ID_DQ = idesc(fmt, kB, 64, 1, 1);  // dQ, 64 columns at a time: A M-major, B N-major
      constexpr uint32_t HI = desc_sw128_hi(1024);
      uint32_t kv_it = 0, qd_it = 0, pr_it = 0, dqr_it = 0, epi_it = 0;
      bool ok = true, first_block = true;
      int units_done = 0;
      // A [128 x d] K-major times B [128 x d] K-major (contraction over d).
      auto mma_kmajor = [&](uint32_t d_tmem, uint32_t a_smem, uint32_t b_smem) {
        const uint32_t a0 = desc_sw128_lo(a_smem, 16), b0 = desc_sw128_lo(b_smem, 16);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * C::CHUNK_BYTES + (kk & 3) * 32) >> 4;
          mma_ss_w(d_tmem, a0 + off, HI, b0 + off, HI, ID_T, kk > 0 ? 1u : 0u, false);
        }
      };
      // D (+)= A[TMEM, 128 x 128] * B[128 x d N-major] (contraction over the 128 queries).
      auto mma_tmem_a = [&](uint32_t d_tmem, uint32_t a_tmem, uint32_t b_smem, bool acc) {
        const uint32_t b0 = desc_sw128_lo(b_smem, C::CHUNK_BYTES);
#pragma unroll
        for (int kk = 0; kk < kB / 16; ++kk)  // 16-bit columns 0..31 and 96..127 (queries 0..63, 64..127)
          mma_ts_w(d_tmem, a_tmem + kk * 8 + (kk >= kB / 32 ? 64 : 0), b0 + ((kk * 16 * 128) >> 4), HI, ID_ACC,
                   (acc || kk > 0) ? 1u : 0u, false);
      };
      for (int r = 0; ok && r * G < p.num_units; ++r) {
        const int u = unit_of(r);
        if (u >= p.num_units) continue;
        int bh, j;
        decode(u, p, bh, j);
        if (!(ok = mbar_wait(BAR(C::B_KV_FULL), kv_it & 1u, wc, attn_internal::kStatusTimeoutMma))) break;
        ++kv_it;
        tc_fence_after();
        const int i0 = p.causal ? j : 0;
        for (int i = i0; i < p.nkb; ++i) {
          const uint32_t st = qd_it % C::QD_STAGES;
          if (!(ok = mbar_wait(BAR(C::B_QD_FULL + st), (qd_it / C::QD_STAGES) & 1u, wc,
                               attn_internal::kStatusTimeoutMma)))
            break;
          ++qd_it;
          if (!first_block) {  // the previous dQ partial has left the S^T columns
            if (!(ok = mbar_wait(BAR(C::B_DQ_READ), dqr_it & 1u, wc, attn_internal::kStatusTimeoutMma))) break;
            ++dqr_it;
          }
          first_block = false;
          tc_fence_after();
          mma_kmajor(tmem + C::TM_S, sK, sQ(st));    // S^T = K Q^T
          mma_kmajor(tmem + C::TM_DP, sV, sDO(st));  // dP^T = V dO^T
          mma_commit(BAR(C::B_SP_FULL));
          if (!(ok = mbar_wait(BAR(C::B_P_READY), pr_it & 1u, wc, attn_internal::kStatusTimeoutMma))) break;
          ++pr_it;
          if (i == i0 && units_done > 0) {  // the previous unit's dV, dK have been read
            if (!(ok = mbar_wait(BAR(C::B_EPI_DONE), epi_it & 1u, wc, attn_internal::kStatusTimeoutMma))) break;
            ++epi_it;
          }
          tc_fence_after();
          {  // dQ_i = dS K first, into columns no product reads, so the compute
             // warps read it out while dV and dK are being accumulated
            const uint32_t a0 = desc_sw128_lo(sDS, C::CHUNK_BYTES);
#pragma unroll
            for (int hq = 0; hq < D / 64; ++hq) {
              const uint32_t b0 = desc_sw128_lo(sK + hq * C::CHUNK_BYTES, C::CHUNK_BYTES);
              const uint32_t dst = tmem + (hq ? C::TM_DP : C::TM_S) + 32;
#pragma unroll
              for (int kk = 0; kk < kB / 16; ++kk) {
                const uint32_t off = (kk * 16 * 128) >> 4;
                mma_ss_w(dst, a0 + off, HI, b0 + off, HI, ID_DQ, kk > 0 ? 1u : 0u, false);
              }
            }
          }
          mma_commit(BAR(C::B_DQ_FULL));
          mma_tmem_a(tmem + C::TM_DV, tmem + C::TM_S, sDO(st), i > i0);   // dV += P^T dO
          mma_tmem_a(tmem + C::TM_DK, tmem + C::TM_DP, sQ(st), i > i0);   // dK += dS^T Q
          mma_commit(BAR(C::B_QD_EMPTY + st));
        }
        if (!ok) break;
        mma_commit(BAR(C::B_ACC_FULL));  // dV, dK of this unit complete
        mma_commit(BAR(C::B_KV_EMPTY));
        ++units_done;
      }
      mma_commit(BAR(C::B_MMA_DONE));
      drain(BAR(C::B_MMA_DONE), 0, 100000000ull);
    }
  }
  } else {
    setmaxnreg_inc<C::COMPUTE_REGS>();
    // ------------------------------------------------ compute (8 warps, 256 threads)
    const int quad = warp & 3, half = warp >> 2;  // TMEM lane quadrant, column half
    const int row = quad * 32 + lane;  // TMEM lane: key row of S^T, dP^T, dV, dK; query row of dQ
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
    uint32_t sp_it = 0, dq_it = 0, acc_it = 0;
    bool ok = true;
    constexpr float kLog2e = 1.4426950408889634f;
    for (int r = 0; ok && r * G < p.num_units; ++r) {
      const int u = unit_of(r);
      if (u >= p.num_units) continue;
      int bh, j;
      decode(u, p, bh, j);
      const int key = j * kB + row;
      const size_t head = static_cast<size_t>(bh) * p.N;
      const int i0 = p.causal ? j : 0;
      // lse (log2 units; +inf past N, so that P = 0 there) and D of this
      // thread's row of the next query block, loaded one block ahead.
      auto fetch = [&](int i, float& l2, float& dd) {
        const int q = i * kB + row;
        const bool in = i < p.nkb && q < p.N;
        l2 = in ? p.lse[head + q] * kLog2e : INFINITY;
        dd = in ? p.dvec[head + q] : 0.f;
      };
      float next_l2, next_d;
      fetch(i0, next_l2, next_d);
      for (int i = i0; i < p.nkb; ++i) {
        // Stage this block's values for the four warps.  The dS buffer below
        // is also the staging of the last dQ reduce: it must have been read.
        // Every warp's dQ reduce-adds have read its staging box before dS
        // overwrites the buffer (the barrier below makes it CTA-wide).
        if (lane == 0) bulk_wait_read_all();
        __syncwarp();
        if (bar_red_or(1, C::COMPUTE, !ok)) { ok = false; break; }
        if (half == 0) {  // the first four warps stage the block's lse and D
          lse_s[row] = next_l2;
          d_s[row] = next_d;
        }
        bar_sync_n(1, C::COMPUTE);
        if (half == 0) fetch(i + 1, next_l2, next_d);
        if (!(ok = mbar_wait_warp(BAR(C::B_SP_FULL), sp_it & 1u, wc, attn_internal::kStatusTimeoutSoftmax))) {
          bar_red_or(2, C::COMPUTE, true);
          break;
        }
        ++sp_it;
        tc_fence_after();
        const bool diag = p.causal && i == j;
        // This warp's 64 queries: S^T and dP^T columns of two 32-query chunks
        // loaded under one wait; lse and D read four at a time.
        {
          const int c2 = half;
          uint32_t s[2][32], dp[2][32];
          tmem_ld32(lane_base + C::TM_S + 64 * c2, s[0]);
          tmem_ld32(lane_base + C::TM_S + 64 * c2 + 32, s[1]);
          tmem_ld32(lane_base + C::TM_DP + 64 * c2, dp[0]);
          tmem_ld32(lane_base + C::TM_DP + 64 * c2 + 32, dp[1]);
          tmem_wait_ld(s[0]);
          reg_pin(s[1]);
          reg_pin(dp[0]);
          reg_pin(dp[1]);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int c = 2 * c2 + h;  // 32-query chunk
            uint32_t pk[16], dk16[16];
#pragma unroll
            for (int t4 = 0; t4 < 8; ++t4) {
              const int qc = 32 * c + 4 * t4;
              const float4 l4 = *reinterpret_cast<const float4*>(lse_s + qc);
              const float4 d4 = *reinterpret_cast<const float4*>(d_s + qc);
              const float lv[4] = {l4.x, l4.y, l4.z, l4.w}, dv4[4] = {d4.x, d4.y, d4.z, d4.w};
              float pv[4], dsv[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                float pe = ex2(p.sl2 * __uint_as_float(s[h][4 * t4 + e]) - lv[e]);
                if (diag && row > qc + e) pe = 0.f;  // key row > query: masked
                pv[e] = pe;
                dsv[e] = pe * (__uint_as_float(dp[h][4 * t4 + e]) - dv4[e]);
              }
              pk[2 * t4] = pack16<BF16>(pv[0], pv[1]);
              pk[2 * t4 + 1] = pack16<BF16>(pv[2], pv[3]);
              dk16[2 * t4] = pack16<BF16>(dsv[0], dsv[1]);
              dk16[2 * t4 + 1] = pack16<BF16>(dsv[2], dsv[3]);
            }
            // The second half of the warps writes its 16-bit values into its own
            // loaded columns (96 .. 127), never into columns the first half may
            // still be reading; the products take that gap into account.
            tmem_st16(lane_base + C::TM_S + 16 * c + 64 * half, pk);
            tmem_st16(lane_base + C::TM_DP + 16 * c + 64 * half, dk16);
            // dS into shared memory: row `row`, queries 32c .. 32c + 31, 128-byte
            // swizzled spans of 64 queries (the layout a tiled copy would give).
            const uint32_t span = sDS + static_cast<uint32_t>(c >> 1) * C::CHUNK_BYTES + static_cast<uint32_t>(row) * 128u;
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              const uint32_t unit = static_cast<uint32_t>((c & 1) * 4 + v) ^ static_cast<uint32_t>(row & 7);
              st_shared_v4(span + (unit << 4), dk16[4 * v], dk16[4 * v + 1], dk16[4 * v + 2], dk16[4 * v + 3]);
            }
          }
        }
        tmem_wait_st();
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(C::B_P_READY));
        // dQ partial of this query block: TMEM lane = query row.
        const bool got = mbar_wait_warp(BAR(C::B_DQ_FULL), dq_it & 1u, wc, attn_internal::kStatusTimeoutSoftmax);
        if (bar_red_or(2, C::COMPUTE, !got)) { ok = false; break; }
        ++dq_it;
        tc_fence_after();
        // Each warp stages its 32 query rows x 32 columns of a round in its own
        // 4 KiB box of the dS buffer (free: the dQ product has read it; 128-byte
        // swizzled rows) and its lane 0 reduce-adds the box into the float32
        // accumulator (rows past N are skipped by the copy): no barrier across
        // warps, each warp waits only for its own previous copy.
        {
          const uint32_t box = sDS + static_cast<uint32_t>(warp) * 4096u + static_cast<uint32_t>(lane) * 128u;
#pragma unroll 1
          for (int rnd = 0; rnd < D / 64; ++rnd) {
            uint32_t v[32];
            tmem_ld32(lane_base + (rnd ? C::TM_DP : C::TM_S) + 32 + 32 * half, v);
            tmem_wait_ld(v);
            if (rnd > 0) {
              if (lane == 0) bulk_wait_read_all();
              __syncwarp();
            }
#pragma unroll
            for (int u4 = 0; u4 < 8; ++u4)
              st_shared_v4(box + ((static_cast<uint32_t>(u4) ^ static_cast<uint32_t>(lane & 7)) << 4), v[4 * u4],
                           v[4 * u4 + 1], v[4 * u4 + 2], v[4 * u4 + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_reduce_add_4d(&tmDQ, sDS + static_cast<uint32_t>(warp) * 4096u, 64 * rnd + 32 * half,
                                i * kB + quad * 32, bh, 0);
              bulk_commit_group();
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(C::B_DQ_READ));
      }
      if (!ok) break;
      // Unit epilogue: dV and scale * dK of this key block, once their last
      // products have completed.
      if (bar_red_or(2, C::COMPUTE, !mbar_wait_warp(BAR(C::B_ACC_FULL), acc_it & 1u, wc,
                                                     attn_internal::kStatusTimeoutSoftmax))) {
        ok = false;
        break;
      }
      ++acc_it;
      tc_fence_after();
      typedef typename std::conditional<BF16, __nv_bfloat16, __half>::type T;
      T* dv_row = static_cast<T*>(p.dv) + (head + key) * D;
      T* dk_row = static_cast<T*>(p.dk) + (head + key) * D;
#pragma unroll 1
      for (int c = half * (D / 64); c < (half + 1) * (D / 64); ++c) {
        uint32_t a[32], b[32];
        tmem_ld32(lane_base + C::TM_DV + 32 * c, a);
        tmem_ld32(lane_base + C::TM_DK + 32 * c, b);
        tmem_wait_ld(a);
        reg_pin(b);
        if (key < p.N) {
          uint32_t pa[16], pb[16];
#pragma unroll
          for (int t = 0; t < 16; ++t) {
            pa[t] = pack16<BF16>(__uint_as_float(a[2 * t]), __uint_as_float(a[2 * t + 1]));
            pb[t] = pack16<BF16>(__uint_as_float(b[2 * t]) * p.scale, __uint_as_float(b[2 * t + 1]) * p.scale);
          }
          uint4* dva = reinterpret_cast<uint4*>(dv_row + 32 * c);
          uint4* dka = reinterpret_cast<uint4*>(dk_row + 32 * c);
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            dva[t] = make_uint4(pa[4 * t], pa[4 * t + 1], pa[4 * t + 2], pa[4 * t + 3]);
            dka[t] = make_uint4(pb[4 * t], pb[4 * t + 1], pb[4 * t + 2], pb[4 * t + 3]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(C::B_EPI_DONE));
    }
  }

  // The reduce-adds of dQ must finish before the CTA exits.
  if (warp < C::LOAD_WARP && lane == 0) bulk_wait_all();  // each compute warp's own groups
  tc_fence_before();
  __syncthreads();
  if (warp == C::MMA_WARP) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// D = rowsum(dO o O) in float32: one warp per row, d / 32 elements per lane.
template <int D, bool BF16>
__global__ void bwd_rowdot_kernel(const void* o, const void* dout, float* dvec, int64_t rows) {
  typedef typename std::conditional<BF16, __nv_bfloat16, __half>::type T;
  const int64_t r = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  const T* a = static_cast<const T*>(o) + r * D;
  const T* b = static_cast<const T*>(dout) + r * D;
  float acc = 0.f;
#pragma unroll
  for (int k = 0; k < D / 32; ++k) acc = fmaf(static_cast<float>(a[lane + 32 * k]), static_cast<float>(b[lane + 32 * k]), acc);
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
  if (lane == 0) dvec[r] = acc;
}

// dQ = scale * accumulator, rounded to the input type.
template <bool BF16>
__global__ void bwd_dq_kernel(const float4* acc, void* dq, float scale, int64_t n4) {
  typedef typename std::conditional<BF16, __nv_bfloat162, __half2>::type T2;
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n4) return;
  const float4 a = acc[i];
  T2* out = static_cast<T2*>(dq) + 2 * i;
  if constexpr (BF16) {
    out[0] = __floats2bfloat162_rn(a.x * scale, a.y * scale);
    out[1] = __floats2bfloat162_rn(a.z * scale, a.w * scale);
  } else {
    out[0] = __floats2half2_rn(a.x * scale, a.y * scale);
    out[1] = __floats2half2_rn(a.z * scale, a.w * scale);
  }
}

inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

template <int D, bool BF16>
attn_status run(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                void* dq, void* dk, void* dv, int B, int H, int N, int causal, float scale, void* ws,
                cudaStream_t s) {
  using C = BCfg<D>;
  const int BH = B * H;
  const size_t rows = static_cast<size_t>(BH) * N;
  float* dq_acc = static_cast<float*>(ws);
  float* dvec = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + align256(rows * D * 4));
  cudaError_t e = cudaMemsetAsync(dq_acc, 0, rows * D * 4, s);
  if (e != cudaSuccess) return attn_internal::cuda_status(e);
  const unsigned rd_blocks = static_cast<unsigned>((rows + 7) / 8);
  bwd_rowdot_kernel<D, BF16><<<rd_blocks, 256, 0, s>>>(o, dout, dvec, static_cast<int64_t>(rows));
  if ((e = cudaGetLastError()) != cudaSuccess) return attn_internal::cuda_status(e);

  // Tensor maps over [BH, N, d] (B folded into H), box 64 elements x 128 rows, 128-byte swizzle.
  const CUtensorMapDataType dt = BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUtensorMap mq, mk, mv, mdo;
  auto encode = [&](CUtensorMap* m, const void* base) {
    const uint64_t dims[4] = {static_cast<uint64_t>(D), static_cast<uint64_t>(N), static_cast<uint64_t>(BH), 1};
    const uint64_t strides[3] = {D * 2ull, static_cast<uint64_t>(N) * D * 2, static_cast<uint64_t>(BH) * N * D * 2};
    const uint32_t box[4] = {64, kB, 1, 1};
    return attn_internal::encode_tmap_4d(m, dt, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
  };
  if (!encode(&mq, q) || !encode(&mk, k) || !encode(&mv, v) || !encode(&mdo, dout)) return ATTN_ERR_CUDA;
  CUtensorMap mdq;  // float32 accumulator [BH, N, d], box 32 floats x 32 rows (one compute warp's)
  {
    const uint64_t dims[4] = {static_cast<uint64_t>(D), static_cast<uint64_t>(N), static_cast<uint64_t>(BH), 1};
    const uint64_t strides[3] = {D * 4ull, static_cast<uint64_t>(N) * D * 4, static_cast<uint64_t>(BH) * N * D * 4};
    const uint32_t box[4] = {32, 32, 1, 1};
    if (!attn_internal::encode_tmap_4d(&mdq, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, dq_acc, dims, strides, box,
                                       CU_TENSOR_MAP_SWIZZLE_128B))
      return ATTN_ERR_CUDA;
  }

  static std::mutex mu;
  static int configured[64] = {0};
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return attn_internal::cuda_status(e);
  if (dev < 0 || dev >= 64) return ATTN_ERR_UNSUPPORTED;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!configured[dev]) {
      if ((e = cudaFuncSetAttribute(attn_bwd_kernel<D, BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    C::SMEM_BYTES)) != cudaSuccess)
        return attn_internal::cuda_status(e);
      configured[dev] = 1;
    }
  }
  BwdParams prm{};
  prm.lse = lse;
  prm.dvec = dvec;
  prm.dq_acc = dq_acc;
  prm.dk = dk;
  prm.dv = dv;
  prm.BH = BH;
  prm.N = N;
  prm.causal = causal ? 1 : 0;
  prm.nkb = (N + kB - 1) / kB;
  prm.num_units = BH * prm.nkb;
  prm.sl2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  prm.scale = scale;
  prm.timeout_ns = attn_internal::wait_timeout_ns();
  const int sms = attn_internal::sm_count();
  if (sms <= 0) return ATTN_ERR_CUDA;
  const int grid = prm.num_units < sms ? prm.num_units : sms;
  attn_bwd_kernel<D, BF16><<<grid, C::THREADS, C::SMEM_BYTES, s>>>(mq, mk, mv, mdo, mdq, prm);
  if ((e = cudaGetLastError()) != cudaSuccess) return attn_internal::cuda_status(e);
  const int64_t n4 = static_cast<int64_t>(rows) * D / 4;
  bwd_dq_kernel<BF16><<<static_cast<unsigned>((n4 + 255) / 256), 256, 0, s>>>(
      reinterpret_cast<const float4*>(dq_acc), dq, scale, n4);
  return attn_internal::cuda_status(cudaGetLastError());
}

}  // namespace bwd

namespace attn_internal {
cudaError_t bwd_status_exchange(unsigned int* out) {
  cudaError_t e = cudaMemcpyFromSymbol(out, bwd::g_status_word, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(bwd::g_status_word, &zero, sizeof(unsigned int));
}
}  // namespace attn_internal

ATTN_EXPORT size_t attn_bwd_workspace_bytes(int B, int H, int N, int d) {
  if (B < 0 || H < 0 || N < 0 || (d != 64 && d != 128)) return 0;
  const size_t rows = static_cast<size_t>(B) * H * N;
  return bwd::align256(rows * d * 4) + bwd::align256(rows * 4);
}

ATTN_EXPORT attn_status attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                                 const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                                 int causal, float scale, attn_dtype dtype, void* workspace, size_t workspace_bytes,
                                 void* stream) {
  if (B < 0 || H < 0 || N < 0) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_FP16 && dtype != ATTN_BF16) return ATTN_ERR_UNSUPPORTED;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(B) * H * ((N + bwd::kB - 1) / bwd::kB) > 0x7fffffff) return ATTN_ERR_INVALID_ARG;
  if (static_cast<int64_t>(B) * H * N == 0) return ATTN_OK;
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv || !workspace) return ATTN_ERR_INVALID_ARG;
  using attn_internal::aligned;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(dout, 16) ||
      !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) || !aligned(lse, 4))
    return ATTN_ERR_MISALIGNED;
  if (!aligned(workspace, 256)) return ATTN_ERR_MISALIGNED;
  if (workspace_bytes < attn_bwd_workspace_bytes(B, H, N, d)) return ATTN_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool bf = dtype == ATTN_BF16;
  if (d == 64)
    return bf ? bwd::run<64, true>(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, causal, scale, workspace, s)
              : bwd::run<64, false>(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, causal, scale, workspace, s);
  return bf ? bwd::run<128, true>(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, causal, scale, workspace, s)
            : bwd::run<128, false>(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, causal, scale, workspace, s);
}
