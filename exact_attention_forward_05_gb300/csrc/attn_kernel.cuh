// attn_kernel.cuh -- the fused exact attention forward kernel for GB300
// (sm_103a), templated on the head dimension and on the operand kind
// (fp16, bf16, or FP8 E4M3 with per-block scales).
//
// One persistent CTA per SM walks a static list of work units.  A unit is one
// (batch*head, block of query rows) pair: two 128-row Q tiles for d <= 128,
// one for d = 256.  Inside a CTA the warps specialise:
//
//   softmax group t (4 warps per Q tile): thread = one query row = one TMEM
//       lane.  Loads its row of S from TMEM, runs the online softmax, writes P
//       back over S, rescales O when needed, and at the end divides O by the
//       running sum and writes O (through shared memory and a bulk tensor
//       store) and lse.
//   load warp: TMA loads of Q (once per unit) and of K_j / V_j blocks into a
//       ring of shared-memory stages guarded by mbarriers (two Q tiles: K_j and
//       V_{j-1} share one ring slot with one full and one empty barrier).
//   MMA warp: one thread issues tcgen05.mma: S = Q K_j^T (both operands in
//       shared memory) and O += P V_j (P read from TMEM, V from shared memory),
//       accumulating in TMEM, and signals completion with tcgen05.commit.
//       Every instruction of this thread is on the critical path (one
//       tcgen05.mma takes about as long to issue as a 128x128x16 product takes
//       to run), so its waits, commits and descriptor arithmetic are kept few.
// Two Q tiles: 12 warps = 3 warpgroups; the third (load, MMA, 2 idle warps)
// hands registers to the two softmax warpgroups with setmaxnreg.
//
// The pages' method: tiles of Q, K, V moved to on-chip memory, the softmax
// computed blockwise with a running maximum and a separately tracked running
// denominator, the normalisation deferred to the end ("FlashAttention -- one,
// two, three!", sections "FlashAttention v1." and "FlashAttention v2."), the
// softmax of one tile overlapped with the matrix products of another, and
// asynchronous copies overlapped with compute ("Overlapping GEMM and Softmax
// (Asynchrony)" on the FlashAttention-3 podcast page; comrad404 review,
// "Метод", items 1 and 2).  The Hopper ping-pong between two warpgroups is
// re-expressed for tcgen05: the single MMA issuer alternates between the two Q
// tiles, so one tile's softmax runs while the other tile's products run.
//
// Online softmax, base 2 with c = scale * log2(e):
//   m_blk = c * rowmax(S_j)           (rowmin when c < 0)
//   if m_blk > m + 8: O *= 2^(m - m_blk), l *= 2^(m - m_blk), m = m_blk
//   P_j = 2^(c S_j - m),  l += rowsum(P_j),  O += P_j V_j
//   O /= l at the end,  lse = (m + log2 l) * ln 2.
// Keeping a stale m while the block maximum stays within 2^8 of it is exact:
// O and l carry the same factor 2^-m, which cancels in O / l and is added back
// in lse; P stays below 2^8, far from overflow in any operand format.
//
// FP8 operands (block quantisation, comrad404 review "Метод" item 3): the
// kernel reads E4M3 codes and float32 scales, one per 128 rows of a head.  The
// true logit is scale * sq * sk_j * (Q8 K8_j^T), so the per-block multiplier
// c_j = c * sq * sk_j replaces c.  The V block scale enters through P: the
// stored weights are P'_j = P_j * sv_j / svmax (svmax = the largest V scale of
// the head, so P' <= P), l still sums P_j, and O is multiplied by svmax at
// the end.  In real arithmetic this is the same result; only the rounding
// point of P moves.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <cmath>
#include <type_traits>

#include "host_common.h"
#include "sm103.cuh"

namespace attn_kernel {

using namespace sm103;

// Each translation unit that includes this header owns one status word.
namespace {
__device__ unsigned int g_status_word = 0;
}

enum Kind : int { KIND_F16 = 0, KIND_BF16 = 1, KIND_E4M3 = 2 };

constexpr int kBM = 128;  // query rows per Q tile (= TMEM lanes)
constexpr int kBN = 128;  // keys per K/V block
constexpr float kRescaleThreshold = 8.0f;

// Most CTAs whose stream-K ranges share one unit: the host cuts at least
// half a unit's key blocks per CTA, so a unit meets at most three ranges.
constexpr int kMaxParts = 3;

#ifndef ATTN_FP8_POLY_QUADS
#define ATTN_FP8_POLY_QUADS 0
#endif

template <int D, int KIND>
struct Cfg {
  static constexpr int ELEM = KIND == KIND_E4M3 ? 1 : 2;  // operand bytes
  static constexpr int NQ = D <= 128 ? 2 : 1;              // Q tiles per unit
  static constexpr int ROW_BYTES = D * ELEM;
  // Swizzle span: 128 bytes, or 64 for the 64-byte rows of E4M3 at d = 64.
  static constexpr int SW = ROW_BYTES >= 128 ? 128 : 64;
  static constexpr int CHUNK_BYTES = kBM * SW;  // 128 rows x one swizzle span
  static constexpr int CHUNK_ELEMS = SW / ELEM;
  static constexpr int CHUNKS = ROW_BYTES / SW;
  static constexpr int TILE_BYTES = CHUNKS * CHUNK_BYTES;
  static constexpr int K_PER_SPAN = SW / 32;     // MMA K steps (32 bytes each) per swizzle span
  static constexpr int KSTEP = 32 / ELEM;       // K elements per MMA instruction
  static constexpr int QK_STEPS = D / KSTEP;
  static constexpr int PV_STEPS = kBN / KSTEP;
  static constexpr int P_COLS = kBN * ELEM / 4;  // TMEM columns holding one row of P
  static constexpr int STAGES = KIND == KIND_E4M3 ? (D == 64 ? 12 : (D == 128 ? 8 : 4))
                                                 : (D == 64 ? 6 : (D == 128 ? 4 : 2));
  // E4M3 weights: quadruples out of every 8 (32 keys) whose 2^x runs on the
  // FMA pipe instead of the multi-function unit (unmasked blocks only).
  static constexpr int POLY_QUADS = KIND == KIND_E4M3 ? ATTN_FP8_POLY_QUADS : 0;
  static_assert(POLY_QUADS >= 0 && POLY_QUADS <= 8, "quadruples per 32-key chunk");
  // Two Q tiles: the stages form pairs, one per key-block step j holding K_j
  // and V_{j-1} (consumed and released together), with one full and one
  // empty barrier per pair.  One Q tile: single-tile stages.
  static constexpr bool KV_PAIRS = NQ == 2;
  static constexpr int RING = KV_PAIRS ? STAGES / 2 : STAGES;
  static constexpr int SOFTMAX_WARPS = 4 * NQ;
  // Two Q tiles: the products P_{j-1} V_{j-1} signal nothing of their own;
  // the softmax learns of their completion from the S_FULL commit of the next
  // Q K^T, which is issued after them (only the tile's last product signals
  // O_DONE), which saves the MMA-issuing thread two commits per key block.
  static constexpr bool LAST_O_DONE_ONLY = NQ == 2;
  static constexpr int LOAD_WARP = SOFTMAX_WARPS;
  static constexpr int MMA_WARP = SOFTMAX_WARPS + 1;
  // Two Q tiles: three whole warpgroups (softmax, softmax, load + MMA + two
  // idle warps), so that the softmax warpgroups can take registers from the
  // third one with setmaxnreg: 2 x 128 x 208 + 128 x 88 = 384 x 168, the
  // registers the CTA is launched with.  One Q tile: six warps, no split.
  static constexpr bool REG_SPLIT = NQ == 2;
  static constexpr int SOFTMAX_REGS = 208, OTHER_REGS = 88;
  static constexpr int THREADS = REG_SPLIT ? 384 : 32 * (SOFTMAX_WARPS + 2);
  static_assert(!REG_SPLIT || 2 * 128 * SOFTMAX_REGS + 128 * OTHER_REGS <= THREADS * 168,
                "register split exceeds the launch allocation");
  // TMEM columns: two S buffers, then the O accumulator(s).
  static constexpr uint32_t TM_S0 = 0, TM_S1 = 128, TM_O0 = 256, TM_O1 = 256 + D;
  static constexpr uint32_t TMEM_COLS = 512;
  // Barrier indices.
  static constexpr int B_Q_FULL = 0, B_Q_EMPTY = 1, B_KV_FULL = 2, B_KV_EMPTY = 2 + STAGES,
                       B_S_FULL = 2 + 2 * STAGES, B_P_FULL = B_S_FULL + 2,
                       B_O_DONE = B_P_FULL + 2, B_MMA_DONE = B_O_DONE + 2, NBARS = B_MMA_DONE + 1;
  // Shared memory layout (offsets from a 1024-byte aligned base).
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_KV = NQ * TILE_BYTES;
  // O staging for the bulk tensor store: per Q tile one 128-byte column span
  // of the 16-bit output (128 rows x 64 columns), 128-byte swizzled.
  static constexpr int OST_BYTES = kBM * 128;
  static constexpr int OFF_OST = OFF_KV + STAGES * TILE_BYTES;
  static constexpr int OFF_BAR = OFF_OST + NQ * OST_BYTES;
  // After the barriers: TMEM address, abort flag, two last-part flags, then
  // the stream-K segment list.
  static constexpr int OFF_SEGS = OFF_BAR + 8 * NBARS + 16;
  static constexpr int SMEM_BYTES = OFF_SEGS + 64 + 1024;
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
  static_assert(SMEM_BYTES > 114 * 1024, "one CTA per SM (TMEM is allocated whole)");
  static_assert(ROW_BYTES % SW == 0, "rows span whole swizzle spans");
};

struct FwdParams {
  void* o;
  float* lse;
  int BH, N;      // N: query rows per head
  int Nk;         // keys per head
  int H;          // heads: unit head index bh = b * H + h
  int layout;     // ATTN_LAYOUT_BHND or ATTN_LAYOUT_BNHD, of q, k, v and o
  int causal;
  int causal_off; // causal: query i sees keys j <= i + causal_off (>= 0)
  float sl2;  // scale * log2(e)
  int units_per_head;
  int num_units;   // work entries: [0, full_units) whole units, then half units
  int full_units;
  uint64_t timeout_ns;
  // FP8 only: scales, element (bh, block) at [bh * bh_stride + block * blk_stride].
  const float* q_scale;
  const float* k_scale;
  const float* v_scale;
  int scale_bh_stride, scale_blk_stride;
  // Stream-K tail (full attention, two Q tiles, with a workspace): units
  // [0, sk_unit0) run round-robin in whole rounds; the (unit, key block)
  // steps of the rest are cut into gridDim.x equal contiguous ranges, one per
  // CTA, so every CTA ends after the same number of key blocks.  A unit cut between CTAs is done in parts: every part writes its
  // unnormalised O, running maximum m and sum l to its slot in the workspace,
  // and the last part to finish (an arrival counter per unit tile) combines
  // them and writes O and lse.  CTA c owns slots 2c (the unit its range
  // starts in) and 2c + 1 (the unit it ends in), and the counter pair of the
  // unit its range starts in.
  int stream_k;         // 0 = round-robin units
  int sk_unit0;         // stream-K: first unit of the tail cut into ranges
  float* ws_o;          // [slot][tile][d/4][128 rows][4] float
  float* ws_ml;         // [slot][tile][m | l][128 rows] float
  unsigned int* ws_cnt; // [cta][tile] arrivals, zero at launch
};

struct Unit {
  int bh, m0, nkb;
  int nb[2];  // key blocks visited by each Q tile: [jb, nb[t]) (nb[t] = 0: tile inactive)
  int jb;     // first key block (0 unless a stream-K part)
  int u;      // unit index
  bool part;  // stream-K: only some of the unit's key blocks
};

// Tensor maps are 4-D over the operand as it lies in memory: [B, H, N, d] as
// {d, N, H, B}, [B, N, H, d] as {d, H, N, B}.  A tile is 128 rows of one head
// either way and lands in shared memory the same way; only the order of the
// row and head coordinates differs.
__device__ __forceinline__ void tma_load_rows(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x,
                                              int row, int b, int h, bool bnhd) {
  tma_load_4d(dst, map, bar, x, bnhd ? h : row, bnhd ? row : h, b);
}
__device__ __forceinline__ void tma_store_rows(const CUtensorMap* map, uint32_t src, int x, int row, int b,
                                               int h, bool bnhd) {
  tma_store_4d(map, src, x, bnhd ? h : row, bnhd ? row : h, b);
}

// Unit order: causal units longest-first (highest query block first, all heads
// of one query block together); full attention head-major so that CTAs that
// run at the same time share K/V through L2.  Entries from full_units on are
// half units: the two Q tiles of one of the last units, one entry each, so that
// a short last round of the persistent schedule costs half a unit.
template <int NQ>
__device__ __forceinline__ Unit decode_unit(int e, const FwdParams& p) {
  Unit w;
  int u = e, half = -1;
  w.jb = 0;
  w.part = false;
  if (e >= p.full_units) {
    u = p.full_units + (e - p.full_units) / 2;
    half = (e - p.full_units) & 1;
  }
  w.u = u;
  int qu;
  if (p.causal) {
    qu = p.units_per_head - 1 - u / p.BH;
    w.bh = u % p.BH;
  } else {
    w.bh = u / p.units_per_head;
    qu = u % p.units_per_head;
  }
  w.m0 = qu * kBM * NQ + (half > 0 ? kBM : 0);
  w.nkb = (p.Nk + kBN - 1) / kBN;
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int r0 = w.m0 + kBM * t;
    if (t >= NQ || r0 >= p.N || (half >= 0 && t > 0))
      w.nb[t] = 0;
    else
      w.nb[t] = p.causal ? min(w.nkb, (r0 + kBM - 1 + p.causal_off) / kBN + 1) : w.nkb;
  }
  return w;
}

// Static persistent schedule, snake order across rounds so that the
// longest-first causal list spreads evenly over the CTAs.
__device__ __forceinline__ int unit_of_round(int r, int num_units) {
  const int G = gridDim.x, c = blockIdx.x;
  const int u = r * G + ((r & 1) ? (G - 1 - c) : c);
  return u < num_units ? u : -1;
}

// Stream-K part of the schedule: the (unit x key block) steps of units
// [sk_unit0, num_units), cut into gridDim.x equal contiguous ranges.
struct SkSpan {
  int64_t base, total;  // first step, number of steps
  __device__ __forceinline__ SkSpan(const FwdParams& p, int nkb)
      : base(static_cast<int64_t>(p.sk_unit0) * nkb), total(static_cast<int64_t>(p.num_units - p.sk_unit0) * nkb) {}
  // First step of CTA c's range.
  __device__ __forceinline__ int64_t begin(int c) const {
    return base + total * c / static_cast<int64_t>(gridDim.x);
  }
  // The CTA whose range holds step `pos`.
  __device__ __forceinline__ int cta_of(int64_t pos) const {
    const int G = static_cast<int>(gridDim.x);
    int c = static_cast<int>((pos - base) * G / total);
    while (c + 1 < G && begin(c + 1) <= pos) ++c;
    while (c > 0 && begin(c) > pos) --c;
    return c;
  }
  // Workspace slot of CTA c's part of unit u: 2c for the unit its range
  // starts in, 2c + 1 for the unit it ends in.
  __device__ __forceinline__ int slot(int c, int u, int nkb) const {
    return 2 * c + (static_cast<int64_t>(u) != begin(c) / nkb ? 1 : 0);
  }
};

// Stream-K segments of one CTA (at most kMaxSegs: its range holds less than
// 1.5 units' key blocks): unit, first and end key block.  Computed once per
// CTA by one thread into shared memory, so that the roles iterating over them
// keep only an index in registers.
constexpr int kMaxSegs = 3;
struct SkSegs {
  int n;
  int u[kMaxSegs], jb[kMaxSegs], je[kMaxSegs];
};
__device__ __forceinline__ void sk_segments(const FwdParams& p, SkSegs* out) {
  const int nkb = (p.Nk + kBN - 1) / kBN;
  const SkSpan sk(p, nkb);
  int64_t pos = sk.begin(blockIdx.x);
  const int64_t end = sk.begin(blockIdx.x + 1);
  int n = 0;
  while (pos < end && n < kMaxSegs) {
    const int u = static_cast<int>(pos / nkb);
    const int jb = static_cast<int>(pos - static_cast<int64_t>(u) * nkb);
    const int je = static_cast<int>(min(static_cast<int64_t>(nkb), jb + (end - pos)));
    out->u[n] = u;
    out->jb[n] = jb;
    out->je[n] = je;
    ++n;
    pos += je - jb;
  }
  out->n = n;
}

// The work of one CTA, the same sequence for every role: whole units in
// persistent round-robin (snake) order -- units [0, sk_unit0) when the
// stream-K tail is on -- then, with it, the CTA's stream-K segments.
struct WorkIter {
  int r = 0, seg = 0;
  template <int NQ>
  __device__ __forceinline__ bool next(Unit& w, const FwdParams& p, const SkSegs* segs) {
    const int rr_units = p.stream_k ? p.sk_unit0 : p.num_units;
    while (r * static_cast<int>(gridDim.x) < rr_units) {
      const int u = unit_of_round(r++, rr_units);
      if (u < 0) continue;
      w = decode_unit<NQ>(u, p);
      return true;
    }
    if (!p.stream_k || seg >= segs->n) return false;
    const int je = segs->je[seg];
    w = decode_unit<NQ>(segs->u[seg], p);
    if (w.nb[0] > 0) w.nb[0] = je;
    if (w.nb[1] > 0) w.nb[1] = je;
    w.jb = segs->jb[seg];
    w.part = w.jb > 0 || je < w.nkb;
    ++seg;
    return true;
  }
};

// Two weights -> one 32-bit TMEM column of 16-bit P (first key in the low half).
template <int KIND>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (KIND == KIND_F16) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

// Four weights -> one 32-bit TMEM column of E4M3 P (first key in byte 0).
__device__ __forceinline__ uint32_t pack4_e4m3(float a, float b, float c, float d) {
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return lo | (hi << 16);
}

__device__ __forceinline__ bool mbar_drain(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > limit_ns) return false;
  return true;
}

template <int D, int KIND>
__global__ void __launch_bounds__(Cfg<D, KIND>::THREADS, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                    const FwdParams p) {
  using C = Cfg<D, KIND>;
  constexpr int NQ = C::NQ;
  constexpr bool F8 = KIND == KIND_E4M3;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);

  const uint32_t sQ = smem_u32(smem + C::OFF_Q);
  const uint32_t sKV = smem_u32(smem + C::OFF_KV);
  const uint32_t bar0 = smem_u32(smem + C::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + 8 * C::NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  auto BAR = [&](int i) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(i); };

  const int warp = static_cast<int>(warp_id());
  const int lane = static_cast<int>(lane_id());
  SkSegs* segs = reinterpret_cast<SkSegs*>(smem + C::OFF_SEGS);
  static_assert(sizeof(SkSegs) <= 64, "segment list space");

  if (threadIdx.x == 0) {
    if (p.stream_k) sk_segments(p, segs);
    else segs->n = 0;
    mbar_init(BAR(C::B_Q_FULL), 1);
    mbar_init(BAR(C::B_Q_EMPTY), 1);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(BAR(C::B_KV_FULL + s), 1);
      mbar_init(BAR(C::B_KV_EMPTY + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(BAR(C::B_S_FULL + b), 1);
      mbar_init(BAR(C::B_P_FULL + b), 4);
      mbar_init(BAR(C::B_O_DONE + b), 1);
    }
    mbar_init(BAR(C::B_MMA_DONE), 1);
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
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // The register budget changes inside each warpgroup's own branch, so that
  // the compiler allocates every role's code against its own budget.
  if (warp >= C::SOFTMAX_WARPS) {
  if constexpr (C::REG_SPLIT) setmaxnreg_dec<C::OTHER_REGS>();
  if (warp == C::LOAD_WARP) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const WaitCtx wc{abort_flag, &g_status_word, p.timeout_ns};
      uint32_t kv_fill = 0, q_iter = 0;
      bool ok = true;
      const bool bnhd = p.layout == ATTN_LAYOUT_BNHD;
      auto load_block = [&](const CUtensorMap* map, int j, int ub, int uh) -> bool {
        const uint32_t s = kv_fill % C::STAGES;
        const uint32_t ph = (kv_fill / C::STAGES) & 1u;
        if (!mbar_wait(BAR(C::B_KV_EMPTY + s), ph ^ 1u, wc, attn_internal::kStatusTimeoutLoad))
          return false;
        mbar_arrive_expect_tx(BAR(C::B_KV_FULL + s), C::TILE_BYTES);
#pragma unroll
        for (int c = 0; c < C::CHUNKS; ++c)
          tma_load_rows(sKV + s * C::TILE_BYTES + c * C::CHUNK_BYTES, map, BAR(C::B_KV_FULL + s),
                        c * C::CHUNK_ELEMS, j * kBN, ub, uh, bnhd);
        ++kv_fill;
        return true;
      };
      // Pair slot s holds K_j in tile 2s and V_{j-1} in tile 2s+1 (either may
      // be absent at the ends of a unit: step jb has no V, step nbmax no K).
      auto load_pair = [&](int j, int jb, int nbmax, int ub, int uh) -> bool {
        const uint32_t s = kv_fill % C::RING;
        const uint32_t ph = (kv_fill / C::RING) & 1u;
        if (!mbar_wait(BAR(C::B_KV_EMPTY + s), ph ^ 1u, wc, attn_internal::kStatusTimeoutLoad))
          return false;
        const bool has_k = j < nbmax, has_v = j > jb;
        mbar_arrive_expect_tx(BAR(C::B_KV_FULL + s), (has_k + has_v) * C::TILE_BYTES);
#pragma unroll
        for (int c = 0; c < C::CHUNKS; ++c) {
          if (has_k)
            tma_load_rows(sKV + (2 * s) * C::TILE_BYTES + c * C::CHUNK_BYTES, &tmK,
                          BAR(C::B_KV_FULL + s), c * C::CHUNK_ELEMS, j * kBN, ub, uh, bnhd);
          if (has_v)
            tma_load_rows(sKV + (2 * s + 1) * C::TILE_BYTES + c * C::CHUNK_BYTES, &tmV,
                          BAR(C::B_KV_FULL + s), c * C::CHUNK_ELEMS, (j - 1) * kBN, ub, uh, bnhd);
        }
        ++kv_fill;
        return true;
      };
      WorkIter wi;
      for (Unit w; ok && wi.next<NQ>(w, p, segs);) {
        const int nbmax = max(w.nb[0], w.nb[1]);
        if (nbmax == 0) continue;  // no query row of this entry is below N
        const int ub = w.bh / p.H, uh = w.bh - ub * p.H;
        if (!mbar_wait(BAR(C::B_Q_EMPTY), (q_iter & 1u) ^ 1u, wc, attn_internal::kStatusTimeoutLoad)) {
          ok = false;
          break;
        }
        ++q_iter;
        const int nact = (w.nb[0] > 0) + (NQ == 2 && w.nb[1] > 0);
        mbar_arrive_expect_tx(BAR(C::B_Q_FULL), nact * C::TILE_BYTES);
        for (int t = 0; t < NQ; ++t) {
          if (w.nb[t] == 0) continue;
#pragma unroll
          for (int c = 0; c < C::CHUNKS; ++c)
            tma_load_rows(sQ + t * C::TILE_BYTES + c * C::CHUNK_BYTES, &tmQ, BAR(C::B_Q_FULL),
                          c * C::CHUNK_ELEMS, w.m0 + kBM * t, ub, uh, bnhd);
        }
        // K/V in the order the MMA warp consumes them: K_0, then (K_j, V_{j-1}).
        const int jb = w.jb;
        for (int j = jb; j <= nbmax && ok; ++j) {
          if constexpr (C::KV_PAIRS) {
            ok = load_pair(j, jb, nbmax, ub, uh);
          } else {
            if (j < nbmax) ok = load_block(&tmK, j, ub, uh);
            if (ok && j >= 1) ok = load_block(&tmV, j - 1, ub, uh);
          }
        }
      }
      // Never leave the CTA with copies in flight: wait for the last fill of
      // every ring slot and of Q (already complete on the normal path).
      for (uint32_t i = 0; i < C::RING && i < kv_fill; ++i) {
        const uint32_t f = kv_fill - 1 - i;
        mbar_drain(BAR(C::B_KV_FULL + f % C::RING), (f / C::RING) & 1u, 100000000ull);
      }
      if (q_iter > 0) mbar_drain(BAR(C::B_Q_FULL), (q_iter - 1) & 1u, 100000000ull);
    }
  } else if (warp == C::MMA_WARP) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const WaitCtx wc{abort_flag, &g_status_word, p.timeout_ns};
      // kind::f16: 0 = F16, 1 = BF16; kind::f8f6f4: 0 = E4M3.
      constexpr uint32_t fmt = KIND == KIND_BF16 ? 1u : 0u;
      constexpr uint32_t IDESC_QK = instr_desc(fmt, fmt, kBM, kBN, 0);
      constexpr uint32_t IDESC_PV = instr_desc(fmt, fmt, kBM, D, 1);
      uint32_t kv_use = 0, q_iter = 0;
      uint32_t pph = 0u;  // bit b: wait parity of P_FULL[b]
      bool ok = true;

      auto next_stage = [&](uint32_t& slot) -> bool {
        slot = kv_use % C::STAGES;
        const uint32_t ph = (kv_use / C::STAGES) & 1u;
        ++kv_use;
        if (!mbar_wait(BAR(C::B_KV_FULL + slot), ph, wc, attn_internal::kStatusTimeoutMma)) return false;
        tc_fence_after();
        return true;
      };
      // S[sbuf] = Q[qt] K^T   (K-major A and B, 128-byte swizzle; 32 bytes of K per MMA)
      // Descriptors: base low word once per call, a constant offset per product.
      // 8-row groups of SW-byte rows: stride 8 * SW bytes.
      constexpr uint32_t DESC_HI = C::SW == 128 ? desc_sw128_hi(1024) : desc_sw64_hi(512);
      auto issue_qk = [&](int qt, int sbuf, uint32_t kslot) {
        const uint32_t d_tmem = tmem + (sbuf ? C::TM_S1 : C::TM_S0);
        const uint32_t a0 = desc_sw128_lo(sQ + qt * C::TILE_BYTES, 16);
        const uint32_t b0 = desc_sw128_lo(sKV + kslot * C::TILE_BYTES, 16);
#pragma unroll
        for (int kk = 0; kk < C::QK_STEPS; ++kk) {
          const uint32_t off = ((kk / C::K_PER_SPAN) * C::CHUNK_BYTES + (kk % C::K_PER_SPAN) * 32) >> 4;
          mma_ss_w(d_tmem, a0 + off, DESC_HI, b0 + off, DESC_HI, IDESC_QK, kk > 0 ? 1u : 0u, F8);
        }
      };
      // O[ot] (+)= P[sbuf] V   (P from TMEM, V N-major in shared memory; 32 bytes of keys per MMA)
      auto issue_pv = [&](int ot, int sbuf, uint32_t vslot, bool acc) {
        const uint32_t d_tmem = tmem + (ot ? C::TM_O1 : C::TM_O0);
        const uint32_t a_tmem = tmem + (sbuf ? C::TM_S1 : C::TM_S0);
        const uint32_t b0 = desc_sw128_lo(sKV + vslot * C::TILE_BYTES, C::CHUNK_BYTES);
#pragma unroll
        for (int kk = 0; kk < C::PV_STEPS; ++kk) {
          mma_ts_w(d_tmem, a_tmem + kk * 8, b0 + ((kk * C::KSTEP * C::SW) >> 4), DESC_HI, IDESC_PV,
                   (acc || kk > 0) ? 1u : 0u, F8);
        }
      };
      auto wait_p = [&](int b) -> bool {
        if (!mbar_wait(BAR(C::B_P_FULL + b), (pph >> b) & 1u, wc, attn_internal::kStatusTimeoutMma)) return false;
        pph ^= 1u << b;
        tc_fence_after();
        return true;
      };

      WorkIter wi;
      for (Unit w; ok && wi.next<NQ>(w, p, segs);) {
        const int nbmax = max(w.nb[0], w.nb[1]);
        if (nbmax == 0) continue;
        if (!mbar_wait(BAR(C::B_Q_FULL), q_iter & 1u, wc, attn_internal::kStatusTimeoutMma)) { ok = false; break; }
        ++q_iter;
        tc_fence_after();
        uint32_t ks = 0, vs = 0;
        if constexpr (NQ == 2) {
          // One wait and one release per key-block step: pair slot ps holds
          // K_j (tile 2 ps) and V_{j-1} (tile 2 ps + 1).
          auto next_pair = [&](uint32_t& slot) -> bool {
            slot = kv_use % C::RING;
            const uint32_t ph = (kv_use / C::RING) & 1u;
            ++kv_use;
            if (!mbar_wait(BAR(C::B_KV_FULL + slot), ph, wc, attn_internal::kStatusTimeoutMma)) return false;
            tc_fence_after();
            return true;
          };
          uint32_t ps = 0;
          if (!(ok = next_pair(ps))) break;
          for (int t = 0; t < 2; ++t)
            if (w.nb[t] > 0) {
              issue_qk(t, t, 2 * ps);
              mma_commit(BAR(C::B_S_FULL + t));
            }
          mma_commit(BAR(C::B_KV_EMPTY + ps));
          const int jb = w.jb, nb0 = w.nb[0], nb1 = w.nb[1];
          if (nbmax - jb == 1) mma_commit(BAR(C::B_Q_EMPTY));
          for (int j = jb + 1; j <= nbmax && ok; ++j) {
            if (!(ok = next_pair(ps))) break;
#pragma unroll
            for (int t = 0; t < 2; ++t) {
              const int nbt = t ? nb1 : nb0;
              if (!ok) break;
              if (j - 1 < nbt) {
                if (!(ok = wait_p(t))) break;
                issue_pv(t, t, 2 * ps + 1, j - 1 > jb);
                if (!C::LAST_O_DONE_ONLY || j >= nbt) mma_commit(BAR(C::B_O_DONE + t));
              }
              if (j < nbt) {
                issue_qk(t, t, 2 * ps);
                mma_commit(BAR(C::B_S_FULL + t));
              }
            }
            if (!ok) break;
            if (j == nbmax - 1) mma_commit(BAR(C::B_Q_EMPTY));
            mma_commit(BAR(C::B_KV_EMPTY + ps));
          }
        } else {
          const int nb = w.nb[0];
          if (!(ok = next_stage(ks))) break;
          issue_qk(0, 0, ks);
          mma_commit(BAR(C::B_S_FULL + 0));
          mma_commit(BAR(C::B_KV_EMPTY + ks));
          if (nb == 1) mma_commit(BAR(C::B_Q_EMPTY));
          for (int j = 1; j <= nb && ok; ++j) {
            if (j < nb) {
              if (!(ok = next_stage(ks))) break;
              issue_qk(0, j & 1, ks);
              mma_commit(BAR(C::B_S_FULL + (j & 1)));
              mma_commit(BAR(C::B_KV_EMPTY + ks));
              if (j == nb - 1) mma_commit(BAR(C::B_Q_EMPTY));
            }
            if (!(ok = next_stage(vs))) break;
            if (!(ok = wait_p((j - 1) & 1))) break;
            issue_pv(0, (j - 1) & 1, vs, j - 1 > 0);
            mma_commit(BAR(C::B_O_DONE + 0));
            mma_commit(BAR(C::B_KV_EMPTY + vs));
          }
        }
      }
      // Every MMA issued by this CTA has finished before TMEM is released.
      mma_commit(BAR(C::B_MMA_DONE));
      mbar_drain(BAR(C::B_MMA_DONE), 0, 100000000ull);
    }
  }
  } else {
    // ------------------------------------------------------------ softmax
    if constexpr (C::REG_SPLIT) setmaxnreg_inc<C::SOFTMAX_REGS>();
    const WaitCtx wc{abort_flag, &g_status_word, p.timeout_ns};
    const int wg = warp >> 2;                 // Q tile / O accumulator of this group
    const int wq = warp & 3;                  // TMEM lane quarter of this warp
    const int row = wq * 32 + lane;           // row within the Q tile
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const uint32_t tm_o = lane_base + (wg == 0 ? C::TM_O0 : C::TM_O1);
    uint32_t sph = 0u, oph = 0u;  // sph bit b: wait parity of S_FULL[b]
    bool ok = true;

    WorkIter wi;
    for (Unit w; ok && wi.next<NQ>(w, p, segs);) {
      const int nb = wg ? w.nb[1] : w.nb[0];
      const int jb = w.jb;
      if (nb == 0) continue;
      const int tile_row0 = w.m0 + wg * kBM;
      const int qi = tile_row0 + row;                  // query row of this thread
      // First key block with a key some row of the tile must not see.
      const int mask_from = (tile_row0 + p.causal_off + 1) / kBN;
      float m_used = -INFINITY, l = 0.f;
      // FP8: query-block scale and the largest V scale of the blocks visited.
      float c_q = p.sl2, sv_max = 1.f;
      if constexpr (F8) {
        const int sb = w.bh * p.scale_bh_stride;
        c_q = p.sl2 * p.q_scale[sb + (tile_row0 / kBM) * p.scale_blk_stride];
        // The lanes share the nb scale loads, then reduce across the warp.
        float mx = 0.f;
        for (int j = jb + lane; j < nb; j += 32) mx = fmaxf(mx, p.v_scale[sb + j * p.scale_blk_stride]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        sv_max = mx > 0.f ? mx : 1.f;
      }

      for (int j = jb; j < nb; ++j) {
        const int b = NQ == 2 ? wg : (j & 1);
        // Per-block multiplier of S and the V fold (FP8); plain scale otherwise.
        float cj = c_q, lg2_ratio = 0.f, inv_ratio = 1.f;
        if constexpr (F8) {
          const int sb = w.bh * p.scale_bh_stride + j * p.scale_blk_stride;
          cj = c_q * p.k_scale[sb];
          const float sv = p.v_scale[sb];
          if (sv > 0.f && sv < sv_max) {
            lg2_ratio = log2f(sv / sv_max);
            inv_ratio = sv_max / sv;
          }
        }
        if (!(ok = mbar_wait_warp(BAR(C::B_S_FULL + b), (sph >> b) & 1u, wc, attn_internal::kStatusTimeoutSoftmax))) break;
        sph ^= 1u << b;
        tc_fence_after();
        const uint32_t tm_s = lane_base + (b ? C::TM_S1 : C::TM_S0);

        const bool masked = (p.causal && j >= mask_from) || (j == w.nkb - 1 && (p.Nk % kBN) != 0);
        // Blocks without masked keys: the loads also give the row's extreme
        // (maximum, or minimum when the scale is negative): of each 32-column
        // chunk for the 16-bit kernels, of all 128 columns in one load for E4M3.
        uint32_t s[4][32];
        float ext[4] = {0.f, 0.f, 0.f, 0.f};
        if (masked) {
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld32(tm_s + 32 * c, s[c]);
        } else if constexpr (F8) {
          // One load for the whole row; the other slots hold the identity of
          // the reduction (ext[0] may be read only after the wait below).
          if (cj >= 0.f) {
            tmem_ld128_red<false>(tm_s, s, ext[0]);
            ext[1] = ext[2] = ext[3] = -INFINITY;
          } else {
            tmem_ld128_red<true>(tm_s, s, ext[0]);
            ext[1] = ext[2] = ext[3] = INFINITY;
          }
        } else if (cj >= 0.f) {
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld32_red<false>(tm_s + 32 * c, s[c], ext[c]);
        } else {
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld32_red<true>(tm_s + 32 * c, s[c], ext[c]);
        }
        tmem_wait_ld(s[0]);
        reg_pin(s[1]);
        reg_pin(s[2]);
        reg_pin(s[3]);
        reg_pin(ext);

        float mblk;
        if (masked) {
          // Scale first, then mask: t = c*s for visible keys, -inf otherwise.
          const int key0 = j * kBN;
          const int kmax = p.causal ? min(qi + p.causal_off, p.Nk - 1) : p.Nk - 1;  // last visible key
          float mx = -INFINITY;
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float t = (key0 + 32 * c + i <= kmax) ? cj * __uint_as_float(s[c][i]) : -INFINITY;
              s[c][i] = __float_as_uint(t);
              mx = fmaxf(mx, t);
            }
          mblk = mx;
        } else {
          const float mx = cj >= 0.f ? fmaxf(fmaxf(ext[0], ext[1]), fmaxf(ext[2], ext[3]))
                                     : fminf(fminf(ext[0], ext[1]), fminf(ext[2], ext[3]));
          mblk = cj * mx;
        }

        float alpha = 1.f;
        bool rescale = false;
        if (j == jb) {
          m_used = (mblk == -INFINITY) ? 0.f : mblk;
        } else if (mblk > m_used + kRescaleThreshold) {
          alpha = ex2(m_used - mblk);
          m_used = mblk;
          rescale = true;
        }

        // P = 2^(c*s - m) (FP8: times sv_j / svmax), written over S.
        float rowsum = 0.f;
        const float neg_m = lg2_ratio - m_used;
        if constexpr (!F8) {
          float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
          const float2 c2 = masked ? make_float2(1.f, 1.f) : make_float2(cj, cj);
          const float2 m2 = make_float2(neg_m, neg_m);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float2 a = ffma2(make_float2(__uint_as_float(s[c][2 * i]), __uint_as_float(s[c][2 * i + 1])), c2, m2);
              const float2 pp = make_float2(ex2(a.x), ex2(a.y));
              if (i & 1) acc1 = fadd2(acc1, pp); else acc0 = fadd2(acc0, pp);
              pk[i] = pack2<KIND>(pp.x, pp.y);
            }
            tmem_st16(tm_s + 16 * c, pk);
          }
          rowsum = (acc0.x + acc0.y) + (acc1.x + acc1.y);
        } else {
          // E4M3 weights, four per TMEM column; each 32-column chunk is stored
          // as soon as it is packed.  In blocks without masked keys the last
          // POLY_QUADS quadruples of every chunk take 2^x on the FMA pipe
          // (exp2_poly2), the rest on the multi-function unit, whose rate
          // the weights of both Q tiles otherwise share; masked blocks take
          // every weight from ex2.approx, which gives masked keys exact zeros.
          float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
          const float2 c2 = masked ? make_float2(1.f, 1.f) : make_float2(cj, cj);
          const float2 m2 = make_float2(neg_m, neg_m);
          auto weights = [&](auto poly) {
            constexpr bool kPoly = decltype(poly)::value;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              uint32_t pk[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const float2 a = ffma2(make_float2(__uint_as_float(s[c][4 * i]), __uint_as_float(s[c][4 * i + 1])), c2, m2);
                const float2 bq = ffma2(make_float2(__uint_as_float(s[c][4 * i + 2]), __uint_as_float(s[c][4 * i + 3])), c2, m2);
                float2 p01, p23;
                if (kPoly && i >= 8 - C::POLY_QUADS) {
                  p01 = exp2_poly2(a);
                  p23 = exp2_poly2(bq);
                } else {
                  p01 = make_float2(ex2(a.x), ex2(a.y));
                  p23 = make_float2(ex2(bq.x), ex2(bq.y));
                }
                acc0 = fadd2(acc0, p01);
                acc1 = fadd2(acc1, p23);
                pk[i] = pack4_e4m3(p01.x, p01.y, p23.x, p23.y);
              }
              tmem_st8(tm_s + 8 * c, pk);
            }
          };
          if (masked || C::POLY_QUADS == 0)
            weights(std::false_type{});
          else
            weights(std::true_type{});
          rowsum = (acc0.x + acc0.y) + (acc1.x + acc1.y);
        }

        if (j > jb) {
          // O holds P_{j-1} V_{j-1} once the previous product has completed.
          if constexpr (!C::LAST_O_DONE_ONLY) {
            if (!(ok = mbar_wait_warp(BAR(C::B_O_DONE + wg), oph, wc, attn_internal::kStatusTimeoutSoftmax))) break;
            oph ^= 1u;
            tc_fence_after();
          }
          if (__any_sync(0xffffffffu, rescale)) {
            // Up to 128 columns of O in flight under one wait (the registers
            // that held S are free by now).
            constexpr int GRP = D / 32 < 4 ? D / 32 : 4;
#pragma unroll 1
            for (int c0 = 0; c0 < D / 32; c0 += GRP) {
              uint32_t o[GRP][32];
#pragma unroll
              for (int g = 0; g < GRP; ++g) tmem_ld32(tm_o + 32 * (c0 + g), o[g]);
              tmem_wait_ld(o[0]);
#pragma unroll
              for (int g = 1; g < GRP; ++g) reg_pin(o[g]);
#pragma unroll
              for (int g = 0; g < GRP; ++g) {
#pragma unroll
                for (int i = 0; i < 32; ++i) o[g][i] = __float_as_uint(__uint_as_float(o[g][i]) * alpha);
                tmem_st32(tm_o + 32 * (c0 + g), o[g]);
              }
            }
          }
        }
        l = l * alpha + rowsum * inv_ratio;
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(C::B_P_FULL + b));
      }
      // A failed wait above (ok = false) still leads to the tile barrier below,
      // where the four warps leave together.

      // Epilogue: O / l (times svmax for FP8), rounded to the output dtype, and
      // lse.  O leaves through this tile's staging buffer, 64 columns at a
      // time, by a bulk tensor store (rows past N are not written).  The four
      // warps of the tile first agree that every one of them saw O_DONE, so
      // that none waits at a tile barrier another has left.
      const bool got_o = ok && mbar_wait_warp(BAR(C::B_O_DONE + wg), oph, wc, attn_internal::kStatusTimeoutSoftmax);
      const uint32_t tile_bar = 1u + static_cast<uint32_t>(wg);
      if (bar_red_or(tile_bar, 128, !got_o)) {
        ok = false;
        break;
      }
      oph ^= 1u;
      tc_fence_after();
      float inv_l = sv_max / l;
      float lse_m = m_used, lse_l = l;
      // Stream-K part: publish this part, and combine if it is the last one.
      int parts = 0;
      const float* part_o[kMaxParts] = {};
      float part_w[kMaxParts] = {};
      if constexpr (NQ == 2) {
        if (w.part) {
          const SkSpan sk(p, w.nkb);
          const int c_first = sk.cta_of(static_cast<int64_t>(w.u) * w.nkb);
          const int c_last = sk.cta_of(static_cast<int64_t>(w.u) * w.nkb + w.nkb - 1);
          const int me = static_cast<int>(blockIdx.x);
          const size_t tile_o = static_cast<size_t>(D) * kBM, tile_ml = 2 * kBM;
          const int my_slot = sk.slot(me, w.u, w.nkb);
          float* po = p.ws_o + (static_cast<size_t>(my_slot) * 2 + wg) * tile_o;
          float* pml = p.ws_ml + (static_cast<size_t>(my_slot) * 2 + wg) * tile_ml;
          // This part's O (at its true scale, times svmax for FP8), m and l.
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tm_o + 32 * c, o);
            tmem_wait_ld(o);
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4)
              *reinterpret_cast<float4*>(po + ((8 * c + q4) * kBM + row) * 4) =
                  make_float4(__uint_as_float(o[4 * q4]) * sv_max, __uint_as_float(o[4 * q4 + 1]) * sv_max,
                              __uint_as_float(o[4 * q4 + 2]) * sv_max, __uint_as_float(o[4 * q4 + 3]) * sv_max);
          }
          pml[row] = m_used;
          pml[kBM + row] = l;
          __threadfence();
          bar_sync_n(tile_bar, 128);
          volatile int* last_flag = reinterpret_cast<volatile int*>(tmem_slot + 2 + wg);
          if (wq == 0 && lane == 0) {
            const unsigned int old = atomicAdd(p.ws_cnt + 2 * c_last + wg, 1u);
            *last_flag = old + 1 == static_cast<unsigned int>(c_last - c_first + 1) ? 1 : 0;
          }
          bar_sync_n(tile_bar, 128);
          if (!*last_flag) {
            tc_fence_before();
            continue;  // another part of this unit tile finishes later and combines
          }
          __threadfence();
          // Every part of this unit tile is in the workspace (this one too).
          parts = c_last - c_first + 1;
          float M = -INFINITY, mp[kMaxParts], lp[kMaxParts];
#pragma unroll
          for (int q = 0; q < kMaxParts; ++q) {
            mp[q] = -INFINITY;
            lp[q] = 0.f;
            if (q < parts) {
              const int slot = sk.slot(c_first + q, w.u, w.nkb);
              const float* ml = p.ws_ml + (static_cast<size_t>(slot) * 2 + wg) * tile_ml;
              mp[q] = __ldcg(ml + row);
              lp[q] = __ldcg(ml + kBM + row);
              part_o[q] = p.ws_o + (static_cast<size_t>(slot) * 2 + wg) * tile_o;
              M = fmaxf(M, mp[q]);
            }
          }
          float L = 0.f;
#pragma unroll
          for (int q = 0; q < kMaxParts; ++q)
            if (q < parts) {
              part_w[q] = ex2(mp[q] - M);
              L += part_w[q] * lp[q];
            }
          inv_l = 1.f / L;
          lse_m = M;
          lse_l = L;
        }
      }
      const uint32_t ost = smem_u32(smem + C::OFF_OST + wg * C::OST_BYTES);
      const uint32_t ost_row = ost + static_cast<uint32_t>(row) * 128u;
      const uint32_t swz = static_cast<uint32_t>(row & 7);
      const int ob = w.bh / p.H, oh = w.bh - ob * p.H;
#pragma unroll 1
      for (int c2 = 0; c2 < D / 64; ++c2) {
        uint32_t o[2][32];
        if (parts > 0) {
          // Combined O: the parts' weighted sum (their slots are in L2).
#pragma unroll
          for (int q4 = 0; q4 < 16; ++q4) {
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int q = 0; q < kMaxParts; ++q)
              if (q < parts) {
                const float4 v4 = __ldcg(reinterpret_cast<const float4*>(part_o[q] + ((16 * c2 + q4) * kBM + row) * 4));
                acc.x = fmaf(part_w[q], v4.x, acc.x);
                acc.y = fmaf(part_w[q], v4.y, acc.y);
                acc.z = fmaf(part_w[q], v4.z, acc.z);
                acc.w = fmaf(part_w[q], v4.w, acc.w);
              }
            const int h = q4 >> 3, i = (q4 & 7) * 4;
            o[h][i] = __float_as_uint(acc.x);
            o[h][i + 1] = __float_as_uint(acc.y);
            o[h][i + 2] = __float_as_uint(acc.z);
            o[h][i + 3] = __float_as_uint(acc.w);
          }
        } else {
          tmem_ld32(tm_o + 64 * c2, o[0]);
          tmem_ld32(tm_o + 64 * c2 + 32, o[1]);
          tmem_wait_ld(o[0]);
          reg_pin(o[1]);
        }
        // The previous bulk store from this buffer must have read it.
        if (wq == 0 && lane == 0) bulk_wait_read_all();
        bar_sync_n(tile_bar, 128);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pk[i] = pack2<F8 ? KIND_BF16 : KIND>(__uint_as_float(o[h][2 * i]) * inv_l,
                                                 __uint_as_float(o[h][2 * i + 1]) * inv_l);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const uint32_t unit = static_cast<uint32_t>(4 * h + v);
            st_shared_v4(ost_row + ((unit ^ swz) << 4), pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
          }
        }
        fence_proxy_async_smem();
        bar_sync_n(tile_bar, 128);
        if (wq == 0 && lane == 0) {
          tma_store_rows(&tmO, ost, 64 * c2, tile_row0, ob, oh, p.layout == ATTN_LAYOUT_BNHD);
          bulk_commit_group();
        }
      }
      if (qi < p.N && p.lse != nullptr)
        p.lse[static_cast<size_t>(w.bh) * p.N + qi] = (lse_m + log2f(lse_l)) * 0.69314718055994531f;
      tc_fence_before();
    }
  }

  // The bulk stores of O read shared memory: let them finish before the CTA exits.
  if (warp < C::SOFTMAX_WARPS && (warp & 3) == 0 && lane == 0) bulk_wait_all();
  tc_fence_before();
  __syncthreads();
  if (warp == C::MMA_WARP) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Workspace of the stream-K schedule on a GPU with `sms` multiprocessors:
// two slots per CTA of (two tiles x (128 x D floats of O, 128 m, 128 l)),
// then two arrival counters per CTA.  0 where the schedule is not used (one
// Q tile per CTA, d = 256).
inline size_t stream_k_ws_bytes(int D, int sms) {
  if (D > 128 || sms <= 0) return 0;
  const size_t slots = 2 * static_cast<size_t>(sms);
  return align256(slots * 2 * D * kBM * 4) + align256(slots * 2 * 2 * kBM * 4) +
         align256(static_cast<size_t>(sms) * 2 * 4);
}

// Host side: encode the three tensor maps, set the shared-memory attribute
// once per device, and launch one CTA per SM (or per unit, if fewer).  With
// a workspace of at least stream_k_ws_bytes(D, SMs) bytes (256-byte aligned),
// full attention over at least one unit per SM whose units do not divide
// evenly over the SMs runs the stream-K schedule.
template <int D, int KIND>
attn_status launch_fwd(const void* q, const void* k, const void* v, FwdParams prm, int B, int H,
                       int N, int Nk, float scale, cudaStream_t stream, void* ws = nullptr,
                       size_t ws_bytes = 0) {
  using C = Cfg<D, KIND>;
  const CUtensorMapDataType dt = KIND == KIND_E4M3   ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                 : KIND == KIND_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                     : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const uint64_t BH = static_cast<uint64_t>(B) * H;
  CUtensorMap mq, mk, mv, mo;
  const CUtensorMapDataType dto = KIND == KIND_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  // {d, N, H, B} for [B, H, N, d], {d, H, N, B} for [B, N, H, d], N being the
  // query length for Q and O and the key length for K and V; the box is box_x
  // elements of `rows` consecutive rows of one head.
  const bool bnhd = prm.layout == ATTN_LAYOUT_BNHD;
  auto encode = [&](CUtensorMap* m, CUtensorMapDataType t, const void* base, uint64_t elem, uint32_t box_x,
                    uint32_t rows, int len) {
    const uint64_t dims[4] = {static_cast<uint64_t>(D), static_cast<uint64_t>(bnhd ? H : len),
                              static_cast<uint64_t>(bnhd ? len : H), static_cast<uint64_t>(B)};
    const uint64_t strides[3] = {D * elem, dims[1] * D * elem, dims[2] * dims[1] * D * elem};
    const uint32_t box[4] = {box_x, bnhd ? 1u : rows, bnhd ? rows : 1u, 1u};
    return attn_internal::encode_tmap_4d(m, t, base, dims, strides, box,
                                         box_x * elem == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B);
  };
  if (!encode(&mq, dt, q, C::ELEM, C::CHUNK_ELEMS, kBM, N) || !encode(&mk, dt, k, C::ELEM, C::CHUNK_ELEMS, kBN, Nk) ||
      !encode(&mv, dt, v, C::ELEM, C::CHUNK_ELEMS, kBN, Nk) || !encode(&mo, dto, prm.o, 2, 64, kBM, N))
    return ATTN_ERR_CUDA;

  static int configured_for[64] = {0};  // per device: dynamic shared memory attribute set
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return attn_internal::cuda_status(e);
  if (dev >= 64 || !configured_for[dev]) {
    e = cudaFuncSetAttribute(attn_fwd_kernel<D, KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::SMEM_BYTES);
    if (e != cudaSuccess) return attn_internal::cuda_status(e);
    if (dev < 64) configured_for[dev] = 1;
  }
  prm.BH = static_cast<int>(BH);
  prm.H = H;
  prm.N = N;
  prm.Nk = Nk;
  prm.sl2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  prm.units_per_head = (N + kBM * C::NQ - 1) / (kBM * C::NQ);
  const int units = prm.units_per_head * prm.BH;
  prm.timeout_ns = attn_internal::wait_timeout_ns();
  const int sms = attn_internal::sm_count();
  if (sms <= 0) return ATTN_ERR_CUDA;
  // Full attention with two Q tiles per unit: when the last round of the
  // persistent schedule would be at most half full, its units are split into
  // half units (one Q tile each, one per CTA), so that round costs half a unit.
  prm.full_units = units;
  prm.num_units = units;
  prm.stream_k = 0;
  const size_t sk_bytes = stream_k_ws_bytes(D, sms);
  // Stream-K tail for every kind whenever a workspace is given, except in
  // the one-tile (no overlap) schedule.
  const int mode = attn_internal::schedule_mode();
  if (C::NQ == 2 && !prm.causal && ws != nullptr && sk_bytes > 0 && ws_bytes >= sk_bytes &&
      mode != ATTN_SCHEDULE_ONE_TILE && units >= sms && units % sms != 0) {
    // The last `tail` units go to stream-K (at least half a round, so every
    // range holds half a unit's key blocks or more); the rest run in whole
    // round-robin rounds, head-major, so that CTAs working at the same time
    // share K and V through L2.
    const int rest = units % sms;
    const int tail = 2 * rest >= sms ? rest : rest + sms;
    const size_t slots = 2 * static_cast<size_t>(sms);
    uint8_t* base = static_cast<uint8_t*>(ws);
    prm.stream_k = 1;
    prm.sk_unit0 = units - tail;
    prm.ws_o = reinterpret_cast<float*>(base);
    prm.ws_ml = reinterpret_cast<float*>(base + align256(slots * 2 * D * kBM * 4));
    prm.ws_cnt = reinterpret_cast<unsigned int*>(base + align256(slots * 2 * D * kBM * 4) +
                                                 align256(slots * 2 * 2 * kBM * 4));
    cudaError_t me = cudaMemsetAsync(prm.ws_cnt, 0, static_cast<size_t>(sms) * 2 * 4, stream);
    if (me != cudaSuccess) return attn_internal::cuda_status(me);
  } else if (C::NQ == 2 && mode == ATTN_SCHEDULE_ONE_TILE) {
    prm.full_units = 0;  // every entry a half unit: one Q tile per CTA at a time
    prm.num_units = 2 * units;
  } else if (C::NQ == 2 && !prm.causal) {
    const int rest = units % sms;
    if (units <= sms / 2) {
      prm.full_units = 0;
      prm.num_units = 2 * units;
    } else if (units > sms && rest > 0 && 2 * rest <= sms) {
      prm.full_units = units - rest;
      prm.num_units = units + rest;
    }
  }
  const int grid = prm.stream_k ? sms : (prm.num_units < sms ? prm.num_units : sms);
  attn_fwd_kernel<D, KIND><<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(mq, mk, mv, mo, prm);
  return attn_internal::cuda_status(cudaGetLastError());
}

inline cudaError_t status_exchange(unsigned int* out) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_status_word, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_status_word, &zero, sizeof(unsigned int));
}

}  // namespace attn_kernel
