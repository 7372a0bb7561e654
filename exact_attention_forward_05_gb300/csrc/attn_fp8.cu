// attn_fp8.cu -- FP8 (E4M3) path of the exact attention forward.
//
// Pre-pass ("Incoherent Processing for FP8 Accuracy", FlashAttention-3 podcast
// page; comrad404 review, "Метод", item 3): every row of Q and K is multiplied
// by diag(sigma_h) H_d / sqrt(d) -- random signs of its head, then the
// Sylvester Hadamard transform, O(d log d) butterflies -- and Q, K, V are
// quantised to E4M3 with one float32 scale per 128 rows of a head:
// s = amax / 448 (1 when the block is all zero), code = RNE_satfinite(x / s).
// The rotation is orthogonal and shared by Q and K of a head, so Q K^T is
// unchanged; V is not rotated.  A per-tensor mode (one scale per tensor, no
// rotation) gives the naive FP8 baseline the pages compare against.
//
// The same section names rotary embeddings as the memory-bound step the
// Hadamard transform is fused into: given cos / sin tables, the pre-pass first
// applies the rotary embedding to Q and K (RoFormer's pairwise rotation, pairs
// (2i, 2i+1) or (i, i + d/2)), in the registers that then take the rotation,
// so the fused step reads and writes each row once.
//
// The pre-pass takes d = 64, 128 or 256; the attention kernel itself is
// attn_kernel::attn_fwd_kernel<d, E4M3>.
#include "attn_kernel.cuh"

using attn_kernel::FwdParams;
using attn_kernel::KIND_E4M3;
using sm103::fadd2;
using sm103::ffma2;
using sm103::fmul2;
using sm103::fsub2;

namespace {

using namespace sm103;

constexpr int kQuantRows = 128;   // rows per scale block
constexpr int kPrepThreads = 512; // 128 rows x 4 lanes; a lane holds d / 4 values of its row
constexpr float kE4M3Max = 448.0f;

enum PrepMode : int { PREP_BLOCK = 0, PREP_AMAX = 1, PREP_QUANT_GLOBAL = 2 };

struct PrepParams {
  const void* src[3];
  uint8_t* dst[3];
  float* scale[3];
  const int8_t* signs;  // [H][d] +-1, or nullptr (no rotation)
  const float* rcos;    // [N][d/2] rotary tables, or nullptr (no rotary embedding)
  const float* rsin;
  int rope_interleaved; // pairs (2i, 2i+1) if nonzero, else (i, i + d/2)
  int H, N, nblk, BH;
  int codes_align32;    // Q and K code buffers start on 32-byte boundaries
};

// Correctly rounded x / s from y = RN(1 / s) with one FMA correction of the
// product (Markstein, "Computation of elementary functions on the IBM RISC
// System/6000 processor", IBM J. Res. Dev. 34(1), 1990): q0 = RN(x y),
// e = q0 s - x exactly, q = RN(q0 - e y).  The residual is taken as q0 s - x
// (not x - q0 s) so that a zero keeps its sign: x = -0 gives e = +0 and
// q = RN(-0 + -0) = -0, where RN(q0 + r y) with r = x - q0 s gives +0.  Used
// where |x / s| <= 448 and s is a normal number far from the exponent limits;
// other scales take the division itself.  Two quotients at a time:
// s2 = (s, s), ny2 = (-y, -y), y2 = (y, y).
__device__ __forceinline__ float2 div_by_scale2(float2 x, float2 s2, float2 ny2, float2 y2) {
  const float2 q0 = fmul2(x, y2);
  const float2 e = ffma2(q0, s2, fmul2(x, make_float2(-1.f, -1.f)));
  return ffma2(e, ny2, q0);
}

template <int VPL>
__device__ __forceinline__ float2 pair(const float (&x)[VPL], int e) { return make_float2(x[e], x[e + 1]); }
template <int VPL>
__device__ __forceinline__ void put(float (&x)[VPL], int e, float2 v) {
  x[e] = v.x;
  x[e + 1] = v.y;
}

// Sylvester-ordered fast Walsh-Hadamard transform of one row of 4 * VPL
// elements held by the 4 lanes of its group (lane g owns elements
// VPL g .. VPL g + VPL - 1): butterflies of stride 1 .. VPL / 2 inside the
// thread, VPL and 2 VPL across the group.  The stages commute, so any order
// gives the transform.  Strides from 2 on combine whole element pairs with
// paired instructions.
template <int VPL>
__device__ __forceinline__ void fwht_row(float (&x)[VPL], int g) {
#pragma unroll
  for (int e = 0; e < VPL; e += 2) {
    const float a = x[e], b = x[e + 1];
    x[e] = a + b;
    x[e + 1] = a - b;
  }
#pragma unroll
  for (int m = 2; m < VPL; m <<= 1)
#pragma unroll
    for (int e = 0; e < VPL; e += 2)
      if ((e & m) == 0) {
        const float2 a = pair(x, e), b = pair(x, e + m);
        put(x, e, fadd2(a, b));
        put(x, e + m, fsub2(a, b));
      }
#pragma unroll
  for (int m = 1; m < 4; m <<= 1) {
    const float sgn = (g & m) ? -1.f : 1.f;  // upper half of the pair: partner - own
    const float2 sg2 = make_float2(sgn, sgn);
#pragma unroll
    for (int e = 0; e < VPL; e += 2) {
      const float2 o = make_float2(__shfl_xor_sync(0xffffffffu, x[e], m),
                                   __shfl_xor_sync(0xffffffffu, x[e + 1], m));
      put(x, e, ffma2(pair(x, e), sg2, o));
    }
  }
}

// Rotary embedding of this lane's VPL values of a row: (a, b) -> (a cos - b sin,
// a sin + b cos), table entries from `cr` / `sr` (the row's d/2 cos and sin
// values, shared or global memory).  Interleaved pairs (2i, 2i+1) are inside
// the lane; half-split pairs (i, i + d/2) pair lane g with lane g ^ 2 of the
// row's group, one shuffle per value (every lane of the warp takes part).
template <int VPL>
__device__ __forceinline__ void rotary_row(float (&x)[VPL], int g, const float* cr, const float* sr,
                                           bool interleaved, bool have) {
  const float4 zero4 = make_float4(0.f, 0.f, 0.f, 0.f);
  if (interleaved) {
    // This lane's elements VPL g .. are the pairs i = VPL g / 2 ...
    const float4* c4 = reinterpret_cast<const float4*>(cr + (VPL / 2) * g);
    const float4* s4 = reinterpret_cast<const float4*>(sr + (VPL / 2) * g);
#pragma unroll
    for (int w = 0; w < VPL / 8; ++w) {
      const float4 cv = have ? c4[w] : zero4, sv = have ? s4[w] : zero4;
      const float cc[4] = {cv.x, cv.y, cv.z, cv.w}, ss[4] = {sv.x, sv.y, sv.z, sv.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int e = 8 * w + 2 * u;
        const float a = x[e], b = x[e + 1];
        // (a c - b s, a s + b c): b (-s, c), then a (c, s) added with one rounding.
        const float2 t2 = fmul2(make_float2(b, b), make_float2(-ss[u], cc[u]));
        put(x, e, ffma2(make_float2(a, a), make_float2(cc[u], ss[u]), t2));
      }
    }
  } else {
    // Pair i = VPL (g & 1) + e is (element i, element i + d/2): lanes g and g ^ 2
    // of the row's group hold its two halves.
    const float4* c4 = reinterpret_cast<const float4*>(cr + VPL * (g & 1));
    const float4* s4 = reinterpret_cast<const float4*>(sr + VPL * (g & 1));
    const float sgn = (g & 2) ? 1.f : -1.f;  // second half: b cos + a sin
#pragma unroll
    for (int w = 0; w < VPL / 4; ++w) {
      const float4 cv = have ? c4[w] : zero4, sv = have ? s4[w] : zero4;
      const float cc[4] = {cv.x, cv.y, cv.z, cv.w}, ss[4] = {sv.x, sv.y, sv.z, sv.w};
#pragma unroll
      for (int u = 0; u < 4; u += 2) {
        const int e = 4 * w + u;
        const float2 o = make_float2(__shfl_xor_sync(0xffffffffu, x[e], 2),
                                     __shfl_xor_sync(0xffffffffu, x[e + 1], 2));
        const float2 t2 = fmul2(pair(x, e), make_float2(cc[u], cc[u + 1]));
        put(x, e, ffma2(o, make_float2(sgn * ss[u], sgn * ss[u + 1]), t2));
      }
    }
  }
}

// One CTA of 512 threads per (128-row block, tensor, head) item; two CTAs
// share an SM at d <= 128.  Every lane loads its d / 4 values of its row
// (row-contiguous 16-byte loads), applies the rotary embedding, the signs and
// the Hadamard transform (Q and K), the block maximum is reduced across the
// CTA, and the lane quantises and stores its codes.
template <int D, bool BF16IN, int MODE>
__global__ void __launch_bounds__(kPrepThreads, D <= 128 ? 2 : 1) fp8_prepare_kernel(const PrepParams p) {
  constexpr int VPL = D / 4;
  const int t = blockIdx.y;                     // 0 = Q, 1 = K, 2 = V
  const int blk = blockIdx.x % p.nblk;
  const int bh = blockIdx.x / p.nblk;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane & 3;                       // lane within the row's group of 4
  const bool qk = t < 2;
  const size_t head = static_cast<size_t>(bh) * p.N * D;
  // Operands chosen by selects, not by indexing the parameter arrays (which
  // would copy them to local memory).
  const uint8_t* src = static_cast<const uint8_t*>(t == 0 ? p.src[0] : t == 1 ? p.src[1] : p.src[2]);
  float* scale_t = t == 0 ? p.scale[0] : t == 1 ? p.scale[1] : p.scale[2];
  uint8_t* dst = t == 0 ? p.dst[0] : t == 1 ? p.dst[1] : p.dst[2];

  const int row = blk * kQuantRows + warp * 8 + (lane >> 2);
  const bool have = row < p.N;
  // Without a rotary embedding the signs go on the 16-bit input words, before
  // the conversion (a sign-bit XOR commutes with it): per pair of values one
  // byte permute moves the two sign bytes under bits 15 and 31 and one logic
  // op applies them (block-uniform choice).
  const bool pre_signs = qk && p.signs != nullptr && p.rcos == nullptr;
  const int4* sgn = reinterpret_cast<const int4*>(p.signs + (bh % p.H) * D + VPL * g);
  float x[VPL];
  if (have) {
    const uint4* ptr = reinterpret_cast<const uint4*>(src + (head + static_cast<size_t>(row) * D + VPL * g) * 2);
#pragma unroll
    for (int v = 0; v < VPL / 8; ++v) {
      const uint4 r = ptr[v];
      uint32_t w4[4] = {r.x, r.y, r.z, r.w};
      if (pre_signs) {
        // Sign bytes of elements 8v .. 8v + 7: two words of the 16-byte load v / 2.
        const int4 sv = sgn[v >> 1];
        const uint32_t s0 = static_cast<uint32_t>((v & 1) ? sv.z : sv.x);
        const uint32_t s1 = static_cast<uint32_t>((v & 1) ? sv.w : sv.y);
        w4[0] ^= __byte_perm(s0, 0u, 0x1404u) & 0x80008000u;
        w4[1] ^= __byte_perm(s0, 0u, 0x3424u) & 0x80008000u;
        w4[2] ^= __byte_perm(s1, 0u, 0x1404u) & 0x80008000u;
        w4[3] ^= __byte_perm(s1, 0u, 0x3424u) & 0x80008000u;
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float2 f;
        if constexpr (BF16IN) f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w4[k]));
        else f = __half22float2(*reinterpret_cast<const __half2*>(&w4[k]));
        x[8 * v + 2 * k] = f.x;
        x[8 * v + 2 * k + 1] = f.y;
      }
    }
  } else {
#pragma unroll
    for (int e = 0; e < VPL; ++e) x[e] = 0.f;
  }
  if (qk && p.rcos != nullptr) {
    // Block-uniform branch (the half-split form shuffles); rows past N are
    // zero and skip the table loads.
    const float* cr = p.rcos + static_cast<size_t>(have ? row : 0) * (D / 2);
    const float* sr = p.rsin + static_cast<size_t>(have ? row : 0) * (D / 2);
    rotary_row<VPL>(x, g, cr, sr, p.rope_interleaved != 0, have);
  }
  if (qk && p.signs != nullptr) {
    // Signs (+1 = 0x01, -1 = 0xff): bit 7 of each byte becomes the float's sign
    // bit (here only after a rotary embedding; otherwise applied above).
    const int4* sp = sgn;
#pragma unroll
    for (int v = 0; v < VPL / 16 && !pre_signs; ++v) {
      const int4 sv = sp[v];
      const uint32_t sw[4] = {static_cast<uint32_t>(sv.x), static_cast<uint32_t>(sv.y),
                              static_cast<uint32_t>(sv.z), static_cast<uint32_t>(sv.w)};
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const uint32_t bit = (sw[e >> 2] << (24 - 8 * (e & 3))) & 0x80000000u;
        x[16 * v + e] = __uint_as_float(__float_as_uint(x[16 * v + e]) ^ bit);
      }
    }
    fwht_row<VPL>(x, g);
    constexpr float inv_sqrt_d = D == 64 ? 0.125f : (D == 128 ? 0.08838834764831845f : 0.0625f);
    const float2 isd = make_float2(inv_sqrt_d, inv_sqrt_d);
#pragma unroll
    for (int e = 0; e < VPL; e += 2) put(x, e, fmul2(pair(x, e), isd));
  }

  // amax of the block
  __shared__ float warp_max[kPrepThreads / 32];
  float a = 0.f;
#pragma unroll
  for (int e = 0; e < VPL; e += 2) a = max3(a, fabsf(x[e]), fabsf(x[e + 1]));
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, m));
  if (lane == 0) warp_max[warp] = a;
  __syncthreads();
  float amax = 0.f;
#pragma unroll
  for (int w = 0; w < kPrepThreads / 32; ++w) amax = fmaxf(amax, warp_max[w]);

  if constexpr (MODE == PREP_AMAX) {
    if (threadIdx.x == 0) atomicMax(reinterpret_cast<unsigned int*>(scale_t), __float_as_uint(amax));
    return;
  } else {
    float s;
    if constexpr (MODE == PREP_BLOCK) {
      s = amax > 0.f ? amax / kE4M3Max : 1.f;
      if (threadIdx.x == 0) scale_t[static_cast<size_t>(bh) * p.nblk + blk] = s;
    } else {
      const float g_amax = __uint_as_float(*reinterpret_cast<const unsigned int*>(scale_t));
      s = g_amax > 0.f ? g_amax / kE4M3Max : 1.f;
    }
    // Block-uniform choice: the FMA-corrected quotient for ordinary scales.
    const bool fast = s >= 0x1p-100f && s <= 0x1p+100f;
    const float y = __frcp_rn(s);
    if (have) {
      uint32_t pk[VPL / 4];
      const float2 s2 = make_float2(s, s), ny2 = make_float2(-y, -y), y2 = make_float2(y, y);
#pragma unroll
      for (int k = 0; k < VPL / 4; ++k) {
        float2 q01, q23;
        if (fast) {
          q01 = div_by_scale2(pair(x, 4 * k), s2, ny2, y2);
          q23 = div_by_scale2(pair(x, 4 * k + 2), s2, ny2, y2);
        } else {
          q01 = make_float2(__fdiv_rn(x[4 * k], s), __fdiv_rn(x[4 * k + 1], s));
          q23 = make_float2(__fdiv_rn(x[4 * k + 2], s), __fdiv_rn(x[4 * k + 3], s));
        }
        const uint32_t lo = __nv_cvt_float2_to_fp8x2(q01, __NV_SATFINITE, __NV_E4M3);
        const uint32_t hi = __nv_cvt_float2_to_fp8x2(q23, __NV_SATFINITE, __NV_E4M3);
        pk[k] = lo | (hi << 16);
      }
      uint4* out = reinterpret_cast<uint4*>(dst + head + static_cast<size_t>(row) * D + VPL * g);
#pragma unroll
      for (int v = 0; v < VPL / 16; ++v) out[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
    }
  }
}

// ---------------------------------------------------------------------------
// d = 128 with per-block scales: the streaming pre-pass.
//
// A persistent grid (two 512-thread CTAs per SM; one when the rotary tables
// are staged in shared memory) walks the (row block, head) units in
// contiguous ranges, head fastest, so consecutive units read the same rotary
// table rows.  A unit is three steps, Q, K and V of its 128 rows, each with its
// own 32 KiB stage: while a CTA works on one step, each lane already has its
// row of the next one or two steps in flight (16-byte asynchronous copies,
// zero-filled past N, into the lane's own slots of the stage); a stage is
// refilled as soon as its step has read it.  The three steps are unrolled, so
// the code has no branch on the tensor.  One barrier per Q and K step gathers
// the block maxima; V has none of its own (its maximum, taken from the 16-bit
// words in the K step, is published by the K barrier).
//
// Row layout over the 4 lanes of its group: lane g holds the four 8-element
// runs v*32 + g*8 + j (register index e = 8 v + j), so the group's global
// accesses are 64 contiguous bytes.  The Hadamard butterflies of element bits
// 0, 1, 2 (j) and 5, 6 (v) run in registers; a transpose through the warp's
// slots of the step's stage (two halves of 16 values, XOR-swizzled so that
// neither side has bank conflicts) then gives lane g the contiguous elements
// 32 g .. 32 g + 31 (register index = element - 32 g), whose bits 3 and 4 take
// the last two stages in registers.
//
// With the rotation, 1 / sqrt(d) is folded into the quantisation: the block
// maximum of the unscaled values times 1 / sqrt(d) (rounding is monotone, so
// this is the maximum of the scaled values, and s is the same float), and the
// codes are RNE_satfinite(x * 448 / amax_unscaled) from the hardware
// reciprocal, within a few float32 roundings of x / (sqrt(d) s).  Without the
// rotation the codes keep the FMA-corrected quotient, bit-exact against the
// float32 division.
constexpr int kStreamD = 128;
constexpr int kStreamStageBytes = kQuantRows * kStreamD * 2;  // 32 KiB: one tensor of a unit
constexpr int kStreamSlotStride = kPrepThreads * 16;          // bytes between a lane's 4 slots
constexpr int kStreamSmemBytes = 3 * kStreamStageBytes;
// Rotary tables of the current 128-row block in shared memory (rotary kernel,
// one CTA per SM): per row and lane g, the 16 cos and 16 sin entries the lane
// uses, as 8 float4 in the order it reads them, XOR-swizzled within the lane's
// 128 bytes so that a warp's reads are conflict-free.
constexpr int kStreamTableBytes = kQuantRows * 4 * 8 * 16;  // 64 KiB

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 r;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "r"(addr)
               : "memory");
  return r;
}

// 32-byte store (the address is 32-byte aligned).
__device__ __forceinline__ void st_global_v8(void* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d, uint32_t e,
                                             uint32_t f, uint32_t g, uint32_t h) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(a), "r"(b), "r"(c), "r"(d),
               "r"(e), "r"(f), "r"(g), "r"(h)
               : "memory");
}

// Per-halfword unsigned maximum of two packed pairs.
__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// (x0 + x1, x0 - x1) of the 16-bit pair w (x0 in the low half), each with one
// rounding, as the float32 sum and difference of the widened values: the
// mixed-precision add and subtract take x0 in its 16-bit form.
template <bool BF16IN>
__device__ __forceinline__ float2 widen_butterfly(uint32_t w) {
  float s, d;
  if constexpr (BF16IN) {
    const float x1 = __uint_as_float(w & 0xffff0000u);
    asm("{.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tadd.rn.f32.bf16 %0, l, %3;\n\tsub.rn.f32.bf16 %1, l, %3;}"
        : "=f"(s), "=f"(d)
        : "r"(w), "f"(x1));
  } else {
    asm("{.reg .b16 l, h;\n\t.reg .f32 x1;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 x1, h;\n\t"
        "add.rn.f32.f16 %0, l, x1;\n\tsub.rn.f32.f16 %1, l, x1;}"
        : "=f"(s), "=f"(d)
        : "r"(w));
  }
  return make_float2(s, d);
}

// q = RN(a / b) from y = RN(1 / b) (FMA correction, as div_by_scale2).
__device__ __forceinline__ float div_corrected(float a, float b, float y) {
  const float q0 = a * y;
  const float r = fmaf(-q0, b, a);
  return fmaf(r, y, q0);
}

// Word i of a head's sign masks (signs: its d = 128 bytes, +1 = 0x01,
// -1 = 0xff).  i < 64: lane g = i / 16, run v, pair q of the 16-bit input:
// bits 15 and 31 are the signs of elements 32 v + 8 g + 2 q and + 1, XORed onto
// the packed pair.  i >= 64 (rotary step, k = i mod 16): the product of the
// two signs of rotary pair k of lane g at bit 31, XORed onto its sine
// (half-split pairs: element 32 v + 8 g + j and + 64, k = 8 v + j; interleaved:
// elements 32 v + 8 g + 2 q and + 1, k = 4 v + q).
__device__ __forceinline__ uint32_t sign_mask_word(const int8_t* sg, int i, bool interleaved) {
  const int g = (i >> 4) & 3;
  if (i < 64) {
    const int e = ((i >> 2) & 3) * 32 + g * 8 + (i & 3) * 2;
    return (static_cast<uint32_t>(static_cast<uint8_t>(sg[e]) & 0x80u) << 8) |
           (static_cast<uint32_t>(static_cast<uint8_t>(sg[e + 1]) & 0x80u) << 24);
  }
  const int k = i & 15;
  const int ea = interleaved ? (k >> 2) * 32 + g * 8 + (k & 3) * 2 : (k >> 3) * 32 + g * 8 + (k & 7);
  const int eb = interleaved ? ea + 1 : ea + 64;
  return static_cast<uint32_t>((static_cast<uint8_t>(sg[ea]) ^ static_cast<uint8_t>(sg[eb])) & 0x80u) << 24;
}

// Position of sign_mask_word i in the shared table: lane g's input masks at
// g * 36, its rotary sine masks at g * 36 + 16.
__device__ __forceinline__ int mask_slot(int i) { return ((i >> 4) & 3) * 36 + (i >= 64 ? 16 : 0) + (i & 15); }

// Lane indices of the thread, read through an empty volatile asm so that the
// compiler re-derives them (and the addresses built from them) where they are
// used instead of holding them in registers for the whole kernel.
struct LaneIds {
  int tid, warp, lane, g, rw, rib;  // rib: row in the 128-row block
};
__device__ __forceinline__ LaneIds lane_ids() {
  int t = threadIdx.x;
  asm volatile("" : "+r"(t));
  LaneIds l;
  l.tid = t;
  l.warp = t >> 5;
  l.lane = t & 31;
  l.g = t & 3;
  l.rw = (t & 31) >> 2;
  l.rib = l.warp * 8 + l.rw;
  return l;
}

// Unit cursor: row block and head (h = bh mod H), head fastest.
struct PrepUnit {
  int bh, h, blk;
};
__device__ __forceinline__ void next_unit(PrepUnit& u, int BH, int H) {
  if (++u.h == H) u.h = 0;
  if (++u.bh == BH) {
    u.bh = 0;
    ++u.blk;
  }
}

template <bool BF16IN, bool ROPE, bool ROTATE>
__global__ void __launch_bounds__(kPrepThreads, ROPE ? 1 : 2) fp8_prepare_stream_kernel(const PrepParams p, int n_units) {
  constexpr int D = kStreamD, VPL = D / 4;
  constexpr float kInvSqrtD = 0.08838834764831845f;
  extern __shared__ __align__(128) uint8_t stream_smem[];
  // Block maxima (float bits) of Q, K and V, double-buffered by unit parity.
  __shared__ unsigned int blk_amax[2][3];
  // The sign masks (sign_mask_word) of the head of this unit and of the next,
  // by unit parity.
  // Lane g's 32 words at g * 36 (16-byte aligned, no bank conflicts between the
  // four lanes of a row).
  __shared__ __align__(16) uint32_t mask_tab[2][4 * 36];
  // Lane indices are re-read in every step (lane_ids), so that the per-lane
  // addresses derived from them are not kept live across the whole loop.
  const int tid0 = threadIdx.x;
  const uint32_t sbase = smem_u32(stream_smem);
  const int begin = static_cast<int>(static_cast<long long>(n_units) * blockIdx.x / gridDim.x);
  const int end = static_cast<int>(static_cast<long long>(n_units) * (blockIdx.x + 1) / gridDim.x);
  constexpr bool rotate = ROTATE;  // the caller passed signs
  if (tid0 < 6) (&blk_amax[0][0])[tid0] = 0u;

  // Row of this lane in a unit, as an index into the [B*H*N] rows (below 2^31:
  // the host takes the generic kernel otherwise); rows past N copy nothing.
  auto lane_row = [&](const PrepUnit& u, uint32_t& bytes) -> int {
    const int row = u.blk * kQuantRows + lane_ids().rib;
    bytes = row < p.N ? 16u : 0u;
    return u.bh * p.N + (row < p.N ? row : 0);
  };
  // Copies of tensor T's rows of a unit into stage T (one commit group, empty
  // past the CTA's range, so that every step waits for the same group count).
  auto issue = [&](auto tc, bool live, int ridx, uint32_t bytes) {
    constexpr int T = decltype(tc)::value;
    if (live) {
      const LaneIds L = lane_ids();
      const uint8_t* src = static_cast<const uint8_t*>(p.src[T]) + static_cast<size_t>(ridx) * (D * 2) + L.g * 16;
      const uint32_t dst = sbase + T * kStreamStageBytes + L.tid * 16;
#pragma unroll
      for (int v = 0; v < 4; ++v) cp_async16(dst + v * kStreamSlotStride, src + v * 64, bytes);
    }
    cp_async_commit();
  };

  PrepUnit cur;
  cur.blk = begin / p.BH;
  cur.bh = begin - cur.blk * p.BH;
  cur.h = cur.bh % p.H;
  constexpr int kMaskWords = ROPE ? 128 : 64;
  if (rotate && tid0 < kMaskWords)
    mask_tab[begin & 1][mask_slot(tid0)] = sign_mask_word(p.signs + cur.h * D, tid0, p.rope_interleaved != 0);
  __syncthreads();
  {
    uint32_t bytes;
    const int ridx = lane_row(cur, bytes);
    const bool live = begin < end;
    issue(std::integral_constant<int, 0>(), live, ridx, bytes);
    issue(std::integral_constant<int, 1>(), live, ridx, bytes);
  }

  // Rotary kernel: float4 k of lane block lb = 4 r + g (row r of the block)
  // holds cos (k even) or sin (k odd) entries of quad k / 2: half-split pairs
  // i = 32 v + 8 g + 4 hh + 0..3 with k / 2 = 2 v + hh; interleaved pairs
  // i = 16 v + 4 g + 0..3 with k / 2 = v.
  const uint32_t tbase = sbase + 3 * kStreamStageBytes;
  auto load_tables = [&](int blk) {
    const float4 zero4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int f = tid0 + kPrepThreads * i, lb = f >> 3, k = f & 7, gg = lb & 3;
      const int row = blk * kQuantRows + (lb >> 2);
      const int quad = k >> 1;
      const int idx = p.rope_interleaved ? 16 * quad + 4 * gg : 32 * (quad >> 1) + 8 * gg + 4 * (quad & 1);
      const float* tab = (k & 1) ? p.rsin : p.rcos;
      const float4 val = row < p.N ? *reinterpret_cast<const float4*>(tab + static_cast<size_t>(row) * (D / 2) + idx)
                                   : zero4;
      st_shared_v4(tbase + (lb * 8 + (k ^ (lb & 7))) * 16, __float_as_uint(val.x), __float_as_uint(val.y),
                   __float_as_uint(val.z), __float_as_uint(val.w));
    }
  };
  int table_blk = -1;

  for (int u = begin; u < end; ++u) {
    const int par = u & 1;
    if constexpr (ROPE) {
      if (cur.blk != table_blk) {
        // The previous block's tables were last read before the previous K barrier.
        load_tables(cur.blk);
        __syncthreads();
        table_blk = cur.blk;
      }
    }
    // Per-lane values are recomputed where they are used (registers are the
    // limit at two CTAs per SM: 64 per thread).

    auto step = [&](auto tc) {
      constexpr int T = decltype(tc)::value;
      constexpr bool QK = T < 2;
      const bool fwht = QK && rotate;  // uniform over the grid
      const LaneIds L = lane_ids();
      const int tid = L.tid, warp = L.warp, lane = L.lane, g = L.g, rw = L.rw, rib = L.rib;
      // Refill the stage the previous step read: V of this unit before Q, then
      // Q and K of the next unit; this step's copies are two commit groups back.
      if constexpr (T == 0) {
        uint32_t bytes;
        const int r = lane_row(cur, bytes);
        issue(std::integral_constant<int, 2>(), true, r, bytes);
      } else {
        PrepUnit nx = cur;
        next_unit(nx, p.BH, p.H);
        uint32_t bytes;
        const int r = lane_row(nx, bytes);
        issue(std::integral_constant<int, T - 1>(), u + 1 < end, r, bytes);
      }
      // Without the rotary step the widening and the first butterfly (element
      // bit 0) are one step: x0 + x1 and x0 - x1 straight from the 16-bit pair.
      const bool fused = fwht && !ROPE;
      const uint32_t* mt = mask_tab[par] + g * 36;  // this lane's sign masks
      cp_async_wait<2>();  // this step's group; the next two steps' stay in flight
      if constexpr (T == 1) {
        // V of this unit (its copies are one group behind K's): its block
        // maximum goes out before K's registers fill up.
        cp_async_wait<1>();
        const uint32_t sv = sbase + 2 * kStreamStageBytes + tid * 16;
        uint32_t vm = 0u;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const uint4 r = ld_shared_v4(sv + v * kStreamSlotStride);
          vm = max_u16x2(vm, max_u16x2(max_u16x2(r.x & 0x7fff7fffu, r.y & 0x7fff7fffu),
                                       max_u16x2(r.z & 0x7fff7fffu, r.w & 0x7fff7fffu)));
        }
        vm = max(vm & 0xffffu, vm >> 16);
        float va;
        if constexpr (BF16IN) va = __uint_as_float(vm << 16);
        else va = __half2float(__ushort_as_half(static_cast<unsigned short>(vm)));
        const unsigned int vwmax = __reduce_max_sync(0xffffffffu, __float_as_uint(va));
        if (lane == 0) atomicMax(&blk_amax[par][2], vwmax);
      }
      const uint32_t st = sbase + T * kStreamStageBytes;
      float x[VPL];
      {
        uint4 raw[4];
#pragma unroll
        for (int v = 0; v < 4; ++v) raw[v] = ld_shared_v4(st + v * kStreamSlotStride + tid * 16);
        if (fwht) {
          // Signs (+1 = 0x01, -1 = 0xff) onto the 16-bit words: bit 7 of each
          // sign byte becomes the sign bit of its value (commutes with the
          // widening and, through the sign of each sine, with the rotary step).
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const uint4 m = *reinterpret_cast<const uint4*>(mt + v * 4);
            raw[v].x ^= m.x;
            raw[v].y ^= m.y;
            raw[v].z ^= m.z;
            raw[v].w ^= m.w;
          }
        }
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const uint32_t w4[4] = {raw[v].x, raw[v].y, raw[v].z, raw[v].w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            float2 f;
            if (fused) f = widen_butterfly<BF16IN>(w4[q]);
            else if constexpr (BF16IN) f = make_float2(__uint_as_float(w4[q] << 16), __uint_as_float(w4[q] & 0xffff0000u));
            else f = __half22float2(*reinterpret_cast<const __half2*>(&w4[q]));
            x[8 * v + 2 * q] = f.x;
            x[8 * v + 2 * q + 1] = f.y;
          }
        }
      }
      if constexpr (QK && ROPE) {
        // With the signs already on the inputs, pair (a, b) with signs (sa, sb)
        // takes the rotation with sin * sa * sb, which gives sa (a c - b s) and
        // sb (a s + b c), bit for bit (rounding is odd-symmetric).  Table
        // entries from the block's shared copy (zero past N).
        const int lb = rib * 4 + g;
        auto tab4 = [&](int k) -> float4 {
          const uint4 r = ld_shared_v4(tbase + (lb * 8 + (k ^ (lb & 7))) * 16);
          return make_float4(__uint_as_float(r.x), __uint_as_float(r.y), __uint_as_float(r.z), __uint_as_float(r.w));
        };
        if (p.rope_interleaved) {
          // Pairs (2i, 2i+1): elements j, j+1 of run v, i = 16 v + 4 g + j / 2.
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const float4 c4 = tab4(2 * v);
            float4 s4 = tab4(2 * v + 1);
            if (fwht) {
              const uint4 m = *reinterpret_cast<const uint4*>(mt + 16 + v * 4);
              s4.x = __uint_as_float(__float_as_uint(s4.x) ^ m.x);
              s4.y = __uint_as_float(__float_as_uint(s4.y) ^ m.y);
              s4.z = __uint_as_float(__float_as_uint(s4.z) ^ m.z);
              s4.w = __uint_as_float(__float_as_uint(s4.w) ^ m.w);
            }
            const float cc[4] = {c4.x, c4.y, c4.z, c4.w}, ss[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int e = 8 * v + 2 * q;
              const float a = x[e], b = x[e + 1];
              x[e] = fmaf(a, cc[q], -(b * ss[q]));
              x[e + 1] = fmaf(a, ss[q], b * cc[q]);
            }
          }
        } else {
          // Pairs (i, i + d/2): element j of run v and of run v + 2, i = 32 v + 8 g + j.
#pragma unroll
          for (int v = 0; v < 2; ++v) {
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const float4 c4 = tab4(2 * (2 * v + hh));
              const float4 s4 = tab4(2 * (2 * v + hh) + 1);
              const uint4 mm = fwht ? *reinterpret_cast<const uint4*>(mt + 16 + 8 * v + 4 * hh) : make_uint4(0u, 0u, 0u, 0u);
              const uint32_t m[4] = {mm.x, mm.y, mm.z, mm.w};
              const float sv[4] = {s4.x, s4.y, s4.z, s4.w}, cv[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
              for (int q = 0; q < 4; q += 2) {
                const int e = 8 * v + 4 * hh + q;
                const float2 sp = make_float2(__uint_as_float(__float_as_uint(sv[q]) ^ m[q]),
                                              __uint_as_float(__float_as_uint(sv[q + 1]) ^ m[q + 1]));
                const float2 sn = make_float2(-sp.x, -sp.y);
                const float2 a = pair(x, e), b = pair(x, e + 16);
                const float2 c2 = make_float2(cv[q], cv[q + 1]);
                put(x, e, ffma2(b, sn, fmul2(a, c2)));
                put(x, e + 16, ffma2(a, sp, fmul2(b, c2)));
              }
            }
          }
        }
      }

      if (fwht) {
        // Element bits 0 (scalar: the two halves of a register pair; done with
        // the widening when fused), 1, 2, 5, 6.
        if (!fused) {
#pragma unroll
          for (int e = 0; e < VPL; e += 2) {
            const float a = x[e], b = x[e + 1];
            x[e] = a + b;
            x[e + 1] = a - b;
          }
        }
#pragma unroll
        for (int m = 2; m < VPL; m <<= 1)
#pragma unroll
          for (int e = 0; e < VPL; e += 2)
            if ((e & m) == 0) {
              const float2 a = pair(x, e), b = pair(x, e + m);
              put(x, e, fadd2(a, b));
              put(x, e + m, fsub2(a, b));
            }
        // Transpose within the row's group: unit (run 4 a + b, half hh) of row rw
        // sits in segment a at byte rw * 64 + ((b ^ a) * 16) of the warp's
        // 512-byte share; the writer is lane b (a = its run v), the reader lane a.
        __syncwarp();  // every lane has read its own slots
        const uint32_t wbase = st + warp * 512 + rw * 64;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const int e = 8 * v + 4 * hh;
            st_shared_v4(wbase + v * kStreamSlotStride + ((g ^ v) << 4), __float_as_uint(x[e]),
                         __float_as_uint(x[e + 1]), __float_as_uint(x[e + 2]), __float_as_uint(x[e + 3]));
          }
          __syncwarp();
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint4 r = ld_shared_v4(wbase + g * kStreamSlotStride + ((k ^ g) << 4));
            const int e = 8 * k + 4 * hh;
            x[e] = __uint_as_float(r.x);
            x[e + 1] = __uint_as_float(r.y);
            x[e + 2] = __uint_as_float(r.z);
            x[e + 3] = __uint_as_float(r.w);
          }
          __syncwarp();
        }
        // Element bits 3 and 4 (register index bits 3 and 4 of 32 g + e).
#pragma unroll
        for (int m = 8; m < VPL; m <<= 1)
#pragma unroll
          for (int e = 0; e < VPL; e += 2)
            if ((e & m) == 0) {
              const float2 a = pair(x, e), b = pair(x, e + m);
              put(x, e, fadd2(a, b));
              put(x, e + m, fsub2(a, b));
            }
      }

      // Block maximum of |x|.  Q and K: max and min over four independent
      // chains (no per-value absolute value), the warp's maximum on the float
      // bits (non-negative values order as unsigned integers), one shared
      // atomic per warp and one barrier.  V has no barrier of its own: the K
      // step takes V's maximum from its 16-bit words (|x| orders as the bits
      // without the sign, read as unsigned) and its barrier publishes both.
      if constexpr (QK) {
        float mx[4], mn[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          mx[c] = fmaxf(x[8 * c], x[8 * c + 1]);
          mn[c] = fminf(x[8 * c], x[8 * c + 1]);
#pragma unroll
          for (int e = 8 * c + 2; e < 8 * c + 8; e += 2) {
            mx[c] = max3(mx[c], x[e], x[e + 1]);
            mn[c] = min3(mn[c], x[e], x[e + 1]);
          }
        }
        const float m = fmaxf(max3(mx[0], mx[1], mx[2]), mx[3]);
        const float n = fminf(min3(mn[0], mn[1], mn[2]), mn[3]);
        const unsigned int wmax = __reduce_max_sync(0xffffffffu, __float_as_uint(fmaxf(m, -n)) & 0x7fffffffu);
        if (lane == 0) atomicMax(&blk_amax[par][T], wmax);
        __syncthreads();
        // Unit u - 1 read its maxima before this barrier; unit u + 1 adds to them
        // only after the K barrier, which these threads reach after the reset.
        if (T == 0 && tid < 3) blk_amax[par ^ 1][tid] = 0u;
      }
      float amax = __uint_as_float(blk_amax[par][T]);
      const float amax_u = amax;  // with the rotation: the maximum before 1 / sqrt(d)
      if (fwht) amax *= kInvSqrtD;
      // Ordinary maxima take s by the FMA-corrected quotient and the codes by
      // products; the rest (uniform over the CTA) divide.
      const bool fast = __all_sync(0xffffffffu, amax >= 0x1p-90f && amax <= 0x1p+100f);
      const float s = fast ? div_corrected(amax, kE4M3Max, 1.0f / kE4M3Max) : (amax > 0.f ? amax / kE4M3Max : 1.f);
      if (tid == 0) p.scale[T][cur.bh * p.nblk + cur.blk] = s;
      const int row = cur.blk * kQuantRows + rib;
      const bool have = row < p.N;
      uint8_t* dst = p.dst[T] + (static_cast<size_t>(cur.bh) * p.N + (have ? row : 0)) * D;
      // Codes are packed four to a word and stored as soon as a store's words
      // are ready (rotated rows: lane g holds bytes 32 g ..; otherwise the four
      // 8-byte runs 32 v + 8 g ..).
      auto pack4 = [](float2 a, float2 b) -> uint32_t {
        return __nv_cvt_float2_to_fp8x2(a, __NV_SATFINITE, __NV_E4M3) |
               (static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(b, __NV_SATFINITE, __NV_E4M3)) << 16);
      };
      if (fast && fwht) {
        // Rotated rows (float32 butterflies, compared within one E4M3 step):
        // x / (sqrt(d) s) as x times 448 / amax_u, from the hardware reciprocal
        // (within a few float32 roundings of the quotient), so the path from
        // the barrier to the codes is one reciprocal and products.
        float r;
        asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(amax_u));
        const float yds = r * kE4M3Max;
        const float2 y2 = make_float2(yds, yds);
        uint32_t wk[4];
#pragma unroll
        for (int o = 0; o < 2; ++o) {
          uint32_t w[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int e = 16 * o + 4 * q;
            w[q] = pack4(fmul2(pair(x, e), y2), fmul2(pair(x, e + 2), y2));
          }
          if (have) {
            if (p.codes_align32) {
              // Lane g's 32 code bytes in one store, so each store fills whole sectors.
              if (o == 0) {
                wk[0] = w[0]; wk[1] = w[1]; wk[2] = w[2]; wk[3] = w[3];
              } else {
                st_global_v8(dst + 32 * g, wk[0], wk[1], wk[2], wk[3], w[0], w[1], w[2], w[3]);
              }
            } else {
              reinterpret_cast<uint4*>(dst + 32 * g)[o] = make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
        }
      } else if (fast) {
        // -RN(x / s) by the FMA correction taken on the negated product, then
        // the codes' sign bits flipped (E4M3 is sign-magnitude and its rounding
        // symmetric): one product fewer per pair than div_by_scale2, zeros keep
        // their sign (x = -0: -q = +0, code 0x80).
        const float y = __frcp_rn(s);
        const float2 s2 = make_float2(s, s), ny2 = make_float2(-y, -y);
        auto neg_q = [&](int e) {
          const float2 xv = pair(x, e);
          const float2 q0n = fmul2(xv, ny2);
          return ffma2(ffma2(q0n, s2, xv), ny2, q0n);
        };
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const int e = 8 * v;
          const uint32_t w0 = pack4(neg_q(e), neg_q(e + 2)) ^ 0x80808080u;
          const uint32_t w1 = pack4(neg_q(e + 4), neg_q(e + 6)) ^ 0x80808080u;
          if (have) *reinterpret_cast<uint2*>(dst + 32 * v + 8 * g) = make_uint2(w0, w1);
        }
      } else {
        const float c = fwht ? kInvSqrtD : 1.f;
        uint32_t pk[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float2 q01 = make_float2(__fdiv_rn(x[4 * q] * c, s), __fdiv_rn(x[4 * q + 1] * c, s));
          const float2 q23 = make_float2(__fdiv_rn(x[4 * q + 2] * c, s), __fdiv_rn(x[4 * q + 3] * c, s));
          pk[q] = pack4(q01, q23);
        }
        if (have) {
          if (fwht) {
            uint4* out = reinterpret_cast<uint4*>(dst + 32 * g);
            out[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            out[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
          } else {
#pragma unroll
            for (int v = 0; v < 4; ++v)
              *reinterpret_cast<uint2*>(dst + 32 * v + 8 * g) = make_uint2(pk[2 * v], pk[2 * v + 1]);
          }
        }
      }
      if constexpr (T == 0) {
        // The next unit's sign masks into the other slot: its last reader,
        // unit u - 1, finished before the previous K barrier, and this unit's
        // K barrier publishes it.
        if (rotate && tid < kMaskWords && u + 1 < end) {
          const int hn = cur.h + 1 == p.H ? 0 : cur.h + 1;
          mask_tab[par ^ 1][mask_slot(tid)] = sign_mask_word(p.signs + hn * D, tid, p.rope_interleaved != 0);
        }
      }
    };
    step(std::integral_constant<int, 0>());
    step(std::integral_constant<int, 1>());
    step(std::integral_constant<int, 2>());
    next_unit(cur, p.BH, p.H);
  }
}

// Per-tensor mode: the scale slot held the tensor amax (as bits); turn it into s.
__global__ void fp8_finalize_scale_kernel(float* q_scale, float* k_scale, float* v_scale) {
  float* sc[3] = {q_scale, k_scale, v_scale};
  if (threadIdx.x < 3) {
    const float g = __uint_as_float(*reinterpret_cast<unsigned int*>(sc[threadIdx.x]));
    *sc[threadIdx.x] = g > 0.f ? g / kE4M3Max : 1.f;
  }
}

// d = 128, per-block scales: the streaming pre-pass (two CTAs per SM; the rotary kernel one).
template <bool BF16IN, bool ROPE, bool ROTATE>
attn_status run_prepare_stream(const PrepParams& prm, cudaStream_t s) {
  constexpr int smem = kStreamSmemBytes + (ROPE ? kStreamTableBytes : 0);
  static int configured_for[64] = {0};  // per device: dynamic shared memory attribute set
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return attn_internal::cuda_status(e);
  if (dev >= 64 || !configured_for[dev]) {
    e = cudaFuncSetAttribute(fp8_prepare_stream_kernel<BF16IN, ROPE, ROTATE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem);
    if (e != cudaSuccess) return attn_internal::cuda_status(e);
    if (dev < 64) configured_for[dev] = 1;
  }
  const int sms = attn_internal::sm_count();
  if (sms <= 0) return ATTN_ERR_CUDA;
  const int n_units = prm.BH * prm.nblk;  // (row block, head) units, three steps each
  const int per_sm = ROPE ? 1 : 2;  // the rotary kernel keeps its block's tables in shared memory
  const int grid = n_units < per_sm * sms ? n_units : per_sm * sms;
  fp8_prepare_stream_kernel<BF16IN, ROPE, ROTATE><<<grid, kPrepThreads, smem, s>>>(prm, n_units);
  return attn_internal::cuda_status(cudaGetLastError());
}

template <int D, bool BF16IN>
attn_status run_prepare_d(const PrepParams& prm, int per_tensor, cudaStream_t s) {
  const dim3 grid(static_cast<unsigned>(prm.BH) * prm.nblk, 3);
  if constexpr (D == kStreamD) {
    if (!per_tensor && static_cast<long long>(prm.BH) * prm.N < 0x7fffffffll)
    {
      const bool rope = prm.rcos != nullptr, rot = prm.signs != nullptr;
      if (rope) return rot ? run_prepare_stream<BF16IN, true, true>(prm, s) : run_prepare_stream<BF16IN, true, false>(prm, s);
      return rot ? run_prepare_stream<BF16IN, false, true>(prm, s) : run_prepare_stream<BF16IN, false, false>(prm, s);
    }
  }
  if (!per_tensor) {
    fp8_prepare_kernel<D, BF16IN, PREP_BLOCK><<<grid, kPrepThreads, 0, s>>>(prm);
    return attn_internal::cuda_status(cudaGetLastError());
  }
  for (int t = 0; t < 3; ++t) {
    cudaError_t e = cudaMemsetAsync(prm.scale[t], 0, sizeof(float), s);
    if (e != cudaSuccess) return attn_internal::cuda_status(e);
  }
  fp8_prepare_kernel<D, BF16IN, PREP_AMAX><<<grid, kPrepThreads, 0, s>>>(prm);
  fp8_prepare_kernel<D, BF16IN, PREP_QUANT_GLOBAL><<<grid, kPrepThreads, 0, s>>>(prm);
  fp8_finalize_scale_kernel<<<1, 32, 0, s>>>(prm.scale[0], prm.scale[1], prm.scale[2]);
  return attn_internal::cuda_status(cudaGetLastError());
}

template <bool BF16IN>
attn_status run_prepare(const PrepParams& prm, int d, int per_tensor, cudaStream_t s) {
  switch (d) {
    case 64: return run_prepare_d<64, BF16IN>(prm, per_tensor, s);
    case 128: return run_prepare_d<128, BF16IN>(prm, per_tensor, s);
    default: return run_prepare_d<256, BF16IN>(prm, per_tensor, s);
  }
}

// Head dimensions of the FP8 pre-pass, and of the FP8 attention kernel.
bool prep_head_dim(int d) { return d == 64 || d == 128 || d == 256; }
bool fwd_fp8_head_dim(int d) { return d == 64 || d == 128 || d == 256; }

// One CTA of 128 threads: thread r puts row r of x (COLS = 32 or 128 floats)
// into TMEM lane r and reads it back with the reducing load the attention
// softmax uses for its row maximum (tmem_ld32_red, or tmem_ld128_red for the
// whole 128-column row), then writes the values and the extreme (maximum, or
// minimum with MIN).
template <bool MIN, int COLS>
__global__ void debug_tmem_red_kernel(const float* x, float* vals, float* ext) {
  __shared__ uint32_t slot;
  const int warp = threadIdx.x >> 5, row = threadIdx.x;
  if (warp == 0) {
    tmem_alloc(smem_u32(&slot), COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = slot;
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
#pragma unroll
  for (int c = 0; c < COLS / 32; ++c) {
    uint32_t v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(x[row * COLS + 32 * c + i]);
    tmem_st32(lane_base + 32 * c, v);
  }
  tmem_wait_st();
  uint32_t r[4][32];
  float e[4] = {0.f, 0.f, 0.f, 0.f};
  if constexpr (COLS == 128)
    tmem_ld128_red<MIN>(lane_base, r, e[0]);
  else
    tmem_ld32_red<MIN>(lane_base, r[0], e[0]);
  tmem_wait_ld(r[0]);
#pragma unroll
  for (int c = 1; c < COLS / 32; ++c) reg_pin(r[c]);
  reg_pin(e);
#pragma unroll
  for (int c = 0; c < COLS / 32; ++c)
#pragma unroll
    for (int i = 0; i < 32; ++i) vals[row * COLS + 32 * c + i] = __uint_as_float(r[c][i]);
  ext[row] = e[0];
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, COLS);
  }
}

attn_status check_common(int B, int H, int N) {
  if (B < 0 || H < 0 || N < 0) return ATTN_ERR_INVALID_ARG;
  if (static_cast<int64_t>(B) * H > 0x7fffffff / 64) return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

}  // namespace

namespace attn_internal {
cudaError_t fp8_status_exchange(unsigned int* out) { return attn_kernel::status_exchange(out); }
}  // namespace attn_internal

ATTN_EXPORT attn_status attn_debug_tmem_ld_red(const float* x, float* vals, float* ext, int cols, int use_min,
                                              void* stream) {
  if (!x || !vals || !ext || (cols != 32 && cols != 128)) return ATTN_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cols == 128) {
    if (use_min)
      debug_tmem_red_kernel<true, 128><<<1, 128, 0, s>>>(x, vals, ext);
    else
      debug_tmem_red_kernel<false, 128><<<1, 128, 0, s>>>(x, vals, ext);
  } else if (use_min) {
    debug_tmem_red_kernel<true, 32><<<1, 128, 0, s>>>(x, vals, ext);
  } else {
    debug_tmem_red_kernel<false, 32><<<1, 128, 0, s>>>(x, vals, ext);
  }
  return attn_internal::cuda_status(cudaGetLastError());
}

ATTN_EXPORT attn_status attn_fp8_prepare_rotary(const void* q, const void* k, const void* v,
                                                attn_dtype in_dtype, void* q8, void* k8, void* v8,
                                                float* q_scale, float* k_scale, float* v_scale,
                                                const int8_t* signs, int per_tensor, const float* rope_cos,
                                                const float* rope_sin, int rope_interleaved, int B, int H,
                                                int N, int d, void* stream) {
  attn_status st = check_common(B, H, N);
  if (st != ATTN_OK) return st;
  if (!prep_head_dim(d)) return ATTN_ERR_UNSUPPORTED;
  if (in_dtype != ATTN_FP16 && in_dtype != ATTN_BF16) return ATTN_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(B) * H * ((N + kQuantRows - 1) / kQuantRows) > 0x7fffffff) return ATTN_ERR_INVALID_ARG;
  if ((rope_cos == nullptr) != (rope_sin == nullptr)) return ATTN_ERR_INVALID_ARG;
  if (static_cast<int64_t>(B) * H * N == 0) return ATTN_OK;
  if (!q || !k || !v || !q8 || !k8 || !v8 || !q_scale || !k_scale || !v_scale) return ATTN_ERR_INVALID_ARG;
  using attn_internal::aligned;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(q8, 16) || !aligned(k8, 16) ||
      !aligned(v8, 16))
    return ATTN_ERR_MISALIGNED;
  if (!aligned(q_scale, 4) || !aligned(k_scale, 4) || !aligned(v_scale, 4)) return ATTN_ERR_MISALIGNED;
  if (signs && !aligned(signs, 16)) return ATTN_ERR_MISALIGNED;  // read 16 signs per load
  if (rope_cos && (!aligned(rope_cos, 16) || !aligned(rope_sin, 16))) return ATTN_ERR_MISALIGNED;
  PrepParams prm;
  prm.src[0] = q; prm.src[1] = k; prm.src[2] = v;
  prm.dst[0] = static_cast<uint8_t*>(q8);
  prm.dst[1] = static_cast<uint8_t*>(k8);
  prm.dst[2] = static_cast<uint8_t*>(v8);
  prm.scale[0] = q_scale; prm.scale[1] = k_scale; prm.scale[2] = v_scale;
  prm.signs = signs;
  prm.rcos = rope_cos;
  prm.rsin = rope_sin;
  prm.rope_interleaved = rope_interleaved ? 1 : 0;
  prm.H = H;
  prm.N = N;
  prm.nblk = (N + kQuantRows - 1) / kQuantRows;
  prm.BH = B * H;
  prm.codes_align32 = attn_internal::aligned(q8, 32) && attn_internal::aligned(k8, 32);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return in_dtype == ATTN_BF16 ? run_prepare<true>(prm, d, per_tensor, s)
                               : run_prepare<false>(prm, d, per_tensor, s);
}

ATTN_EXPORT attn_status attn_fp8_prepare(const void* q, const void* k, const void* v, attn_dtype in_dtype,
                                         void* q8, void* k8, void* v8, float* q_scale, float* k_scale,
                                         float* v_scale, const int8_t* signs, int per_tensor, int B,
                                         int H, int N, int d, void* stream) {
  return attn_fp8_prepare_rotary(q, k, v, in_dtype, q8, k8, v8, q_scale, k_scale, v_scale, signs,
                                 per_tensor, nullptr, nullptr, 0, B, H, N, d, stream);
}

ATTN_EXPORT attn_status attn_fwd_fp8_ws(const void* q8, const void* k8, const void* v8, const float* q_scale,
                                        const float* k_scale, const float* v_scale, int per_tensor, void* o,
                                        float* lse, int B, int H, int N, int d, int causal, float scale,
                                        void* workspace, size_t workspace_bytes, void* stream) {
  attn_status st = check_common(B, H, N);
  if (st != ATTN_OK) return st;
  if (!fwd_fp8_head_dim(d)) return ATTN_ERR_UNSUPPORTED;
  if (!std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (static_cast<int64_t>(B) * H * N == 0) return ATTN_OK;
  if (!q8 || !k8 || !v8 || !o || !q_scale || !k_scale || !v_scale) return ATTN_ERR_INVALID_ARG;
  using attn_internal::aligned;
  if (!aligned(q8, 16) || !aligned(k8, 16) || !aligned(v8, 16) || !aligned(o, 16)) return ATTN_ERR_MISALIGNED;
  if (!aligned(q_scale, 4) || !aligned(k_scale, 4) || !aligned(v_scale, 4)) return ATTN_ERR_MISALIGNED;
  if (lse && !aligned(lse, 4)) return ATTN_ERR_MISALIGNED;
  FwdParams prm{};
  prm.o = o;
  prm.lse = lse;
  prm.causal = causal ? 1 : 0;
  prm.q_scale = q_scale;
  prm.k_scale = k_scale;
  prm.v_scale = v_scale;
  const int nblk = (N + kQuantRows - 1) / kQuantRows;
  prm.scale_bh_stride = per_tensor ? 0 : nblk;
  prm.scale_blk_stride = per_tensor ? 0 : 1;
  if (workspace != nullptr && !attn_internal::aligned(workspace, 256)) return ATTN_ERR_MISALIGNED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* w = workspace;
  const size_t wb = workspace_bytes;
  switch (d) {
    case 64: return attn_kernel::launch_fwd<64, KIND_E4M3>(q8, k8, v8, prm, B, H, N, N, scale, s, w, wb);
    case 128: return attn_kernel::launch_fwd<128, KIND_E4M3>(q8, k8, v8, prm, B, H, N, N, scale, s, w, wb);
    default: return attn_kernel::launch_fwd<256, KIND_E4M3>(q8, k8, v8, prm, B, H, N, N, scale, s, w, wb);
  }
}

ATTN_EXPORT attn_status attn_fwd_fp8(const void* q8, const void* k8, const void* v8, const float* q_scale,
                                     const float* k_scale, const float* v_scale, int per_tensor, void* o,
                                     float* lse, int B, int H, int N, int d, int causal, float scale,
                                     void* stream) {
  return attn_fwd_fp8_ws(q8, k8, v8, q_scale, k_scale, v_scale, per_tensor, o, lse, B, H, N, d, causal, scale,
                         nullptr, 0, stream);
}
