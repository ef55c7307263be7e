// codec.cuh -- exact NVFP4 / E4M3 conversions on the device.
//
// Page format (vllm.models.minimax_m3.nvidia.indexer_nvfp4, module
// description): per token 64 bytes of E2M1 codes (element e in byte e/2, low
// nibble for even e) then 8 E4M3 scales, scale j for elements 16j..16j+15.
//
// Exactness: an E2M1 magnitude has at most 2 significant bits and an E4M3
// value at most 4, so a dequantised key c*s has at most 6 significant bits and
// lies in [2^-10, 2688]; every such value, and every E4M3 query value, is an
// fp16 normal number.  fp16 products below are therefore exact, and so are
// the fp16 x fp16 products the tensor core forms.
#pragma once
#include <cstdint>
#include <cuda_fp16.h>

namespace nvfp4idx {

// Two E2M1 codes (one byte, low nibble first) -> f16x2 {lo: low nibble,
// hi: high nibble}.
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t out;
  asm("{\n\t.reg .b8 b;\n\tcvt.u8.u32 b, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b;\n\t}" : "=r"(out) : "r"(byte));
  return out;
}

// Four E2M1 byte-pairs packed in a 32-bit word -> four f16x2 words
// (elements 0..7 of the word, in order).
__device__ __forceinline__ void e2m1x8_to_f16x2x4(uint32_t w, uint32_t& o0, uint32_t& o1,
                                                  uint32_t& o2, uint32_t& o3) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(o0), "=r"(o1), "=r"(o2), "=r"(o3)
      : "r"(w));
}

// Two E4M3 bytes (low byte first) -> f16x2.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
  uint32_t out;
  asm("{\n\t.reg .b16 h;\n\tcvt.u16.u32 h, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, h;\n\t}" : "=r"(out) : "r"(two_bytes));
  return out;
}

// f16x2 product, round-to-nearest (exact for the operands used here).
__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Broadcast the low (sel=0) or high (sel=1) half of an f16x2 to both halves.
__device__ __forceinline__ uint32_t f16x2_bcast_lo(uint32_t v) { return __byte_perm(v, 0, 0x1010); }
__device__ __forceinline__ uint32_t f16x2_bcast_hi(uint32_t v) { return __byte_perm(v, 0, 0x3232); }

// Dequantise 16 elements that share one scale: 8 code bytes (two words) and
// the scale already broadcast as f16x2 -> 8 f16x2 words (elements in order).
__device__ __forceinline__ void dequant16(uint32_t c0, uint32_t c1, uint32_t s2, uint32_t* o) {
  e2m1x8_to_f16x2x4(c0, o[0], o[1], o[2], o[3]);
  e2m1x8_to_f16x2x4(c1, o[4], o[5], o[6], o[7]);
#pragma unroll
  for (int i = 0; i < 8; ++i) o[i] = hmul2_u32(o[i], s2);
}

// ---------------------------------------------------------------- MXFP4
// (page vllm.models.minimax_m3.amd.indexer_mxfp4: e2m1 codes with e8m0
// scales, one per 32 elements.)  A code times 2^(s - 127) has at most two
// significant bits and an exponent anywhere in E8M0's range, so the exact
// operand type is bf16 (fp16's exponent range is too small); E4M3 queries
// are exact in bf16 too.

// f16x2 -> bf16x2 for values that bf16 holds exactly (all here do).
__device__ __forceinline__ uint32_t f16x2_to_bf16x2(uint32_t h2) {
  const float lo = __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
  const float hi = __half2float(__ushort_as_half((unsigned short)(h2 >> 16)));
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));   // first source -> high half
  return r;
}
// Two E8M0 bytes (low byte first) -> bf16x2 {2^(lo - 127), 2^(hi - 127)};
// 0xFF -> NaN.  bf16 holds every E8M0 value (2^-127 as a subnormal).
__device__ __forceinline__ uint32_t e8m0x2_to_bf16x2(uint32_t two_bytes) {
  uint32_t out;
  asm("{\n\t.reg .b16 h;\n\tcvt.u16.u32 h, %1;\n\tcvt.rn.bf16x2.ue8m0x2 %0, h;\n\t}" : "=r"(out) : "r"(two_bytes));
  return out;
}
// bf16x2 product, round-to-nearest (exact for the operands used here).
__device__ __forceinline__ uint32_t bmul2_u32(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// 16 MXFP4 elements sharing one scale: 8 code bytes (two words) and the
// scale already broadcast as bf16x2 -> 8 bf16x2 words (elements in order).
__device__ __forceinline__ void dequant16_mx(uint32_t c0, uint32_t c1, uint32_t s2, uint32_t* o) {
  uint32_t h[8];
  e2m1x8_to_f16x2x4(c0, h[0], h[1], h[2], h[3]);
  e2m1x8_to_f16x2x4(c1, h[4], h[5], h[6], h[7]);
#pragma unroll
  for (int i = 0; i < 8; ++i) o[i] = bmul2_u32(f16x2_to_bf16x2(h[i]), s2);
}
// floor(log2(a)) of a positive finite fp32 (normal or subnormal).
__device__ __forceinline__ int floor_log2_f32(float a) {
  const uint32_t u = __float_as_uint(a);
  const int e = (int)(u >> 23);
  if (e > 0) return e - 127;
  return (31 - __clz((int)(u & 0x7FFFFFu))) - 149;   // m * 2^-149
}
// 2^E as fp32 for E in [-127, 127] (2^-127 is a subnormal).
__device__ __forceinline__ float exp2i_f32(int E) {
  return E >= -126 ? __uint_as_float((uint32_t)(E + 127) << 23) : __uint_as_float(1u << 22);
}

// ------------------------------------------------------ page formats
// What the scoring kernels need from a page format: the page size the TMA
// unit copies, the MMA operand type, the queries widened to it, and one
// token's 128 elements as 64 words of that type, 16 elements at a time.
struct Nvfp4Pages {   // [num_blocks, 128, 72]: token rows of 64 code bytes + 8 E4M3 scales
  static constexpr uint32_t kPageBytes = 128 * 72;
  static constexpr bool kBf16 = false;
  struct Row {
    uint32_t w[16];   // code words
    uint32_t sc[4];   // scale pairs as f16x2 {scale 2j, scale 2j+1}
  };
  __device__ static __forceinline__ void load(const uint8_t* page, int tok, Row& r) {
    const uint2* src = reinterpret_cast<const uint2*>(page + tok * 72);
    uint32_t s01 = 0, s23 = 0;
#pragma unroll
    for (int i = 0; i < 9; ++i) {
      const uint2 t2 = src[i];
      if (i < 8) {
        r.w[2 * i] = t2.x;
        r.w[2 * i + 1] = t2.y;
      } else {
        s01 = t2.x;
        s23 = t2.y;
      }
    }
    r.sc[0] = e4m3x2_to_f16x2(s01 & 0xFFFFu);
    r.sc[1] = e4m3x2_to_f16x2(s01 >> 16);
    r.sc[2] = e4m3x2_to_f16x2(s23 & 0xFFFFu);
    r.sc[3] = e4m3x2_to_f16x2(s23 >> 16);
  }
  __device__ static __forceinline__ void chunk16(const Row& r, int g8, uint32_t* o) {
    const uint32_t s2 = (g8 & 1) ? f16x2_bcast_hi(r.sc[g8 >> 1]) : f16x2_bcast_lo(r.sc[g8 >> 1]);
    dequant16(r.w[2 * g8], r.w[2 * g8 + 1], s2, o);
  }
  __device__ static __forceinline__ uint32_t widen_q(uint32_t two_e4m3) { return e4m3x2_to_f16x2(two_e4m3); }
};

struct Mxfp4Pages {   // [num_blocks, 8704]: 128 x 64 code bytes, then 128 x 4 E8M0 scales
  static constexpr uint32_t kPageBytes = 128 * 64 + 128 * 4;
  static constexpr bool kBf16 = true;
  struct Row {
    uint32_t w[16];   // code words
    uint32_t sc[4];   // scale j (elements 32j .. 32j+31) broadcast as bf16x2
  };
  __device__ static __forceinline__ void load(const uint8_t* page, int tok, Row& r) {
    const uint4* src = reinterpret_cast<const uint4*>(page + tok * 64);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 t4 = src[i];
      r.w[4 * i] = t4.x;
      r.w[4 * i + 1] = t4.y;
      r.w[4 * i + 2] = t4.z;
      r.w[4 * i + 3] = t4.w;
    }
    const uint32_t s4 = *reinterpret_cast<const uint32_t*>(page + 128 * 64 + tok * 4);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t b = (s4 >> (8 * j)) & 0xFFu;
      r.sc[j] = e8m0x2_to_bf16x2(b | (b << 8));
    }
  }
  __device__ static __forceinline__ void chunk16(const Row& r, int g8, uint32_t* o) {
    dequant16_mx(r.w[2 * g8], r.w[2 * g8 + 1], r.sc[g8 >> 1], o);
  }
  __device__ static __forceinline__ uint32_t widen_q(uint32_t two_e4m3) {
    return f16x2_to_bf16x2(e4m3x2_to_f16x2(two_e4m3));
  }
};

// fp32 -> E4M3 byte, round-to-nearest-even, saturating to +-448.
__device__ __forceinline__ uint32_t f32_to_e4m3_satfinite(float x) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(x));
  return r & 0xFFu;   // second source operand lands in the low byte
}

// E4M3 byte -> fp32 (exact, via fp16).
__device__ __forceinline__ float e4m3_to_f32(uint32_t byte) {
  const uint32_t h2 = e4m3x2_to_f16x2(byte & 0xFFu);
  return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
}

// Eight fp32 values -> eight E2M1 codes in one word (element 0 in the low
// nibble), each the round-to-nearest-even of the value, saturating at +-6,
// the sign kept (a negative value that rounds to zero gives -0).
__device__ __forceinline__ uint32_t f32x8_to_e2m1x8(const float* v) {
  uint32_t out;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"   // second source -> low nibble
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(out)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
  return out;
}

// Per bf16 half: max(|a|, |b|), exact; the half's sign bit is the xor of
// the operands' signs (ignored by the callers).
__device__ __forceinline__ uint32_t bf16x2_max_abs(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// The larger magnitude of the two bf16 halves of a word, as fp32.
__device__ __forceinline__ float bf16x2_amax_f32(uint32_t m) {
  return fmaxf(fabsf(__uint_as_float(m << 16)), fabsf(__uint_as_float(m & 0xFFFF0000u)));
}

// 1/s to within one ulp, for a positive normal fp32 s.
__device__ __forceinline__ float rcp_approx(float s) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(s));
  return r;
}

// x / s for a bf16 value x and a positive E4M3 scale s, given r within one
// ulp of 1/s, in a form whose E2M1 rounding is that of the exact quotient
// t = |x| / s: one fused multiply-add rounds |x| r to a multiple of 2^-12
// (3 * 2^10 added has an ulp of 2^-12 while |x| r < 2^10), the addend is
// taken off exactly and the sign of x put back.
// Why it is exact: |x| = X 2^a (X < 2^8) and m s = M S 2^(b-2) for an E2M1
// midpoint m = M/4 (M <= 20) and s = S 2^b (S < 2^4) are multiples of
// 2^min(a, b-2), so t is either a midpoint or at least 2^-9 m >= 2^-11 away
// from each midpoint m nearer than m/2.  |x| r is within 2^-23 t < 2^-19 of
// t there, so at a midpoint (a multiple of 2^-12) the rounding returns it
// exactly, and elsewhere the result stays within 2^-19 + 2^-13 < 2^-11 of
// t: never across a midpoint.  Past 2^10 the quotient saturates either way.
__device__ __forceinline__ float nvfp4_ratio(float x, float r) {
  const float g = __fsub_rn(__fmaf_rn(fabsf(x), r, 3072.0f), 3072.0f);
  return __uint_as_float(__float_as_uint(g) | (__float_as_uint(x) & 0x80000000u));
}

// E4M3 byte of amax / 6, round-to-nearest-even of the exact quotient,
// saturating at 448, for a bf16 value amax >= 0.  v = amax * fl(1/6) is
// within 2^-23 of amax / 6 (relative; clamped at 1024, past which every
// value saturates); Veltkamp's split with the constant 2^12 + 1 rounds it to
// 12 significant bits.  An E4M3 midpoint u = U 2^e (U < 2^5) gives
// 6u = 3U 2^(e+1) with 3U < 2^7 and amax = A 2^a with A < 2^8, so amax / 6
// is either a midpoint (kept exactly by the 12-bit rounding) or at least
// 2^-9 away from it relative to its size, which the 2^-23 + 2^-12 moved
// does not cross; the hardware conversion then rounds as the exact value.
__device__ __forceinline__ uint32_t e4m3_scale_of_amax(float amax) {
  const float v = fminf(__fmul_rn(amax, 1.0f / 6.0f), 1024.0f);
  const float c = __fmul_rn(v, 4097.0f);
  const float hi = __fadd_rn(c, __fsub_rn(v, c));
  return f32_to_e4m3_satfinite(hi);
}

// One 16-element NVFP4 group of bf16-exact fp32 values xg (overwritten) with
// its amax: returns the E4M3 scale byte and leaves the 16 codes in c0, c1
// (element 0 in the low nibble of c0).  A zero scale gives sign-only codes.
__device__ __forceinline__ uint32_t nvfp4_encode16(float* xg, float amax, uint32_t& c0, uint32_t& c1) {
  const uint32_t sb = e4m3_scale_of_amax(amax);
  const float s = e4m3_to_f32(sb);
  if (s > 0.0f) {
    const float r = rcp_approx(s);
#pragma unroll
    for (int i = 0; i < 16; ++i) xg[i] = nvfp4_ratio(xg[i], r);
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) xg[i] = __uint_as_float(__float_as_uint(xg[i]) & 0x80000000u);
  }
  c0 = f32x8_to_e2m1x8(xg);
  c1 = f32x8_to_e2m1x8(xg + 8);
  return sb;
}

}  // namespace nvfp4idx
