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

// E2M1 code of x for a positive scale s: round-to-nearest-even of x/s,
// saturating at 6, sign kept.  Decided by exact comparisons of |x| with the
// midpoints m*s (m in {0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5}; every m*s is an
// exact fp32 product of a <=3-bit and a 4-bit significand); at a midpoint the
// even code wins, so the comparison is '>' where the even code is below and
// '>=' where it is above.
__device__ __forceinline__ uint32_t e2m1_code(float x, float s) {
  const float a = fabsf(x);
  uint32_t m = 0;
  m += (a > 0.25f * s);
  m += (a >= 0.75f * s);
  m += (a > 1.25f * s);
  m += (a >= 1.75f * s);
  m += (a > 2.5f * s);
  m += (a >= 3.5f * s);
  m += (a > 5.0f * s);
  return m | ((__float_as_uint(x) >> 28) & 8u);
}

}  // namespace nvfp4idx
