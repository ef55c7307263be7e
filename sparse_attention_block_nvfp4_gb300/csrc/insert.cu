// insert.cu -- NVFP4 quantise-and-scatter of index keys into the paged cache.
//
// The quantise half of the fused qk-norm/rope insert that writes the index-K
// side cache (vllm.models.minimax_m3.nvidia.indexer_nvfp4, module
// description).  Four threads per token, each covering two 16-element groups
// (32 elements: four 16-byte loads, two 8-byte code stores); the j = 0
// thread gathers the token's 8 scale bytes with two shuffles and stores them
// as one 8-byte word.  The codes come from the hardware E2M1 conversion of a
// quotient rounded so that ties fall exactly (nvfp4_ratio), the scales from
// the E4M3 conversion of a 12-bit rounding of amax / 6 (e4m3_scale_of_amax).
// HBM-bound: 256 B read + 8 B slot + 72 B written per token.
#include <cstdint>
#include <cuda_runtime.h>

#include "codec.cuh"
#include "internal.h"

namespace nvfp4idx {

__global__ void __launch_bounds__(256) nvfp4_insert_kernel(const uint16_t* __restrict__ k,
                                                           const int64_t* __restrict__ slots,
                                                           int n, uint8_t* __restrict__ pages,
                                                           int64_t num_slots,
                                                           int32_t* __restrict__ status) {
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t tok = tid >> 2;
  const int j = (int)(tid & 3);
  const bool live = tok < n;
  int64_t slot = live ? __ldg(slots + tok) : -1;
  if (slot >= num_slots) {
    if (j == 0 && status) atomicOr(status, (int32_t)kStatusBadSlot);
    slot = -1;
  }

  uint32_t sc2 = 0;                  // scale bytes 2j (low) and 2j + 1
  uint32_t cw[4] = {0, 0, 0, 0};     // codes of elements 32j .. 32j + 31
  if (slot >= 0) {
    const uint4* src = reinterpret_cast<const uint4*>(k + tok * 128 + j * 32);
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 v = __ldg(src + i);
      w[4 * i] = v.x;
      w[4 * i + 1] = v.y;
      w[4 * i + 2] = v.z;
      w[4 * i + 3] = v.w;
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {   // group 2j + h, widened to fp32 only now
      uint32_t m = w[8 * h];
#pragma unroll
      for (int i = 1; i < 8; ++i) m = bf16x2_max_abs(m, w[8 * h + i]);
      const float amax = bf16x2_amax_f32(m);
      float xg[16];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        xg[2 * i] = __uint_as_float(w[8 * h + i] << 16);
        xg[2 * i + 1] = __uint_as_float(w[8 * h + i] & 0xFFFF0000u);
      }
      const uint32_t sb = e4m3_scale_of_amax(amax);
      const float s = e4m3_to_f32(sb);
      if (s > 0.0f) {
        const float r = rcp_approx(s);
#pragma unroll
        for (int i = 0; i < 16; ++i) xg[i] = nvfp4_ratio(xg[i], r);
      } else {                       // zero scale: sign-only zero codes
#pragma unroll
        for (int i = 0; i < 16; ++i) xg[i] = __uint_as_float(__float_as_uint(xg[i]) & 0x80000000u);
      }
      sc2 |= sb << (8 * h);
      cw[2 * h] = f32x8_to_e2m1x8(xg);
      cw[2 * h + 1] = f32x8_to_e2m1x8(xg + 8);
    }
  }
  // the token's 4 threads are lanes 4c .. 4c+3 of one warp: pair up the
  // scale halves, then bring lanes 4c+2..3's pair to lane 4c
  const uint32_t pair = sc2 | (__shfl_down_sync(0xffffffffu, sc2, 1) << 16);
  const uint32_t upper = __shfl_down_sync(0xffffffffu, pair, 2);
  if (slot >= 0) {
    uint8_t* row = pages + slot * 72;
    uint2* dst = reinterpret_cast<uint2*>(row + j * 16);
    dst[0] = make_uint2(cw[0], cw[1]);
    dst[1] = make_uint2(cw[2], cw[3]);
    if (j == 0) *reinterpret_cast<uint2*>(row + 64) = make_uint2(pair, upper);
  }
}

cudaError_t launch_insert(const uint16_t* k, const int64_t* slots, int n, uint8_t* pages,
                          int num_blocks, int32_t* status, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  const int64_t threads = (int64_t)n * 4;
  const int block = 256;
  const int64_t grid = (threads + block - 1) / block;
  nvfp4_insert_kernel<<<(unsigned)grid, block, 0, stream>>>(k, slots, n, pages,
                                                             (int64_t)num_blocks * 128, status);
  return cudaGetLastError();
}

// MXFP4 quantise-and-scatter into [num_blocks, 8704] pages (codes of token
// t at 64 t, its four E8M0 scales at 8192 + 4 t; page
// vllm.models.minimax_m3.amd.indexer_mxfp4).  The conversion is the OCP
// microscaling one: per 32-element block the shared exponent is
// floor(log2(amax)) - 2 clamped to [-127, 127], each element the E2M1
// round-to-nearest-even of x / 2^E, saturating at 6 (the power-of-two
// quotient is exact in fp32, so the hardware conversion rounds the exact
// value).  One thread per (token, block): 4
// threads cover a token's 256-byte row with four 16-byte loads each and
// store 16 bytes of codes each; the block-0 thread gathers the 4 scale
// bytes with shuffles.  HBM-bound: 256 B read + 8 B slot + 68 B written per
// token.
__global__ void __launch_bounds__(256) mxfp4_insert_kernel(const uint16_t* __restrict__ k,
                                                           const int64_t* __restrict__ slots,
                                                           int n, uint8_t* __restrict__ pages,
                                                           int64_t num_slots,
                                                           int32_t* __restrict__ status) {
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t tok = tid >> 2;
  const int j = (int)(tid & 3);
  const unsigned lane = threadIdx.x & 31u;
  const bool live = tok < n;
  int64_t slot = live ? __ldg(slots + tok) : -1;
  if (slot >= num_slots) {
    if (j == 0 && status) atomicOr(status, (int32_t)kStatusBadSlot);
    slot = -1;
  }
  uint32_t scale_byte = 0;
  uint32_t cw[4] = {0, 0, 0, 0};
  if (slot >= 0) {
    const uint4* src = reinterpret_cast<const uint4*>(k + tok * 128 + j * 32);
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 v = __ldg(src + i);
      w[4 * i] = v.x;
      w[4 * i + 1] = v.y;
      w[4 * i + 2] = v.z;
      w[4 * i + 3] = v.w;
    }
    uint32_t m = w[0];
#pragma unroll
    for (int i = 1; i < 16; ++i) m = bf16x2_max_abs(m, w[i]);
    const float amax = bf16x2_amax_f32(m);
    const int E = amax > 0.0f ? max(-127, min(127, floor_log2_f32(amax) - 2)) : -127;
    scale_byte = (uint32_t)(E + 127);
    const float r = exp2i_f32(-E);   // x * 2^-E is exact (or underflows to a signed zero)
#pragma unroll
    for (int i = 0; i < 4; ++i) {    // 8 elements at a time, widened to fp32 only now
      float x[8];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        x[2 * h] = __fmul_rn(__uint_as_float(w[4 * i + h] << 16), r);
        x[2 * h + 1] = __fmul_rn(__uint_as_float(w[4 * i + h] & 0xFFFF0000u), r);
      }
      cw[i] = f32x8_to_e2m1x8(x);
    }
  }
  // gather the 4 scale bytes of the token into the block-0 thread
  const unsigned base = lane & ~3u;
  uint32_t s4 = 0;
#pragma unroll
  for (int b = 0; b < 4; ++b) s4 |= __shfl_sync(0xffffffffu, scale_byte, base + b) << (8 * b);
  if (slot >= 0) {
    uint8_t* page = pages + (slot >> 7) * (int64_t)(128 * 64 + 128 * 4);
    const int row = (int)(slot & 127);
    *reinterpret_cast<uint4*>(page + row * 64 + j * 16) = make_uint4(cw[0], cw[1], cw[2], cw[3]);
    if (j == 0) *reinterpret_cast<uint32_t*>(page + 128 * 64 + row * 4) = s4;
  }
}

cudaError_t launch_insert_mxfp4(const uint16_t* k, const int64_t* slots, int n, uint8_t* pages,
                                int num_blocks, int32_t* status, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  const int64_t threads = (int64_t)n * 4;
  const int block = 256;
  const int64_t grid = (threads + block - 1) / block;
  mxfp4_insert_kernel<<<(unsigned)grid, block, 0, stream>>>(k, slots, n, pages,
                                                             (int64_t)num_blocks * 128, status);
  return cudaGetLastError();
}

}  // namespace nvfp4idx
