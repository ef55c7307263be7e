// insert.cu -- NVFP4 quantise-and-scatter of index keys into the paged cache.
//
// The quantise half of the fused qk-norm/rope insert that writes the index-K
// side cache (vllm.models.minimax_m3.nvidia.indexer_nvfp4, module
// description).  One thread per (token, 16-element group): 8 threads cover a
// token's 256-byte bf16 row with two 16-byte loads each, and one 8-byte store
// of codes each; the group-0 thread gathers the 8 scale bytes with shuffles
// and stores them as one 8-byte word.  HBM-bound: 256 B read + 8 B slot +
// 72 B written per token.
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
  const int64_t tok = tid >> 3;
  const int g = (int)(tid & 7);
  const unsigned lane = threadIdx.x & 31u;
  const bool live = tok < n;
  int64_t slot = live ? __ldg(slots + tok) : -1;
  if (slot >= num_slots) {
    if (g == 0 && status) atomicOr(status, (int32_t)kStatusBadSlot);
    slot = -1;
  }

  uint32_t scale_byte = 0;
  uint32_t lo = 0, hi = 0;
  if (slot >= 0) {
    const uint4* src = reinterpret_cast<const uint4*>(k + tok * 128 + g * 16);
    const uint4 v0 = __ldg(src), v1 = __ldg(src + 1);
    const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    float x[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
    // scale = E4M3(amax / 6), round-to-nearest-even; fl32(amax/6) never sits
    // on an E4M3 midpoint unless amax/6 itself does, so this equals rounding
    // the exact quotient.
    scale_byte = f32_to_e4m3_satfinite(__fdiv_rn(amax, 6.0f));
    const float s = e4m3_to_f32(scale_byte);
    uint32_t codes[16];
    if (s > 0.0f) {
#pragma unroll
      for (int i = 0; i < 16; ++i) codes[i] = e2m1_code(x[i], s);
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) codes[i] = (__float_as_uint(x[i]) >> 28) & 8u;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      lo |= (codes[2 * i] | (codes[2 * i + 1] << 4)) << (8 * i);
      hi |= (codes[8 + 2 * i] | (codes[8 + 2 * i + 1] << 4)) << (8 * i);
    }
  }
  // gather the 8 scale bytes of the token into the group-0 thread
  const unsigned base = lane & ~7u;
  uint32_t s_lo = 0, s_hi = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t b = __shfl_sync(0xffffffffu, scale_byte, base + j);
    if (j < 4) s_lo |= b << (8 * j);
    else s_hi |= b << (8 * (j - 4));
  }
  if (slot >= 0) {
    uint8_t* row = pages + slot * 72;
    *reinterpret_cast<uint2*>(row + g * 8) = make_uint2(lo, hi);
    if (g == 0) *reinterpret_cast<uint2*>(row + 64) = make_uint2(s_lo, s_hi);
  }
}

cudaError_t launch_insert(const uint16_t* k, const int64_t* slots, int n, uint8_t* pages,
                          int num_blocks, int32_t* status, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  const int64_t threads = (int64_t)n * 8;
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
// round-to-nearest-even of x / 2^E (exact comparisons of |x| with the
// midpoints times 2^E, saturating at 6).  One thread per (token, block): 4
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
    float x[32];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 v = __ldg(src + i);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        x[8 * i + 2 * h] = __uint_as_float(w[h] << 16);
        x[8 * i + 2 * h + 1] = __uint_as_float(w[h] & 0xFFFF0000u);
      }
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(x[i]));
    const int E = amax > 0.0f ? max(-127, min(127, floor_log2_f32(amax) - 2)) : -127;
    scale_byte = (uint32_t)(E + 127);
    const float s = exp2i_f32(E);
#pragma unroll
    for (int i = 0; i < 32; ++i) cw[i >> 3] |= e2m1_code(x[i], s) << (4 * (i & 7));
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
