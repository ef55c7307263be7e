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
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "codec.cuh"
#include "internal.h"

namespace nvfp4idx {

// Write one token's NVFP4 row from its 4 threads (lanes 4c .. 4c+3 of one
// warp, thread j holding the codes of elements 32j .. 32j+31 and scale bytes
// 2j, 2j+1 in sc2): the scale halves are paired up, lanes 4c+2..3's pair is
// brought to lane 4c, which stores the 8 scale bytes as one word.  Every
// lane of the warp must call it (shuffles); only slot >= 0 stores.
__device__ __forceinline__ void nvfp4_store_token(uint8_t* __restrict__ pages, int64_t slot, int j,
                                                  const uint32_t (&cw)[4], uint32_t sc2) {
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

__global__ void __launch_bounds__(256) nvfp4_insert_kernel(const uint16_t* __restrict__ k,
                                                           const int64_t* __restrict__ slots,
                                                           int n, uint8_t* __restrict__ pages,
                                                           int64_t num_slots,
                                                           int32_t* __restrict__ status) {
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t tok = tid >> 2;
  const int j = (int)(tid & 3);
  const bool live = tok < n;
  // the key's quarter and the slot load independently (one memory latency,
  // not two); a skipped token's key is read and dropped
  uint32_t w[16];
  if (live) {
    const uint4* src = reinterpret_cast<const uint4*>(k + tok * 128 + j * 32);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 v = __ldg(src + i);
      w[4 * i] = v.x;
      w[4 * i + 1] = v.y;
      w[4 * i + 2] = v.z;
      w[4 * i + 3] = v.w;
    }
  }
  int64_t slot = live ? __ldg(slots + tok) : -1;
  if (slot >= num_slots) {
    if (j == 0 && status) atomicOr(status, (int32_t)kStatusBadSlot);
    slot = -1;
  }

  uint32_t sc2 = 0;                  // scale bytes 2j (low) and 2j + 1
  uint32_t cw[4] = {0, 0, 0, 0};     // codes of elements 32j .. 32j + 31
  if (slot >= 0) {
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
      sc2 |= nvfp4_encode16(xg, amax, cw[2 * h], cw[2 * h + 1]) << (8 * h);
    }
  }
  nvfp4_store_token(pages, slot, j, cw, sc2);
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

// 16-byte asynchronous global -> shared copy (both addresses 16-byte
// aligned) and the waits for the calling thread's own copies.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(smem)),
               "l"(gmem)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// Modes of the fused insert, and the two 16-element groups gA < gB of the
// token that thread j holds in each: a NeoX pair (i, i + rd/2) must sit in
// one thread, as element i of group gA and element i of group gB.
enum { kNormOnly = 0, kNeox128 = 1, kNeox64 = 2, kGptj = 3 };
template <int kMode>
__device__ __forceinline__ void norm_rope_groups(int j, int& gA, int& gB) {
  if (kMode == kNeox128) {           // pairs (i, i + 64): groups j, j + 4
    gA = j;
    gB = j + 4;
  } else if (kMode == kNeox64) {     // pairs (i, i + 32) in groups 0..3; 4..7 pass through
    gA = j < 2 ? j : j + 2;
    gB = gA + 2;
  } else {                           // contiguous: elements 32j .. 32j + 31
    gA = 2 * j;
    gB = 2 * j + 1;
  }
}

// Sum of the 8 group sums t_g of a token in the fixed order
// ((t0 + t1) + (t2 + t3)) + ((t4 + t5) + (t6 + t7)), from lane j's tA =
// t_gA and tB = t_gB, on every lane of the token.
template <int kMode>
__device__ __forceinline__ float norm_rope_sumsq(float tA, float tB) {
  if (kMode == kNeox128) {           // lane j: t_j, t_{j+4}
    const float v = __fadd_rn(tA, __shfl_xor_sync(0xffffffffu, tA, 1));   // t0+t1 | t2+t3
    const float w = __fadd_rn(tB, __shfl_xor_sync(0xffffffffu, tB, 1));   // t4+t5 | t6+t7
    const float l = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 2));
    const float r = __fadd_rn(w, __shfl_xor_sync(0xffffffffu, w, 2));
    return __fadd_rn(l, r);
  } else if (kMode == kNeox64) {     // lanes: {0,2} {1,3} {4,6} {5,7}
    const float v = __fadd_rn(tA, __shfl_xor_sync(0xffffffffu, tA, 1));   // t0+t1 | t4+t5
    const float w = __fadd_rn(tB, __shfl_xor_sync(0xffffffffu, tB, 1));   // t2+t3 | t6+t7
    const float u = __fadd_rn(v, w);                                        // left | right half
    return __fadd_rn(u, __shfl_xor_sync(0xffffffffu, u, 2));
  } else {                           // lane j: t_{2j}, t_{2j+1}
    float u = __fadd_rn(tA, tB);
    u = __fadd_rn(u, __shfl_xor_sync(0xffffffffu, u, 1));
    return __fadd_rn(u, __shfl_xor_sync(0xffffffffu, u, 2));
  }
}

// One 16-element group of a token (two 16-byte words of bf16, loaded at
// entry) widened to fp32, and the group sum of squares t = e + o (even / odd
// running sums, one rounding per step).
__device__ __forceinline__ float norm_rope_widen_group(const uint4 (&v)[2], float (&x)[16]) {
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      x[8 * i + 2 * h] = __uint_as_float(w[h] << 16);
      x[8 * i + 2 * h + 1] = __uint_as_float(w[h] & 0xFFFF0000u);
    }
  }
  float e = 0.0f, o = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    e = __fmaf_rn(x[2 * i], x[2 * i], e);
    o = __fmaf_rn(x[2 * i + 1], x[2 * i + 1], o);
  }
  return __fadd_rn(e, o);
}

// y = (x * rs) * w for one group (w: the group's 16 bf16 weights).
__device__ __forceinline__ void norm_rope_scale_group(const uint16_t* wg, float rs, float (&x)[16]) {
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const uint4 wv = __ldg(reinterpret_cast<const uint4*>(wg) + i);
    const uint32_t w[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      x[8 * i + 2 * h] = __fmul_rn(__fmul_rn(x[8 * i + 2 * h], rs), __uint_as_float(w[h] << 16));
      x[8 * i + 2 * h + 1] = __fmul_rn(__fmul_rn(x[8 * i + 2 * h + 1], rs), __uint_as_float(w[h] & 0xFFFF0000u));
    }
  }
}

// bf16 rounding of one group, its amax from the bf16 words, the NVFP4
// codes (c0, c1) and the returned scale byte.
__device__ __forceinline__ uint32_t norm_rope_encode_group(float (&x)[16], uint32_t& c0, uint32_t& c1) {
  uint32_t R[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(R[i]) : "f"(x[2 * i + 1]), "f"(x[2 * i]));
  uint32_t mx = R[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) mx = bf16x2_max_abs(mx, R[i]);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    x[2 * i] = __uint_as_float(R[i] << 16);
    x[2 * i + 1] = __uint_as_float(R[i] & 0xFFFF0000u);
  }
  return nvfp4_encode16(x, bf16x2_amax_f32(mx), c0, c1);
}

// qk-norm + RoPE + NVFP4 quantise-and-scatter: the fused insert that writes
// the index-K side cache (vllm.models.minimax_m3.nvidia.indexer_nvfp4,
// module description).  Per token: RMSNorm over the 128 elements with a bf16
// weight, RoPE from the caller's cos/sin table at the token's position, the
// result rounded to bf16, then the NVFP4 quantiser above.  The fp32 steps
// run in one fixed order, so the keys are the same from run to run and
// differ from the exact qk-norm + RoPE by fp32 rounding only: per
// 16-element group g, running sums e_g / o_g of the even / odd elements'
// squares (one rounding per step: FFMA), t_g = e_g + o_g, ss = ((t0 + t1) +
// (t2 + t3)) + ((t4 + t5) + (t6 + t7)); v = ss/128 + eps; rs = 1 / sqrt(v),
// both correctly rounded; y = (x rs) w; each rotated pair (y1 c - y2 s,
// y2 c + y1 s) with every product and sum rounded (no fused multiply-add).
// Four threads per token, each holding two whole groups, chosen so that a
// NeoX pair (i, i + rd/2) sits in one thread (rd 64 or 128); GPT-J pairs
// (2i, 2i + 1) stay inside a thread anyway.  At entry each thread starts an
// asynchronous copy of its 16 cosines and 16 sines into shared memory, so the
// table's latency hides behind the norm; the key loads are issued first,
// independently of the slot and the position.  HBM-bound: 256 B
// key + 8 B slot + 8 B position + 72 B row per token, plus the table rows.
template <int kMode>
__global__ void __launch_bounds__(256) nvfp4_insert_norm_rope_kernel(const NormRopeArgs a) {
  // per thread: 16 cosines, 16 sines; rows padded to 36 floats so that the
  // 16-byte reads of 8 consecutive lanes fall on 8 different bank quads
  __shared__ __align__(16) float tab_s[256][36];
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t tok = tid >> 2;
  const int j = (int)(tid & 3);
  const bool live = tok < a.n;
  int gA, gB;
  norm_rope_groups<kMode>(j, gA, gB);
  // the key's two groups, the slot and the position load independently (a
  // skipped token's key is read and dropped)
  uint4 ka[2] = {}, kb[2] = {};
  if (live) {
    const uint4* kt = reinterpret_cast<const uint4*>(a.k + tok * 128);
    ka[0] = __ldg(kt + 2 * gA);
    ka[1] = __ldg(kt + 2 * gA + 1);
    kb[0] = __ldg(kt + 2 * gB);
    kb[1] = __ldg(kt + 2 * gB + 1);
  }
  int64_t slot = live ? __ldg(a.slots + tok) : -1;
  int64_t pos = (kMode != kNormOnly && live) ? __ldg(a.positions + tok) : 0;
  if (slot >= a.num_slots) {
    if (j == 0 && a.status) atomicOr(a.status, (int32_t)kStatusBadSlot);
    slot = -1;
  }
  if (kMode != kNormOnly && slot >= 0 && (pos < 0 || pos >= a.max_pos)) {
    if (j == 0 && a.status) atomicOr(a.status, (int32_t)kStatusBadPosition);
    slot = -1;
  }
  if (slot < 0) pos = 0;                           // the table is read only for a kept token
  const bool act = slot >= 0;

  // table slice: pairs p0 .. p0 + 15 (those below rd/2), cosines and sines
  const int h = a.rotary_dim >> 1, p0 = 16 * j;
  const bool rot = kMode != kNormOnly && act && p0 < h;
  const bool vec = kMode == kNeox128 || kMode == kNeox64 || (a.rotary_dim & 7) == 0;
  const float* cs = a.cos_sin + pos * a.rotary_dim;
  float* tab = tab_s[threadIdx.x];
  if (rot && vec) {
    const int nchunk = min(4, (h - p0) >> 2);      // h - p0 is a multiple of 4 here
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      if (v < nchunk) {
        cp_async16(tab + 4 * v, cs + p0 + 4 * v);
        cp_async16(tab + 16 + 4 * v, cs + h + p0 + 4 * v);
      }
    }
  }
  cp_async_commit();

  float xa[16], xb[16];
  const float tA = norm_rope_widen_group(ka, xa);
  const float tB = norm_rope_widen_group(kb, xb);
  const float ss = norm_rope_sumsq<kMode>(tA, tB);
  const float rs = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fmul_rn(ss, 0.0078125f), a.eps)));
  norm_rope_scale_group(a.weight + 16 * gA, rs, xa);
  norm_rope_scale_group(a.weight + 16 * gB, rs, xb);

  cp_async_wait_all();
  if constexpr (kMode == kNeox128 || kMode == kNeox64) {
    if (rot) {                       // element i of gA pairs with element i of gB (pair p0 + i)
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const float4 c4 = *reinterpret_cast<const float4*>(tab + 4 * v);
        const float4 s4 = *reinterpret_cast<const float4*>(tab + 16 + 4 * v);
        const float cc[4] = {c4.x, c4.y, c4.z, c4.w}, sn[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = 4 * v + u;
          const float y1 = xa[i], y2 = xb[i];
          xa[i] = __fsub_rn(__fmul_rn(y1, cc[u]), __fmul_rn(y2, sn[u]));
          xb[i] = __fadd_rn(__fmul_rn(y2, cc[u]), __fmul_rn(y1, sn[u]));
        }
      }
    }
  } else if constexpr (kMode == kGptj) {
    if (rot) {                       // pair p0 + q = elements 32j + 2q, 32j + 2q + 1
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        float cc[4], sn[4];
        if (vec) {
          const float4 c4 = *reinterpret_cast<const float4*>(tab + 4 * v);
          const float4 s4 = *reinterpret_cast<const float4*>(tab + 16 + 4 * v);
          cc[0] = c4.x; cc[1] = c4.y; cc[2] = c4.z; cc[3] = c4.w;
          sn[0] = s4.x; sn[1] = s4.y; sn[2] = s4.z; sn[3] = s4.w;
        } else {
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const bool in = p0 + 4 * v + u < h;
            cc[u] = in ? __ldg(cs + p0 + 4 * v + u) : 0.0f;
            sn[u] = in ? __ldg(cs + h + p0 + 4 * v + u) : 0.0f;
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int q = 4 * v + u;
          if (p0 + q < h) {
            float* xs = q < 8 ? xa : xb;
            const int e = 2 * (q & 7);
            const float y1 = xs[e], y2 = xs[e + 1];
            xs[e] = __fsub_rn(__fmul_rn(y1, cc[u]), __fmul_rn(y2, sn[u]));
            xs[e + 1] = __fadd_rn(__fmul_rn(y2, cc[u]), __fmul_rn(y1, sn[u]));
          }
        }
      }
    }
  }

  uint32_t ca0, ca1, cb0, cb1;
  const uint32_t sbA = norm_rope_encode_group(xa, ca0, ca1);
  const uint32_t sbB = norm_rope_encode_group(xb, cb0, cb1);
  // the token's 8 scale bytes, byte g from the lane holding group g
  uint32_t lo = (gA < 4 ? sbA << (8 * gA) : 0u) | (gB < 4 ? sbB << (8 * gB) : 0u);
  uint32_t hi = (gA >= 4 ? sbA << (8 * (gA - 4)) : 0u) | (gB >= 4 ? sbB << (8 * (gB - 4)) : 0u);
  lo |= __shfl_xor_sync(0xffffffffu, lo, 1);
  hi |= __shfl_xor_sync(0xffffffffu, hi, 1);
  lo |= __shfl_xor_sync(0xffffffffu, lo, 2);
  hi |= __shfl_xor_sync(0xffffffffu, hi, 2);
  if (act) {
    uint8_t* row = a.pages + slot * 72;
    *reinterpret_cast<uint2*>(row + 8 * gA) = make_uint2(ca0, ca1);
    *reinterpret_cast<uint2*>(row + 8 * gB) = make_uint2(cb0, cb1);
    if (j == 0) *reinterpret_cast<uint2*>(row + 64) = make_uint2(lo, hi);
  }
}

cudaError_t launch_insert_norm_rope(const NormRopeArgs& a, cudaStream_t stream) {
  if (a.n <= 0) return cudaSuccess;
  const int64_t threads = (int64_t)a.n * 4;
  const int block = 256;
  const unsigned grid = (unsigned)((threads + block - 1) / block);
  if (a.rotary_dim == 0) nvfp4_insert_norm_rope_kernel<kNormOnly><<<grid, block, 0, stream>>>(a);
  else if (a.is_neox && a.rotary_dim == 128) nvfp4_insert_norm_rope_kernel<kNeox128><<<grid, block, 0, stream>>>(a);
  else if (a.is_neox) nvfp4_insert_norm_rope_kernel<kNeox64><<<grid, block, 0, stream>>>(a);
  else nvfp4_insert_norm_rope_kernel<kGptj><<<grid, block, 0, stream>>>(a);
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
  uint32_t w[16];                    // loaded independently of the slot, as in the NVFP4 insert
  if (live) {
    const uint4* src = reinterpret_cast<const uint4*>(k + tok * 128 + j * 32);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 v = __ldg(src + i);
      w[4 * i] = v.x;
      w[4 * i + 1] = v.y;
      w[4 * i + 2] = v.z;
      w[4 * i + 3] = v.w;
    }
  }
  int64_t slot = live ? __ldg(slots + tok) : -1;
  if (slot >= num_slots) {
    if (j == 0 && status) atomicOr(status, (int32_t)kStatusBadSlot);
    slot = -1;
  }
  uint32_t scale_byte = 0;
  uint32_t cw[4] = {0, 0, 0, 0};
  if (slot >= 0) {
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
