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
#include <algorithm>
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

// Two fp32 values in one 64-bit register (element 2i in the low word,
// 2i + 1 in the high word) and the packed fp32 instructions of sm_100-family
// GPUs, whose lanes each round as the scalar instruction does (round to
// nearest even, subnormals kept): the same results as scalar code, bit for
// bit, from half the instructions.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  return ((uint64_t)__float_as_uint(hi) << 32) | __float_as_uint(lo);
}
__device__ __forceinline__ float f2_lo(uint64_t v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float f2_hi(uint64_t v) { return __uint_as_float((uint32_t)(v >> 32)); }
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
// The two bf16 halves of a word as an exact fp32 pair.
__device__ __forceinline__ uint64_t bf16x2_to_f2(uint32_t w) {
  return ((uint64_t)(w & 0xFFFF0000u) << 32) | (uint32_t)(w << 16);
}

// One 16-element group of a token (two 16-byte words of bf16, loaded at
// entry) widened to 8 fp32 pairs, and the group sum of squares t = e + o
// (running sums of the even / odd elements' squares, one rounding per step:
// the two lanes of one packed fused multiply-add).
__device__ __forceinline__ float norm_rope_widen_group(const uint4 (&v)[2], uint64_t (&x)[8]) {
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    x[4 * i] = bf16x2_to_f2(v[i].x);
    x[4 * i + 1] = bf16x2_to_f2(v[i].y);
    x[4 * i + 2] = bf16x2_to_f2(v[i].z);
    x[4 * i + 3] = bf16x2_to_f2(v[i].w);
  }
  uint64_t eo = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) eo = f2_fma(x[i], x[i], eo);
  return __fadd_rn(f2_lo(eo), f2_hi(eo));
}

// y = (x * rs) * w for one group (wg: the group's 16 bf16 weights; the
// loads do not depend on the token, so they stay out of the token loop).
__device__ __forceinline__ void norm_rope_scale_group(const uint16_t* wg, uint64_t rs2, uint64_t (&x)[8]) {
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const uint4 w = __ldg(reinterpret_cast<const uint4*>(wg) + i);
    x[4 * i] = f2_mul(f2_mul(x[4 * i], rs2), bf16x2_to_f2(w.x));
    x[4 * i + 1] = f2_mul(f2_mul(x[4 * i + 1], rs2), bf16x2_to_f2(w.y));
    x[4 * i + 2] = f2_mul(f2_mul(x[4 * i + 2], rs2), bf16x2_to_f2(w.z));
    x[4 * i + 3] = f2_mul(f2_mul(x[4 * i + 3], rs2), bf16x2_to_f2(w.w));
  }
}

// bf16 rounding of one group, its amax from the bf16 words, the NVFP4
// codes (c0, c1) and the returned scale byte.  The quotients are those of
// nvfp4_ratio taken on the signed value: x r + 3 * 2^10 lies in
// (2^11, 2^12) for |x r| < 2^10, where the ulp is 2^-12 as above 3 * 2^10,
// and round-to-nearest-even on that grid is symmetric about 3 * 2^10 (an
// even multiple of 2^-12), so the difference is minus the rounding of
// |x| r; the sign of x is put back for the quotients that round to zero.
__device__ __forceinline__ uint32_t norm_rope_encode_group(const uint64_t (&x)[8], uint32_t& c0, uint32_t& c1) {
  uint32_t R[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(R[i]) : "f"(f2_hi(x[i])), "f"(f2_lo(x[i])));
  uint32_t mx = R[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) mx = bf16x2_max_abs(mx, R[i]);
  const uint32_t sb = e4m3_scale_of_amax(bf16x2_amax_f32(mx));
  const float s = e4m3_to_f32(sb);
  float q[16];
  if (s > 0.0f) {
    const float r = rcp_approx(s);
    const uint64_t r2 = f2_pack(r, r), k2 = f2_pack(3072.0f, 3072.0f);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint64_t g = f2_sub(f2_fma(bf16x2_to_f2(R[i]), r2, k2), k2);
      q[2 * i] = __uint_as_float(__float_as_uint(f2_lo(g)) | ((R[i] << 16) & 0x80000000u));
      q[2 * i + 1] = __uint_as_float(__float_as_uint(f2_hi(g)) | (R[i] & 0x80000000u));
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      q[2 * i] = __uint_as_float((R[i] << 16) & 0x80000000u);
      q[2 * i + 1] = __uint_as_float(R[i] & 0x80000000u);
    }
  }
  c0 = f32x8_to_e2m1x8(q);
  c1 = f32x8_to_e2m1x8(q + 8);
  return sb;
}

// 32 bytes from a 32-byte aligned address of read-only global memory in one
// load (the 256-bit form of sm_100-family GPUs): both 16-byte halves of a
// sector in one request.
__device__ __forceinline__ void ldg_32B(const uint4* p, uint4& lo, uint4& hi) {
  asm("ld.global.nc.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
      : "=r"(lo.x), "=r"(lo.y), "=r"(lo.z), "=r"(lo.w), "=r"(hi.x), "=r"(hi.y), "=r"(hi.z), "=r"(hi.w)
      : "l"(p));
}

// One token's two key groups, slot and position, loaded independently (a
// skipped token's key is read and dropped; past the end nothing is read).
// kWide: the keys are 32-byte aligned and each group comes in one load.
template <int kMode, bool kWide>
__device__ __forceinline__ void norm_rope_load(const NormRopeArgs& a, int64_t tok, int gA, int gB,
                                               uint4 (&ka)[2], uint4 (&kb)[2], int64_t& slot,
                                               int64_t& pos) {
  const bool live = tok < a.n;
  ka[0] = ka[1] = kb[0] = kb[1] = make_uint4(0u, 0u, 0u, 0u);
  if (live) {
    const uint4* kt = reinterpret_cast<const uint4*>(a.k + tok * 128);
    if constexpr (kWide) {
      ldg_32B(kt + 2 * gA, ka[0], ka[1]);
      ldg_32B(kt + 2 * gB, kb[0], kb[1]);
    } else {
      ka[0] = __ldg(kt + 2 * gA);
      ka[1] = __ldg(kt + 2 * gA + 1);
      kb[0] = __ldg(kt + 2 * gB);
      kb[1] = __ldg(kt + 2 * gB + 1);
    }
  }
  slot = live ? __ldg(a.slots + tok) : -1;
  pos = (kMode != kNormOnly && live) ? __ldg(a.positions + tok) : 0;
}

// A token's slot and position checked (an out-of-range one flags the status
// word and skips the token; the table is read only for a kept token), and
// the asynchronous copy of its table row started: the row's 16-byte chunks
// (rd/2 cosines, then rd/2 sines) go round the token's 4 lanes, lane j
// taking chunks j, j + 4, ..., so that each copy instruction of a warp reads
// 64 contiguous bytes per token.  Chunk c lands at row[c + c / 8] (one pad
// chunk per 8), which puts the chunks 4j + v that lane j reads back on four
// different bank quads.
template <int kMode>
__device__ __forceinline__ bool norm_rope_accept(const NormRopeArgs& a, int j, int64_t& slot, int64_t& pos,
                                                 float4* row) {
  if (slot >= a.num_slots) {
    if (j == 0 && a.status) atomicOr(a.status, (int32_t)kStatusBadSlot);
    slot = -1;
  }
  if (kMode != kNormOnly && slot >= 0 && (pos < 0 || pos >= a.max_pos)) {
    if (j == 0 && a.status) atomicOr(a.status, (int32_t)kStatusBadPosition);
    slot = -1;
  }
  if (slot < 0) pos = 0;
  const bool vec = kMode == kNeox128 || kMode == kNeox64 || (a.rotary_dim & 7) == 0;
  if (kMode != kNormOnly && slot >= 0 && vec) {
    const float* cs = a.cos_sin + pos * a.rotary_dim;
    const int nc = kMode == kNeox128 ? 32 : kMode == kNeox64 ? 16 : a.rotary_dim >> 2;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int c = 4 * i + j;
      if (c < nc) cp_async16(row + c + (c >> 3), cs + 4 * c);
    }
  }
  cp_async_commit();
  return slot >= 0;
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
// (2i, 2i + 1) stay inside a thread anyway.  The element-wise steps run on
// packed fp32 pairs.  The grid is persistent (as many CTAs as fit at once),
// each group of 4 threads stepping through the tokens with the grid's
// stride, and the loads run one token ahead: the key groups, slot and
// position of the next token are issued before the current one is
// computed, and the asynchronous copy of the next token's table row into
// shared memory when the current one is written.  The CTAs have 128 threads
// and up to 96 registers (5 per SM): with the loads one token ahead the
// kernel is limited by the L1 load pipe, not by the warps in flight.
// HBM-bound: 256 B key + 8 B slot + 8 B position + 72 B row per token, plus
// the table rows.
template <int kMode, bool kWide>
__global__ void __launch_bounds__(128, 5) nvfp4_insert_norm_rope_kernel(const NormRopeArgs a) {
  // per token: its table row in 16-byte chunks at c + c / 8, rows 42 chunks
  // apart, so that the two tokens of a quarter warp read different bank quads
  __shared__ __align__(16) float4 row_s[32][42];
  float4* row = row_s[threadIdx.x >> 2];
  const int j = (int)(threadIdx.x & 3);
  int gA, gB;
  norm_rope_groups<kMode>(j, gA, gB);
  const int h = a.rotary_dim >> 1, p0 = 16 * j;
  const bool vec = kMode == kNeox128 || kMode == kNeox64 || (a.rotary_dim & 7) == 0;
  const int64_t stride = (int64_t)gridDim.x * (blockDim.x >> 2);
  const int64_t tok0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 2;
  const int lane_tok = (int)((threadIdx.x & 31) >> 2);   // the warp steps while its first token is live

  uint4 ka[2], kb[2];
  int64_t slot, pos;
  norm_rope_load<kMode, kWide>(a, tok0, gA, gB, ka, kb, slot, pos);
  bool act = norm_rope_accept<kMode>(a, j, slot, pos, row);
  for (int64_t tok = tok0; tok - lane_tok < a.n; tok += stride) {
    uint4 na[2], nb[2];
    int64_t nslot, npos;
    norm_rope_load<kMode, kWide>(a, tok + stride, gA, gB, na, nb, nslot, npos);

    uint64_t xa[8], xb[8];
    const float tA = norm_rope_widen_group(ka, xa);
    const float tB = norm_rope_widen_group(kb, xb);
    const float ss = norm_rope_sumsq<kMode>(tA, tB);
    const float rs = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fmul_rn(ss, 0.0078125f), a.eps)));
    const uint64_t rs2 = f2_pack(rs, rs);
    norm_rope_scale_group(a.weight + 16 * gA, rs2, xa);
    norm_rope_scale_group(a.weight + 16 * gB, rs2, xb);

    const bool rot = kMode != kNormOnly && act && p0 < h;
    cp_async_wait_all();
    __syncwarp();                    // the row, copied by the token's 4 lanes
    if constexpr (kMode == kNeox128 || kMode == kNeox64) {
      if (rot) {                       // element i of gA pairs with element i of gB (pair p0 + i)
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const int c = 4 * j + v, sn_c = (h >> 2) + 4 * j + v;
          const ulonglong2 c4 = *reinterpret_cast<const ulonglong2*>(row + c + (c >> 3));
          const ulonglong2 s4 = *reinterpret_cast<const ulonglong2*>(row + sn_c + (sn_c >> 3));
          const uint64_t cc[2] = {c4.x, c4.y}, sn[2] = {s4.x, s4.y};
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int i = 2 * v + u;
            const uint64_t y1 = xa[i], y2 = xb[i];
            xa[i] = f2_sub(f2_mul(y1, cc[u]), f2_mul(y2, sn[u]));
            xb[i] = f2_add(f2_mul(y2, cc[u]), f2_mul(y1, sn[u]));
          }
        }
      }
    } else if constexpr (kMode == kGptj) {
      if (rot) {                       // pair p0 + q = elements 32j + 2q, 32j + 2q + 1
        const float* cs = a.cos_sin + pos * a.rotary_dim;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          float cc[4], sn[4];
          if (vec) {
            const int c = 4 * j + v, sn_c = (h >> 2) + 4 * j + v;
            const float4 c4 = row[c + (c >> 3)];
            const float4 s4 = row[sn_c + (sn_c >> 3)];
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
              uint64_t& xs = q < 8 ? xa[q] : xb[q - 8];
              const float y1 = f2_lo(xs), y2 = f2_hi(xs);
              xs = f2_pack(__fsub_rn(__fmul_rn(y1, cc[u]), __fmul_rn(y2, sn[u])),
                           __fadd_rn(__fmul_rn(y2, cc[u]), __fmul_rn(y1, sn[u])));
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

    // the next token becomes the current one; its table row is copied once
    // every lane has read this token's
    ka[0] = na[0];
    ka[1] = na[1];
    kb[0] = nb[0];
    kb[1] = nb[1];
    slot = nslot;
    pos = npos;
    __syncwarp();                    // every lane is done with the row
    act = norm_rope_accept<kMode>(a, j, slot, pos, row);
  }
  cp_async_wait_all();
}

// CTAs of the persistent fused insert that fit on the device at once.
template <int kMode, bool kWide>
static int norm_rope_grid(int64_t n) {
  static int per_sm = 0, sms = 0;
  if (per_sm == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, nvfp4_insert_norm_rope_kernel<kMode, kWide>, 128,
                                                      0) != cudaSuccess ||
        per_sm < 1)
      per_sm = 1, sms = sms > 0 ? sms : 1;
  }
  const int64_t need = (n * 4 + 127) / 128;
  return (int)std::min<int64_t>(need, (int64_t)per_sm * sms);
}

template <int kMode>
static void launch_norm_rope_mode(const NormRopeArgs& a, cudaStream_t stream) {
  if ((reinterpret_cast<uintptr_t>(a.k) & 31u) == 0)
    nvfp4_insert_norm_rope_kernel<kMode, true><<<norm_rope_grid<kMode, true>(a.n), 128, 0, stream>>>(a);
  else
    nvfp4_insert_norm_rope_kernel<kMode, false><<<norm_rope_grid<kMode, false>(a.n), 128, 0, stream>>>(a);
}

cudaError_t launch_insert_norm_rope(const NormRopeArgs& a, cudaStream_t stream) {
  if (a.n <= 0) return cudaSuccess;
  if (a.rotary_dim == 0) launch_norm_rope_mode<kNormOnly>(a, stream);
  else if (a.is_neox && a.rotary_dim == 128) launch_norm_rope_mode<kNeox128>(a, stream);
  else if (a.is_neox) launch_norm_rope_mode<kNeox64>(a, stream);
  else launch_norm_rope_mode<kGptj>(a, stream);
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
