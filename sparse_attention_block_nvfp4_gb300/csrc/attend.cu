// attend.cu -- block-sparse attention over the pages the indexer selected.
//
// The consumer of the indexer's [T, H, 16] id buffer
// (vllm.models.minimax_m3.nvidia.indexer_nvfp4, MiniMaxM3IndexerNvfp4Impl
// .forward: the kernels write the ids "straight into the shared [T, H, 16]
// buffer the attend reads"; vllm.models.minimax_m3.nvidia.indexer_flashinfer,
// forward: "The attend reads the shared buffer directly").  Per row t and KV
// head hk (one per index head), the G query heads hk*G .. hk*G+G-1 attend
// over the visible tokens (position <= the row's) of the pages listed in
// ids[t][hk] (-1 skipped), read from a bf16 main cache [num_blocks, 128, H,
// 128] through the page table; o = softmax(scale q.k) v, fp32 out.
//
// Roofline: HBM.  A unit (t, hk) reads up to 16 pages x 128 tokens x 256 B
// of K and as much of V (1 MB) for 4 G flops per K/V byte pair: G = 1 is
// 1 flop per byte, far below the tensor cores' ratio, so the scores and the
// weighted sums run on the CUDA cores in fp32 (bf16 products are exact).
// One CTA of 128 threads per unit; per page:
//   * scores: thread i takes token i (16-byte loads of its K row, the
//     row's 128-element dot products with the G queries held in shared
//     memory as fp32);
//   * online softmax: the page's maximum per head (warp redux + shared
//     memory), the running maximum M, rescale factor alpha = exp(M_old -
//     M), weights p_i = exp(s_i - M) (exp2f on log2e-scaled scores);
//   * weighted sum: warp w takes tokens w, w + 4, ...; lane l holds dims
//     4l .. 4l + 3 (8-byte loads of the V row, coalesced across the warp),
//     a fresh per-page partial (at most 32 terms), added to the running
//     accumulator after its rescale by alpha;
//   * at the end the 4 warps' accumulators and the per-thread weight sums
//     are added in shared memory and o = acc / l is written.
// The longest chain of sequential additions in any sum is 32 + 16 + 4
// (page partial, pages, warps), scores excepted (128 terms).
#include <cstdint>
#include <cuda_runtime.h>
#include <math_constants.h>

#include "internal.h"

namespace nvfp4idx {

constexpr int kAttThreads = 128;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ float warp_max_f32(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}
__device__ __forceinline__ float warp_sum_f32(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <int G>
__global__ void __launch_bounds__(kAttThreads) sparse_attend_kernel(const AttendParams p) {
  __shared__ __align__(16) float q_s[G][kDim];      // the unit's queries, scaled by scale * log2e
  __shared__ float p_s[G][kPage];                   // this page's weights
  __shared__ float red_s[4][G];
  __shared__ __align__(16) float acc_s[4][G][kDim];
  __shared__ int page_s[16];
  __shared__ int npages_s;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t unit = blockIdx.x;
  const int t = (int)(unit / p.H), hk = (int)(unit % p.H);
  const int HQ = p.H * G;
  const int r = __ldg(p.row_req + t), pos = __ldg(p.row_pos + t);

  // ---- the queries, in fp32, pre-scaled so that exp2 of the difference of
  // two scores is exp of the difference of the scaled dot products
  const float qscale = p.scale * kLog2e;
  for (int i = tid; i < G * kDim / 2; i += kAttThreads) {
    const int g = i / (kDim / 2), d2 = i % (kDim / 2);
    const uint32_t w =
        __ldg(reinterpret_cast<const uint32_t*>(p.q + ((int64_t)t * HQ + hk * G + g) * kDim) + d2);
    q_s[g][2 * d2] = bf16_lo(w) * qscale;
    q_s[g][2 * d2 + 1] = bf16_hi(w) * qscale;
  }
  // ---- the selected pages with visible tokens, in id order; an unreadable
  // one (outside the page table or the cache) empties the unit's output
  if (tid == 0) {
    int n = 0, bad = 0;
    if (r < 0 || r >= p.num_reqs) {
      bad = kStatusBadTable;
    } else {
      for (int k = 0; k < 16; ++k) {
        const int j = __ldg(p.ids + ((int64_t)t * p.H + hk) * 16 + k);
        if (j < 0 || (int64_t)j * kPage > pos) continue;
        if (j >= p.pt_stride) {
          bad = kStatusBadTable;
          break;
        }
        const int phys = __ldg(p.page_table + (int64_t)r * p.pt_stride + j);
        if (phys < 0 || phys >= p.num_blocks) {
          bad = kStatusBadPage;
          break;
        }
        page_s[n] = j;
        ++n;
      }
    }
    npages_s = bad ? 0 : n;
    if (bad && p.status) atomicOr(p.status, bad);
  }
  __syncthreads();
  const int npages = npages_s;

  float m_run[G], l_thr[G], acc[G][4];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m_run[g] = -CUDART_INF_F;
    l_thr[g] = 0.0f;
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[g][c] = 0.0f;
  }

  for (int pi = 0; pi < npages; ++pi) {
    const int j = page_s[pi];
    const int phys = __ldg(p.page_table + (int64_t)r * p.pt_stride + j);
    const int n = min(kPage, pos - j * kPage + 1);                // visible tokens of the page
    const int64_t base = (int64_t)phys * kPage * p.H + hk;         // token row 0 of the page, head hk
    // ---- scores: thread = token
    float s[G];
#pragma unroll
    for (int g = 0; g < G; ++g) s[g] = -CUDART_INF_F;
    if (tid < n) {
      const uint4* krow = reinterpret_cast<const uint4*>(p.k_cache + (base + (int64_t)tid * p.H) * kDim);
#pragma unroll
      for (int g = 0; g < G; ++g) s[g] = 0.0f;
#pragma unroll 4
      for (int c = 0; c < kDim / 8; ++c) {
        const uint4 kv = __ldg(krow + c);
        const uint32_t w[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float4 qa = *reinterpret_cast<const float4*>(&q_s[g][8 * c]);
          const float4 qb = *reinterpret_cast<const float4*>(&q_s[g][8 * c + 4]);
          float a = s[g];
          a = fmaf(qa.x, bf16_lo(w[0]), a);
          a = fmaf(qa.y, bf16_hi(w[0]), a);
          a = fmaf(qa.z, bf16_lo(w[1]), a);
          a = fmaf(qa.w, bf16_hi(w[1]), a);
          a = fmaf(qb.x, bf16_lo(w[2]), a);
          a = fmaf(qb.y, bf16_hi(w[2]), a);
          a = fmaf(qb.z, bf16_lo(w[3]), a);
          a = fmaf(qb.w, bf16_hi(w[3]), a);
          s[g] = a;
        }
      }
    }
    // ---- the page's maximum per head, the new running maximum
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float mw = warp_max_f32(s[g]);
      if (lane == 0) red_s[warp][g] = mw;
    }
    __syncthreads();
    float alpha[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float mp = fmaxf(fmaxf(red_s[0][g], red_s[1][g]), fmaxf(red_s[2][g], red_s[3][g]));
      const float mn = fmaxf(m_run[g], mp);
      alpha[g] = m_run[g] == -CUDART_INF_F ? 0.0f : exp2f(m_run[g] - mn);
      m_run[g] = mn;
      const float pw = tid < n ? exp2f(s[g] - mn) : 0.0f;
      p_s[g][tid] = pw;
      l_thr[g] = l_thr[g] * alpha[g] + pw;
    }
    __syncthreads();
    // ---- weighted sum of the V rows: warp w, tokens w, w + 4, ...
    float part[G][4];
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int c = 0; c < 4; ++c) part[g][c] = 0.0f;
    for (int i = warp; i < n; i += 4) {
      const uint2 vv = __ldg(reinterpret_cast<const uint2*>(p.v_cache + (base + (int64_t)i * p.H) * kDim) + lane);
      const float v0 = bf16_lo(vv.x), v1 = bf16_hi(vv.x), v2 = bf16_lo(vv.y), v3 = bf16_hi(vv.y);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float pw = p_s[g][i];
        part[g][0] = fmaf(pw, v0, part[g][0]);
        part[g][1] = fmaf(pw, v1, part[g][1]);
        part[g][2] = fmaf(pw, v2, part[g][2]);
        part[g][3] = fmaf(pw, v3, part[g][3]);
      }
    }
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[g][c] = fmaf(acc[g][c], alpha[g], part[g][c]);
    __syncthreads();                                  // p_s and red_s are rewritten by the next page
  }

  // ---- combine the warps' accumulators and the threads' weight sums
#pragma unroll
  for (int g = 0; g < G; ++g) {
    *reinterpret_cast<float4*>(&acc_s[warp][g][4 * lane]) = make_float4(acc[g][0], acc[g][1], acc[g][2], acc[g][3]);
    const float lw = warp_sum_f32(l_thr[g]);
    if (lane == 0) red_s[warp][g] = lw;
  }
  __syncthreads();
  for (int i = tid; i < G * kDim; i += kAttThreads) {
    const int g = i / kDim, d = i % kDim;
    const float l = (red_s[0][g] + red_s[1][g]) + (red_s[2][g] + red_s[3][g]);
    const float a = (acc_s[0][g][d] + acc_s[1][g][d]) + (acc_s[2][g][d] + acc_s[3][g][d]);
    p.out[((int64_t)t * HQ + hk * G + g) * kDim + d] = l > 0.0f ? a / l : 0.0f;
  }
}

cudaError_t launch_attend(const AttendParams& p, cudaStream_t stream) {
  const int64_t units = (int64_t)p.num_rows * p.H;
  if (units <= 0) return cudaSuccess;
  switch (p.G) {
    case 1: sparse_attend_kernel<1><<<(unsigned)units, kAttThreads, 0, stream>>>(p); break;
    case 2: sparse_attend_kernel<2><<<(unsigned)units, kAttThreads, 0, stream>>>(p); break;
    case 4: sparse_attend_kernel<4><<<(unsigned)units, kAttThreads, 0, stream>>>(p); break;
    default: sparse_attend_kernel<8><<<(unsigned)units, kAttThreads, 0, stream>>>(p); break;
  }
  return cudaGetLastError();
}

}  // namespace nvfp4idx
