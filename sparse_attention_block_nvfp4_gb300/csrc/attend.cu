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
// A unit is split over a cluster of 4 CTAs of 128 threads: CTA q takes the
// unit's pages q, q + 4, ... with its own online softmax, so four pages'
// loads are in flight per unit and the 4 x units CTAs spread over every SM;
// the CTAs' states meet in the first CTA's shared memory (distributed
// shared memory, no global scratch).  Per page, in a CTA:
//   * scores: thread i takes token i (all sixteen 16-byte loads of its K
//     row in flight for G = 1, eight or four for larger G, the row's
//     128-element dot products with the G queries held in shared memory as
//     fp32);
//   * online softmax: the page's maximum per head (warp redux + shared
//     memory), the running maximum M, rescale factor alpha = exp(M_old -
//     M), weights p_i = exp(s_i - M) (exp2f on log2e-scaled scores);
//   * weighted sum: warp w takes tokens w, w + 4, ...; lane l holds dims
//     4l .. 4l + 3 (8-byte loads of the V row, coalesced across the warp,
//     eight tokens' loads in flight), a fresh per-page partial (at most 32
//     terms), added to the running accumulator after its rescale by alpha;
//     for G <= 2 a half warp takes a token (16-byte loads, 16 terms a
//     partial, the halves added at the end); each thread prefetched its
//     token's V row into L2 when the page's work began;
//   * at the end every CTA stores its maximum, its warps' weight sums and
//     accumulators into the first CTA, which merges them in a fixed order:
//     M the largest maximum, each CTA's sums scaled by exp(M_q - M), then
//     o = acc / l.
// The longest chain of sequential additions in any sum is 32 + 4 + 4 + 4
// (page partial, pages of a CTA, warps, CTAs), scores excepted (128 terms);
// a weight carries at most 5 exponentials (its own, 3 rescalings, its CTA's
// merge factor).  The two cluster barriers are hardware barriers every
// thread of the cluster passes unconditionally.
#include <cstdint>
#include <cuda_runtime.h>
#include <math_constants.h>

#include "internal.h"

namespace nvfp4idx {

constexpr int kAttSplit = 4;          // CTAs (a cluster) per unit
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

// ------------------------------------------------ cluster (distributed shared memory)
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// The address of the same shared variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_map(const void* smem_ptr, uint32_t rank) {
  uint32_t d;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
               : "=r"(d)
               : "r"((uint32_t)__cvta_generic_to_shared(smem_ptr)), "r"(rank));
  return d;
}
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ void st_cluster_v4(uint32_t addr, float4 v) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v.x), "f"(v.y), "f"(v.z),
               "f"(v.w)
               : "memory");
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// 32 bytes from a 32-byte aligned address of read-only global memory in one
// load (the 256-bit form of sm_100-family GPUs).
__device__ __forceinline__ void att_ldg_32B(const uint4* p, uint4& lo, uint4& hi) {
  asm("ld.global.nc.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
      : "=r"(lo.x), "=r"(lo.y), "=r"(lo.z), "=r"(lo.w), "=r"(hi.x), "=r"(hi.y), "=r"(hi.z), "=r"(hi.w)
      : "l"(p));
}

// Registers grow with G (accumulators, scores): fewer K loads in flight and
// fewer resident CTAs for the larger groups.
template <int G>
struct AttCfg {
  static constexpr int kKUnroll = G == 1 ? 16 : (G <= 4 ? 8 : 4);
  static constexpr int kKUnroll32 = kKUnroll / 2;   // the same bytes in flight with 32-byte loads
  static constexpr int kMinBlocks = G == 1 ? 8 : (G == 2 ? 6 : (G == 4 ? 3 : 2));
  static constexpr int kSmemAcc = kAttSplit * 4 * G * kDim * 4;   // the leader's [CTA][warp][G][kDim]
  // V rows by 16-byte loads: a half warp per token, lane l % 16 on dims
  // 8 (l % 16) .. + 7, so a warp has twice the bytes in flight; the 8
  // accumulators per head and lane fit the register budget for G <= 2
  static constexpr bool kWideV = G <= 2;
  static constexpr int kVC = kWideV ? 8 : 4;   // dims per lane
};

// One 16-byte chunk c of a token's K row (dims 8c .. 8c + 7) into the G
// heads' dot products with the scaled queries.
template <int G>
__device__ __forceinline__ void att_dot8(float (&s)[G], const uint4 kv, const float (&q_s)[G][kDim], int c) {
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

// kWideK: the K cache is 32-byte aligned and each thread reads its token's
// K row in eight 32-byte loads (whole sectors) instead of sixteen 16-byte
// ones.
template <int G, bool kWideK>
__global__ void __cluster_dims__(kAttSplit, 1, 1) __launch_bounds__(kAttThreads, AttCfg<G>::kMinBlocks)
    sparse_attend_kernel(const AttendParams p) {
  extern __shared__ __align__(16) float acc_all[];     // [kAttSplit * 4 warps][G][kDim], used in CTA 0
  __shared__ __align__(16) float q_s[G][kDim];         // the unit's queries, scaled by scale * log2e
  __shared__ float p_s[G][kPage];                      // this page's weights
  __shared__ float red_s[4][G];
  __shared__ float lq_all[kAttSplit][4][G];            // CTA 0: every warp's weight sum
  __shared__ float mq_all[kAttSplit][G];               // CTA 0: every CTA's running maximum
  __shared__ int page_s[16];
  __shared__ int npages_s;
  const int64_t unit = blockIdx.x / kAttSplit;
  const int t = (int)(unit / p.H), hk = (int)(unit % p.H);
  cluster_arrive_relaxed();                            // this CTA runs: its shared memory may be written

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank();
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
  // ---- the selected pages with visible tokens, in id order (a repeated id
  // once, at its first place); an unreadable one (outside the page table or
  // the cache) empties the unit's output.  Lanes 0..15 of warp 0 take one id
  // each, so the id and page-table loads of the 16 ids are in flight together.
  if (warp == 0) {
    const bool req_ok = r >= 0 && r < p.num_reqs;
    int j = -1, bad = 0;
    bool vis = false;
    if (lane < 16 && req_ok) {
      j = __ldg(p.ids + ((int64_t)t * p.H + hk) * 16 + lane);
      vis = j >= 0 && (int64_t)j * kPage <= pos;
      if (vis) {
        if (j >= p.pt_stride) {
          bad = kStatusBadTable;
        } else {
          const int phys = __ldg(p.page_table + (int64_t)r * p.pt_stride + j);
          if (phys < 0 || phys >= p.num_blocks) bad = kStatusBadPage;
        }
      }
    }
    if (lane == 0 && !req_ok) bad = kStatusBadTable;
    bad = __reduce_or_sync(0xffffffffu, bad);
    // equal visible ids: only the lowest lane's is kept
    const uint32_t same = __match_any_sync(0xffffffffu, vis ? j : -1 - lane);
    const bool keep = vis && (same & ((1u << lane) - 1u)) == 0;
    const uint32_t kept = __ballot_sync(0xffffffffu, keep);
    if (keep) page_s[__popc(kept & ((1u << lane) - 1u))] = j;
    if (lane == 0) {
      npages_s = bad ? 0 : __popc(kept);
      if (bad && p.status && rank == 0) atomicOr(p.status, bad);
    }
  }
  __syncthreads();
  const int npages = npages_s;

  constexpr int VC = AttCfg<G>::kVC;
  float m_run[G], l_thr[G], acc[G][VC];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m_run[g] = -CUDART_INF_F;
    l_thr[g] = 0.0f;
#pragma unroll
    for (int c = 0; c < VC; ++c) acc[g][c] = 0.0f;
  }

  for (int pi = (int)rank; pi < npages; pi += kAttSplit) {
    const int j = page_s[pi];
    const int phys = __ldg(p.page_table + (int64_t)r * p.pt_stride + j);
    const int n = min(kPage, pos - j * kPage + 1);                // visible tokens of the page
    const int64_t base = (int64_t)phys * kPage * p.H + hk;         // token row 0 of the page, head hk
    // the page's V rows start their way into L2 now, behind the K loads
    if (tid < n) {
      const uint16_t* vrow = p.v_cache + (base + (int64_t)tid * p.H) * kDim;
      asm volatile("prefetch.global.L2 [%0];" ::"l"(vrow));
      asm volatile("prefetch.global.L2 [%0];" ::"l"(vrow + 64));
    }
    // ---- scores: thread = token
    float s[G];
#pragma unroll
    for (int g = 0; g < G; ++g) s[g] = -CUDART_INF_F;
    if (tid < n) {
      const uint4* krow = reinterpret_cast<const uint4*>(p.k_cache + (base + (int64_t)tid * p.H) * kDim);
#pragma unroll
      for (int g = 0; g < G; ++g) s[g] = 0.0f;
      if constexpr (kWideK) {
#pragma unroll AttCfg<G>::kKUnroll32
        for (int c2 = 0; c2 < kDim / 16; ++c2) {
          uint4 k0, k1;
          att_ldg_32B(krow + 2 * c2, k0, k1);
          att_dot8<G>(s, k0, q_s, 2 * c2);
          att_dot8<G>(s, k1, q_s, 2 * c2 + 1);
        }
      } else {
#pragma unroll AttCfg<G>::kKUnroll
        for (int c = 0; c < kDim / 8; ++c) att_dot8<G>(s, __ldg(krow + c), q_s, c);
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
    // ---- weighted sum of the V rows
    float part[G][VC];
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int c = 0; c < VC; ++c) part[g][c] = 0.0f;
    if constexpr (AttCfg<G>::kWideV) {
      // warp w, half h = lane / 16: tokens 2w + h, 2w + h + 8, ...
#pragma unroll 8
      for (int i = 2 * warp + (lane >> 4); i < n; i += 8) {
        const uint4 vv =
            __ldg(reinterpret_cast<const uint4*>(p.v_cache + (base + (int64_t)i * p.H) * kDim) + (lane & 15));
        const uint32_t w[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float pw = p_s[g][i];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            part[g][2 * c] = fmaf(pw, bf16_lo(w[c]), part[g][2 * c]);
            part[g][2 * c + 1] = fmaf(pw, bf16_hi(w[c]), part[g][2 * c + 1]);
          }
        }
      }
    } else {
      // warp w, tokens w, w + 4, ...; lane l on dims 4l .. 4l + 3
#pragma unroll 8
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
    }
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int c = 0; c < VC; ++c) acc[g][c] = fmaf(acc[g][c], alpha[g], part[g][c]);
    __syncthreads();                                  // p_s and red_s are rewritten by the next page
  }

  // ---- every CTA's state into CTA 0 of the cluster, which merges them
  cluster_wait_acquire();                             // (the start barrier) every CTA of the cluster runs
#pragma unroll
  for (int g = 0; g < G; ++g) {
    if constexpr (AttCfg<G>::kWideV) {
      // the two half warps' sums of the same dimensions (one addition)
#pragma unroll
      for (int c = 0; c < VC; ++c) acc[g][c] += __shfl_xor_sync(0xffffffffu, acc[g][c], 16);
      if (lane < 16) {
        float* const dst = &acc_all[((rank * 4 + warp) * G + g) * kDim + 8 * lane];
        st_cluster_v4(cluster_map(dst, 0), make_float4(acc[g][0], acc[g][1], acc[g][2], acc[g][3]));
        st_cluster_v4(cluster_map(dst + 4, 0), make_float4(acc[g][4], acc[g][5], acc[g][6], acc[g][7]));
      }
    } else {
      st_cluster_v4(cluster_map(&acc_all[((rank * 4 + warp) * G + g) * kDim + 4 * lane], 0),
                    make_float4(acc[g][0], acc[g][1], acc[g][2], acc[g][3]));
    }
    const float lw = warp_sum_f32(l_thr[g]);
    if (lane == 0) st_cluster_f32(cluster_map(&lq_all[rank][warp][g], 0), lw);
    if (tid == 0) st_cluster_f32(cluster_map(&mq_all[rank][g], 0), m_run[g]);
  }
  cluster_arrive_release();
  if (rank != 0) return;                              // only CTA 0's shared memory is read from here on
  cluster_wait_acquire();
  for (int i = tid; i < G * kDim; i += kAttThreads) {
    const int g = i / kDim, d = i % kDim;
    float M = mq_all[0][g];
#pragma unroll
    for (int q = 1; q < kAttSplit; ++q) M = fmaxf(M, mq_all[q][g]);
    float l = 0.0f, a = 0.0f;
#pragma unroll
    for (int q = 0; q < kAttSplit; ++q) {
      const float f = mq_all[q][g] == -CUDART_INF_F ? 0.0f : exp2f(mq_all[q][g] - M);
      const float lq = (lq_all[q][0][g] + lq_all[q][1][g]) + (lq_all[q][2][g] + lq_all[q][3][g]);
      const float* aq = acc_all + ((4 * q) * G + g) * kDim + d;     // warp w of CTA q at aq + w * G * kDim
      const float sq = (aq[0] + aq[G * kDim]) + (aq[2 * G * kDim] + aq[3 * G * kDim]);
      l = fmaf(f, lq, l);
      a = fmaf(f, sq, a);
    }
    p.out[((int64_t)t * HQ + hk * G + g) * kDim + d] = l > 0.0f ? a / l : 0.0f;
  }
}

template <int G, bool kWideK>
static cudaError_t launch_attend_gk(const AttendParams& p, int64_t units, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(sparse_attend_kernel<G, kWideK>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, AttCfg<G>::kSmemAcc);
  if (e != cudaSuccess) return e;
  sparse_attend_kernel<G, kWideK><<<(unsigned)(units * kAttSplit), kAttThreads, AttCfg<G>::kSmemAcc, stream>>>(p);
  return cudaGetLastError();
}

template <int G>
static cudaError_t launch_attend_g(const AttendParams& p, int64_t units, cudaStream_t stream) {
  return (reinterpret_cast<uintptr_t>(p.k_cache) & 31u) == 0 ? launch_attend_gk<G, true>(p, units, stream)
                                                              : launch_attend_gk<G, false>(p, units, stream);
}

cudaError_t launch_attend(const AttendParams& p, cudaStream_t stream) {
  const int64_t units = (int64_t)p.num_rows * p.H;
  if (units <= 0) return cudaSuccess;
  switch (p.G) {
    case 1: return launch_attend_g<1>(p, units, stream);
    case 2: return launch_attend_g<2>(p, units, stream);
    case 4: return launch_attend_g<4>(p, units, stream);
    default: return launch_attend_g<8>(p, units, stream);
  }
}

}  // namespace nvfp4idx
