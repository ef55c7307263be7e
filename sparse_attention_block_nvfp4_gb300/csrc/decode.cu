// decode.cu -- decode indexer: page scores on the tensor cores + fused top-15.
//
// Follows MiniMaxM3IndexerNvfp4Impl.forward (decode branch) of
// vllm.models.minimax_m3.nvidia.indexer_nvfp4: each request's 1..8 queries are
// read in place, every history page of the request is read ONCE for all of
// its queries and heads, and the top-k goes straight into the output buffer.
//
// Work split.  The history pages of all requests (page j < (seq_len-1)/128 of
// request r) form one list of T pages; CTA c of G = min(grid, T) takes the
// contiguous range [c*T/G, (c+1)*T/G), never empty.  A CTA walks its range
// as segments (one per request it touches).  One CTA per SM, warp roles
// linked by mbarrier rings; page g of the walk uses ring slot g % 4 and is
// handled by the role instance of parity g % 2:
//   * producer warp: reads page ids 32 at a time and has the TMA unit copy
//     each 9216-byte page into an 8-stage shared ring (cp.async.bulk,
//     transaction-count completion);
//   * two dequant warpgroups: thread t reads token t's 72-byte row,
//     dequantises it exactly to fp16 (E2M1 x E4M3 fits fp16) and stores it
//     into tensor-memory lane t (tcgen05.st): the page becomes the MMA's A
//     operand (M = 128 tokens, K = 128); at each segment start both widen the
//     request's E4M3 queries to fp16 into a 128B-swizzled B tile (double
//     buffered);
//   * two MMA warps: one thread each issues 8 tcgen05.mma (K = 16) per page,
//     D[token][row] in fp32 in tensor memory, and commits once per page (a
//     single thread cannot issue small-N MMAs as fast as the tensor core
//     retires them);
//   * two epilogue warpgroups: load D and take the max over each warp's 32
//     token lanes per column with one redux.sync per column, combine the four
//     warps through shared memory, and insert the page score into the row's
//     running top-15 (thread = row); at a segment end group 1 hands its lists
//     to group 0, which merges them.
// A request covered by one CTA is finalised in place; otherwise each segment
// leaves its 15 candidates per row in scratch and decode_merge_kernel merges
// them (and writes the rows of requests with no history page).
#include <cstdint>
#include <cuda_runtime.h>

#include "codec.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "topk.cuh"

namespace nvfp4idx {

constexpr int kDecStages = 8;            // raw page ring (shared memory)
constexpr int kDecA = 4;                 // page g: A buffer g % 4 (columns [64a, 64a+64)) and
constexpr int kDecD = kDecA;             // D buffer g % 4 (columns [256 + 64d, 256 + 64d + NQ))
// warp 0 TMA; 1 / 2 MMA issue; 3-6 / 7-10 dequant; 11-14 / 15-18 epilogue
// (first of each pair: pages of even index, second: odd)
constexpr int kDecThreads = 608;
constexpr int kDqTid0 = 96, kEpTid0 = 352;
constexpr uint32_t kDecTmemCols = 512;

template <int NQ>
struct DecLayout {
  static constexpr uint32_t kQBytes = NQ * 256;                   // fp16 [2][NQ][64], SW128
  static constexpr uint32_t kQOff = 0;                             // two query tiles
  static constexpr uint32_t kStageOff = 2 * kQBytes;               // multiple of 1024
  static constexpr uint32_t kRedOff = kStageOff + kDecStages * kPageBytes;   // [2 groups][2][4 warps][NQ]
  static constexpr uint32_t kMrgOff = kRedOff + 2 * 2 * 4 * NQ * 4;            // [2][64 rows][15] (score, id)
  static constexpr uint32_t kPreOff = kMrgOff + 2 * kMaxRows * kHistK * 8;
  // one CTA per SM: it holds all 512 tensor-memory columns
  static size_t bytes(int num_reqs) {
    const size_t b = 1024 + kPreOff + (size_t)(num_reqs + 1) * 4;
    return b < 120 * 1024 ? 120 * 1024 : b;
  }
};

__device__ __forceinline__ int hist_pages(int seq_len, int pt_stride) {
  const int h = seq_len >= 1 ? (seq_len - 1) >> 7 : 0;
  return h > pt_stride ? 0 : h;   // a history wider than the table is finalised as bad by the merge
}

// CTA owning global page x when T pages are split over G CTAs.
__device__ __forceinline__ int cta_of(int64_t x, int64_t T, int G) {
  return (int)(((x + 1) * G - 1) / T);
}

// Max over the warp's 32 lanes (tokens) of CW <= 32 columns, one redux.sync
// per column; afterwards lane l holds column l (l < CW).
template <int CW>
__device__ __forceinline__ float warp_colmax(const float (&v)[CW], int lane) {
  float m = 0.0f;
#pragma unroll
  for (int k = 0; k < CW; ++k) {
    float r;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v[k]));
    m = (lane == k) ? r : m;
  }
  return m;
}

// Merge a sorted top-15 list `b` (score desc, id asc; id -1 = empty) into `a`.
__device__ __forceinline__ void merge_top15(TopK15& a, const float2* b) {
  float s[15];
  int id[15];
  int i = 0, j = 0;
#pragma unroll
  for (int k = 0; k < 15; ++k) {
    const float2 bj = b[j < 15 ? j : 14];
    const float bs = bj.x;
    const int bi = __float_as_int(bj.y);
    float as = -CUDART_INF_F;
    int ai = -1;
#pragma unroll
    for (int t = 0; t < 15; ++t)
      if (t == i) {
        as = a.s[t];
        ai = a.id[t];
      }
    const bool a_ok = i < 15 && ai >= 0;
    const bool b_ok = j < 15 && bi >= 0;
    const bool take_a = a_ok && (!b_ok || as > bs || (as == bs && ai < bi));
    s[k] = take_a ? as : (b_ok ? bs : -CUDART_INF_F);
    id[k] = take_a ? ai : (b_ok ? bi : -1);
    i += take_a ? 1 : 0;
    j += (!take_a && b_ok) ? 1 : 0;
  }
#pragma unroll
  for (int k = 0; k < 15; ++k) {
    a.s[k] = s[k];
    a.id[k] = id[k];
  }
}

// The CTA's walk over its page range, identical in every role.
struct SegWalk {
  const int32_t* pre;
  int NR;
  int64_t n;        // pages in the range
  int64_t g;        // pages walked
  int r, j;         // current request, page
  __device__ __forceinline__ bool more() const { return g < n; }
  // pages [j, j_end) of request r form the current segment
  __device__ __forceinline__ int seg_end() const {
    const int hist = pre[r + 1] - pre[r];
    const int64_t left = n - g;
    return (int)((int64_t)hist < (int64_t)j + left ? (int64_t)hist : (int64_t)j + left);
  }
  __device__ __forceinline__ void next_request() {
    ++r;
    while (r < NR && pre[r + 1] - pre[r] == 0) ++r;
    j = 0;
  }
};

template <int NQ>
__global__ void __launch_bounds__(kDecThreads, 1) decode_score_kernel(const DecodeParams p) {
  using Lay = DecLayout<NQ>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t raw_full[kDecStages], raw_empty[kDecStages];
  __shared__ __align__(8) uint64_t a_full[kDecA];
  __shared__ __align__(8) uint64_t d_full[kDecD], d_empty[kDecD];
  __shared__ __align__(8) uint64_t q_full[2], q_empty[2];
  __shared__ uint32_t tmem_base_s;
  __shared__ volatile int abort_s;
  __shared__ int warp_sum[kDecThreads / 32];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t sbase = (raw_u32 + 1023u) & ~1023u;
  uint8_t* const base = smem_raw + (sbase - raw_u32);
  float* const red = reinterpret_cast<float*>(base + Lay::kRedOff);
  int32_t* const pre = reinterpret_cast<int32_t*>(base + Lay::kPreOff);

  const int NR = p.num_reqs, R = p.R, c = blockIdx.x;
  constexpr int NW = kDecThreads / 32;

  // ---- 1. history pages per request -> exclusive prefix sums in smem
  {
    const int per = (NR + kDecThreads - 1) / kDecThreads;
    const int r0 = tid * per, r1 = min(NR, r0 + per);
    int sum = 0;
    for (int r = r0; r < r1; ++r) sum += hist_pages(__ldg(p.seq_lens + r), p.pt_stride);
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane == 31) warp_sum[warp] = incl;
    __syncthreads();
    int off = 0;
    for (int w = 0; w < warp; ++w) off += warp_sum[w];
    int run = off + incl - sum;
    for (int r = r0; r < r1; ++r) {
      pre[r] = run;
      run += hist_pages(__ldg(p.seq_lens + r), p.pt_stride);
    }
    if (tid == kDecThreads - 1) {
      int tot = 0;
      for (int w = 0; w < NW; ++w) tot += warp_sum[w];
      pre[NR] = tot;
    }
    __syncthreads();
  }
  const int64_t T = pre[NR];
  // Split the T pages over G = min(grid, T) CTAs: every one of them then owns
  // at least one page, so every CTA between a request's first and last owner
  // holds a segment of it (and writes the slot the merge reads).
  const int G = (int)min((int64_t)gridDim.x, T);
  if (c == 0) {
    for (int r = tid; r < NR; r += kDecThreads) {
      const int h = pre[r + 1] - pre[r];
      int2 info = make_int2(0, 0);
      if (h > 0) {
        const int cf = cta_of(pre[r], T, G), cl = cta_of(pre[r + 1] - 1, T, G);
        info = make_int2(cf, cl - cf + 1);
      }
      p.req_info[r] = info;
    }
  }
  if (c >= G) return;
  const int64_t x0 = (int64_t)c * T / G, x1 = (int64_t)(c + 1) * T / G;
  const int64_t n = x1 - x0;

  // ---- 2. tensor memory, barriers
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_base_s), kDecTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int s = 0; s < kDecStages; ++s) {
      mbar_init(smem_u32(&raw_full[s]), 1);
      mbar_init(smem_u32(&raw_empty[s]), 128);
    }
    for (int b = 0; b < kDecA; ++b) mbar_init(smem_u32(&a_full[b]), 128);
    for (int d = 0; d < kDecD; ++d) {
      mbar_init(smem_u32(&d_full[d]), 1);
      mbar_init(smem_u32(&d_empty[d]), 128);
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(smem_u32(&q_full[k]), 256);   // both dequant groups write the tile
      mbar_init(smem_u32(&q_empty[k]), 2);    // both MMA issuers commit
    }
    abort_s = 0;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_base_s;

  // first request of the range
  int r_start;
  {
    int lo = 0, hi = NR - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pre[mid] <= x0) lo = mid; else hi = mid - 1;
    }
    r_start = lo;
    while (pre[r_start + 1] - pre[r_start] == 0) ++r_start;
  }
  SegWalk walk{pre, NR, n, 0, r_start, (int)(x0 - pre[r_start])};
  auto fail = [&]() {
    if (!abort_s) {
      abort_s = 1;
      atomicOr(p.status, kStatusTimeout);
    }
  };

  if (warp == 0) {
    // ================================================= producer (TMA)
    // The whole warp walks the range; page ids are read 32 at a time (one
    // coalesced load), so no copy waits on a page-table read; lane 0 issues.
    int64_t g = 0;
    bool ok = true;
    while (walk.more() && ok) {
      const int je = walk.seg_end();
      const int32_t* row = p.page_table + (int64_t)walk.r * p.pt_stride;
      for (int jb = walk.j; jb < je && ok; jb += 32) {
        const int cnt = min(32, je - jb);
        const int my_phys = lane < cnt ? __ldg(row + jb + lane) : 0;
        for (int k = 0; k < cnt; ++k, ++g) {
          const int phys = __shfl_sync(0xffffffffu, my_phys, k);
          int issued = 1;
          if (lane == 0) {
            const int s = (int)(g % kDecStages);
            if (!mbar_wait_or_abort(smem_u32(&raw_empty[s]), (uint32_t)(((g / kDecStages) & 1) ^ 1), &abort_s)) {
              fail();
              issued = 0;
            } else {
              const uint32_t fb = smem_u32(&raw_full[s]);
              if (phys < 0 || phys >= p.num_blocks) {
                atomicOr(p.status, kStatusBadPage);
                mbar_arrive(fb);
              } else {
                mbar_arrive_expect_tx(fb, kPageBytes);
                bulk_g2s(sbase + Lay::kStageOff + s * kPageBytes, p.kv + (int64_t)phys * kPageBytes,
                         kPageBytes, fb);
              }
            }
          }
          if (!__shfl_sync(0xffffffffu, issued, 0)) {
            ok = false;
            break;
          }
        }
      }
      walk.g += je - walk.j;
      walk.j = je;
      if (ok && walk.more()) walk.next_request();
    }
    if (!ok && lane == 0) {   // drain issued copies before the CTA may exit
      for (int64_t k = (g > kDecStages ? g - kDecStages : 0); k < g; ++k)
        mbar_wait(smem_u32(&raw_full[k % kDecStages]), (uint32_t)((k / kDecStages) & 1));
    }
  } else if (warp == 1 || warp == 2) {
    // ================================================= MMA issuers
    if (lane == 0) {
      const int mgrp = warp - 1;                      // pages with g % 2 == mgrp
      constexpr uint32_t idesc = idesc_f16_f32(128, NQ);
      int64_t g = 0, g_last = -1;
      int sq = 0;
      while (walk.more() && !abort_s) {
        const int je = walk.seg_end();
        const int qs = sq & 1;
        if (!mbar_wait_or_abort(smem_u32(&q_full[qs]), (uint32_t)((sq >> 1) & 1), &abort_s)) { fail(); break; }
        const uint32_t qaddr = sbase + Lay::kQOff + qs * Lay::kQBytes;
        for (; walk.j < je; ++walk.j, ++walk.g, ++g) {
          if ((int)(g & 1) != mgrp) continue;
          const int b = (int)(g % kDecA);
          if (!mbar_wait_or_abort(smem_u32(&a_full[b]), (uint32_t)((g / kDecA) & 1), &abort_s)) { fail(); break; }
          if (!mbar_wait_or_abort(smem_u32(&d_empty[b]), (uint32_t)(((g / kDecD) & 1) ^ 1), &abort_s)) { fail(); break; }
          tc_fence_after();
          const uint32_t d_t = tbase + 256 + b * 64;
          const uint32_t a_t = tbase + b * 64;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t bdesc = smem_desc_sw128(qaddr + (kk >> 2) * (NQ * 128) + (kk & 3) * 32);
            mma_f16_tmemA(d_t, a_t + kk * 8, bdesc, idesc, kk > 0 ? 1u : 0u);
          }
          // one commit per page: d_full[b] also tells the dequant warps that
          // A buffer b is free again
          mma_commit(smem_u32(&d_full[b]));
          g_last = g;
        }
        if (abort_s) break;
        mma_commit(smem_u32(&q_empty[qs]));
        ++sq;
        if (walk.more()) walk.next_request();
      }
      if (abort_s && g_last >= 0) {   // drain issued MMAs before tensor memory is freed
        mbar_wait(smem_u32(&d_full[g_last % kDecD]), (uint32_t)((g_last / kDecD) & 1));
      }
    }
  } else if (warp < 11) {
    // ================================================= dequant warpgroups
    const int grp = (warp - 3) >> 2;                 // takes pages with g % 2 == grp
    const int tok = ((warp & 3) << 5) | lane;        // tensor-memory lane of this thread
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const int dq = tid - kDqTid0;                     // 0..255 (both groups share the query tile)
    int64_t g = 0;
    int sq = 0;
    bool ok = true;
    while (walk.more() && ok) {
      const int je = walk.seg_end();
      const int qs = sq & 1;
      // the request's queries -> fp16 B tile (128B swizzle, K-major)
      if (!__all_sync(0xffffffffu, mbar_wait_or_abort(smem_u32(&q_empty[qs]),
                                                       (uint32_t)(((sq >> 1) & 1) ^ 1), &abort_s))) {
        fail();
        break;
      }
      uint8_t* qt = base + Lay::kQOff + qs * Lay::kQBytes;
      for (int it = dq; it < NQ * 16; it += 256) {
        const int row = it >> 4, c8 = it & 15;
        uint4 o = make_uint4(0, 0, 0, 0);
        if (row < R) {
          const uint2 e = __ldg(reinterpret_cast<const uint2*>(p.q + ((int64_t)walk.r * R + row) * 128 + c8 * 8));
          o.x = e4m3x2_to_f16x2(e.x & 0xFFFFu);
          o.y = e4m3x2_to_f16x2(e.x >> 16);
          o.z = e4m3x2_to_f16x2(e.y & 0xFFFFu);
          o.w = e4m3x2_to_f16x2(e.y >> 16);
        }
        *reinterpret_cast<uint4*>(qt + (c8 >> 3) * (NQ * 128) + sw128_offset(row, c8 & 7)) = o;
      }
      fence_proxy_async_smem();
      mbar_arrive(smem_u32(&q_full[qs]));
      for (; walk.j < je; ++walk.j, ++walk.g, ++g) {
        if ((int)(g & 1) != grp) continue;
        const int s = (int)(g % kDecStages);
        if (!__all_sync(0xffffffffu, mbar_wait_or_abort(smem_u32(&raw_full[s]),
                                                         (uint32_t)((g / kDecStages) & 1), &abort_s))) {
          fail();
          ok = false;
          break;
        }
        uint32_t w[18];
        {
          const uint2* src = reinterpret_cast<const uint2*>(base + Lay::kStageOff + s * kPageBytes + tok * kRowBytes);
#pragma unroll
          for (int i = 0; i < 9; ++i) {
            const uint2 t2 = src[i];
            w[2 * i] = t2.x;
            w[2 * i + 1] = t2.y;
          }
        }
        mbar_arrive(smem_u32(&raw_empty[s]));
        uint32_t a[64];
        {
          const uint32_t sc[4] = {e4m3x2_to_f16x2(w[16] & 0xFFFFu), e4m3x2_to_f16x2(w[16] >> 16),
                                  e4m3x2_to_f16x2(w[17] & 0xFFFFu), e4m3x2_to_f16x2(w[17] >> 16)};
#pragma unroll
          for (int g8 = 0; g8 < 8; ++g8) {
            const uint32_t s2 = (g8 & 1) ? f16x2_bcast_hi(sc[g8 >> 1]) : f16x2_bcast_lo(sc[g8 >> 1]);
            dequant16(w[2 * g8], w[2 * g8 + 1], s2, a + 8 * g8);
          }
        }
        // A buffer b was last read by the MMAs of page g - kDecA, whose
        // completion is phase g / kDecA - 1 of d_full[b]; the next phase of
        // that barrier needs this page's A, so the parity cannot alias.
        const int b = (int)(g % kDecA);
        if (g >= kDecA &&
            !__all_sync(0xffffffffu, mbar_wait_or_abort(smem_u32(&d_full[b]),
                                                         (uint32_t)(((g / kDecA) - 1) & 1), &abort_s))) {
          fail();
          ok = false;
          break;
        }
        tc_fence_after();
        tmem_st_32x32b_x64(tbase + lane_base + b * 64, a);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(smem_u32(&a_full[b]));
      }
      ++sq;
      if (ok && walk.more()) walk.next_request();
    }
  } else {
    // ================================================= epilogue warpgroups
    // Group `grp` scores pages with g % 2 == grp and keeps its own running
    // top-15 per row; at a segment end group 1 hands its lists to group 0
    // through shared memory and group 0 merges and writes the result.  The
    // walk is never left early, so every barrier is always reached.
    const int grp = (warp - 11) >> 2;
    const int ep = (tid - kEpTid0) & 127;             // row owner within the group
    const int wq = warp & 3;                          // tensor-memory lane quarter
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const uint32_t bar_grp = 2 + grp, bar_both = 4;
    float2* const mrg = reinterpret_cast<float2*>(base + Lay::kMrgOff);   // [2][64][15] by segment parity
    constexpr int CW = NQ < 32 ? NQ : 32;             // columns per load + reduction pass
    TopK15 top;
    int64_t g = 0;
    int sq = 0;
    bool ok = true;                                   // uniform within the group
    while (walk.more()) {
      const int je = walk.seg_end();
      const int r = walk.r;
      const int seq_r = __ldg(p.seq_lens + r);
      const int pos = seq_r - p.qlen + ep / p.H;
      const int L = pos >= 0 ? (pos >> 7) : -1;
      // an unreadable page id anywhere in the segment: checked once, up front
      int seg_bad = 0;
      if (grp == 0) {
        for (int jj = walk.j + ep; jj < je; jj += 128) {
          const int ph = __ldg(p.page_table + (int64_t)r * p.pt_stride + jj);
          seg_bad |= (ph < 0 || ph >= p.num_blocks);
        }
      }
      top.reset();
      for (; walk.j < je; ++walk.j, ++walk.g, ++g) {
        if ((int)(g & 1) != grp) continue;
        const int d = (int)(g % kDecD);
        int wok = 0;
        if (ok) {
          wok = __all_sync(0xffffffffu, mbar_wait_or_abort(smem_u32(&d_full[d]),
                                                            (uint32_t)((g / kDecD) & 1), &abort_s));
          if (!wok) fail();
        }
        float* rd = red + (grp * 2 + ((g >> 1) & 1)) * (4 * NQ);
        if (wok) {
          tc_fence_after();
#pragma unroll
          for (int ch = 0; ch < NQ / CW; ++ch) {
            float v[CW];
            tmem_ld_row<CW>(tbase + lane_base + 256 + d * 64 + ch * CW, v);
            tmem_wait_ld();
            const float m = warp_colmax<CW>(v, lane);
            if (lane < CW) rd[wq * NQ + ch * CW + lane] = m;
          }
          tc_fence_before();
          mbar_arrive(smem_u32(&d_empty[d]));
        }
        ok = !named_bar_red_or(bar_grp, 128, (!wok || abort_s) ? 1 : 0);
        if (ok && ep < R) {
          const int jp = walk.j;
          const float sc = canon_zero(fmaxf(fmaxf(rd[ep], rd[NQ + ep]), fmaxf(rd[2 * NQ + ep], rd[3 * NQ + ep])));
          if (jp < L) {
            top.insert(sc, jp);
            if (p.scores_dbg) p.scores_dbg[((int64_t)r * R + ep) * p.dbg_stride + jp] = sc;
          }
        }
      }
      // ---- hand group 1's lists to group 0, merge, finalise the segment
      float2* mb = mrg + (sq & 1) * (kMaxRows * kHistK);
      if (grp == 1 && ep < R) {
#pragma unroll
        for (int k = 0; k < kHistK; ++k) mb[ep * kHistK + k] = make_float2(top.s[k], __int_as_float(top.id[k]));
      }
      named_bar_sync(bar_both, 256);
      if (grp == 0) {
        const int bad = named_bar_red_or(bar_grp, 128, seg_bad);
        if (ok) {
          const int cf = cta_of(pre[r], T, G), cl = cta_of(pre[r + 1] - 1, T, G);
          if (ep < R) {
            merge_top15(top, mb + ep * kHistK);
            if (cf == cl) {
              write_out_row(p.out + ((int64_t)r * R + ep) * kTopK, top.id, L, bad != 0);
            } else {
              float2* dst = p.cand + ((int64_t)(c + r) * R + ep) * kHistK;
#pragma unroll
              for (int k = 0; k < kHistK; ++k) dst[k] = make_float2(top.s[k], __int_as_float(top.id[k]));
            }
          }
          if (ep == 0 && cf != cl) p.slot_bad[c + r] = bad;
        }
      }
      ++sq;
      if (walk.more()) walk.next_request();
    }
  }

  // ---- free tensor memory once every role is done with it
  __syncwarp();   // lanes without a role wait here for their warp's lane 0
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tbase, kDecTmemCols);
}

// One warp per (request, row): merge the per-segment top-15 lists of split
// requests; write rows of requests with no history page or an unreadable one.
__global__ void __launch_bounds__(256) decode_merge_kernel(const DecodeParams p) {
  __shared__ float2 lists[8][32][kHistK];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t gw = (int64_t)blockIdx.x * 8 + warp;
  if (gw >= (int64_t)p.num_reqs * p.R) return;
  const int r = (int)(gw / p.R), n = (int)(gw % p.R);
  const int seq = __ldg(p.seq_lens + r);
  const int pos = seq - p.qlen + n / p.H;
  const int L = pos >= 0 ? (pos >> 7) : -1;
  const int hist = seq >= 1 ? (seq - 1) >> 7 : 0;
  int32_t* out_row = p.out + gw * kTopK;
  const int none[1] = {-1};
  if (hist > p.pt_stride) {
    if (lane == 0) {
      write_out_row(out_row, none, L, true);
      atomicOr(p.status, kStatusBadTable);
    }
    return;
  }
  const int2 info = p.req_info[r];
  const int nseg = info.y;
  if (nseg == 1) return;                      // finalised by the scoring kernel
  if (nseg == 0) {                            // no history page: local page only
    if (lane == 0) write_out_row(out_row, none, L, false);
    return;
  }
  const int slot0 = info.x + r;
  int bad = 0;
  for (int k = lane; k < nseg; k += 32) bad |= p.slot_bad[slot0 + k];
  if (__any_sync(0xffffffffu, bad)) {
    if (lane == 0) write_out_row(out_row, none, L, true);
    return;
  }
  // lane-local sorted list: list `lane` when nseg <= 32, else a top-15 of
  // lists lane, lane+32, ... (visited in ascending page order)
  float2(&mine)[kHistK] = lists[warp][lane];
  if (nseg <= 32) {
    if (lane < nseg) {
      const float2* src = p.cand + ((int64_t)(slot0 + lane) * p.R + n) * kHistK;
#pragma unroll
      for (int k = 0; k < kHistK; ++k) mine[k] = src[k];
    } else {
#pragma unroll
      for (int k = 0; k < kHistK; ++k) mine[k] = make_float2(0.0f, __int_as_float(-1));
    }
  } else {
    TopK15 t;
    t.reset();
    for (int k = lane; k < nseg; k += 32) {
      const float2* src = p.cand + ((int64_t)(slot0 + k) * p.R + n) * kHistK;
      float2 e[kHistK];
#pragma unroll
      for (int i = 0; i < kHistK; ++i) e[i] = src[i];
#pragma unroll
      for (int i = 0; i < kHistK; ++i)
        if (__float_as_int(e[i].y) >= 0) t.insert(e[i].x, __float_as_int(e[i].y));
    }
#pragma unroll
    for (int k = 0; k < kHistK; ++k) mine[k] = make_float2(t.s[k], __int_as_float(t.id[k]));
  }
  __syncwarp();
  int res[kHistK];
  int cur = 0;
#pragma unroll
  for (int k = 0; k < kHistK; ++k) {
    float2 e = make_float2(0.0f, __int_as_float(-1));
    if (cur < kHistK) e = lists[warp][lane][cur];
    const int id = __float_as_int(e.y);
    const uint32_t key = id >= 0 ? order_key(e.x) : 0u;
    const uint32_t kmax = warp_max_u32(key);
    const uint32_t idmin = warp_min_u32(key == kmax && kmax != 0u ? (uint32_t)id : 0xFFFFFFFFu);
    if (kmax != 0u && key == kmax && (uint32_t)id == idmin) ++cur;
    res[k] = kmax != 0u ? (int)idmin : -1;
  }
  if (lane == 0) write_out_row(out_row, res, L, false);
}

template <int NQ>
static cudaError_t launch_decode_nq(const DecodeParams& p, int grid, cudaStream_t stream) {
  const size_t smem = DecLayout<NQ>::bytes(p.num_reqs);
  cudaError_t e = cudaFuncSetAttribute(decode_score_kernel<NQ>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  decode_score_kernel<NQ><<<grid, kDecThreads, smem, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t warps = (int64_t)p.num_reqs * p.R;
  decode_merge_kernel<<<(unsigned)((warps + 7) / 8), 256, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_decode(const DecodeParams& p, int grid, cudaStream_t stream) {
  switch (decode_nq(p.R)) {
    case 16: return launch_decode_nq<16>(p, grid, stream);
    case 32: return launch_decode_nq<32>(p, grid, stream);
    default: return launch_decode_nq<64>(p, grid, stream);
  }
}

}  // namespace nvfp4idx
