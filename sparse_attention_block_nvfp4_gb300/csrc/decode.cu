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
// as segments (one per request it touches) and each segment as quads of up
// to 4 consecutive pages.  A quad passes through the tensor core as 4 slices:
// slice s holds tokens [32s, 32s+32) of the quad's 4 pages, page q of the
// quad in tensor-memory lanes [32q, 32q+32).  So the MMA of slice s,
// D[lane][row] = K_slice . Q^T, gives the warp that owns lane quarter q the
// scores of 32 tokens of ITS page; after the 4 slices that warp has seen all
// 128 tokens of the page and takes the max over them alone: an in-register
// max over the slices, then a reduction over its 32 lanes, with no exchange
// between warps.  One CTA per SM, 16 or 20 warps, one role per warpgroup (so that
// setmaxnreg can move registers to the epilogue), linked by mbarrier rings
// (slice s of every quad uses A buffer s and D buffer s):
//   * warpgroup 0 (88 / 80 registers): warp 0 reads page ids 32 at a time and has
//     the TMA unit copy each 9216-byte page into a 16-stage shared ring
//     (cp.async.bulk, transaction-count completion); warps 1 / 2 (slices of
//     even / odd index) each have one thread issue the 8 tcgen05.mma (K = 16)
//     of a slice into D buffer s and commit once (a single thread cannot
//     issue small-N MMAs as fast as the tensor core retires them); warp 3
//     idles;
//   * warpgroups 1 / 2 (dequant, 112 / 96 registers, quads of even / odd index): warp q reads the
//     72-byte rows of tokens 32s + lane of page q, dequantises them exactly to
//     fp16 (E2M1 x E4M3 fits fp16) and stores them into its lane quarter of A
//     buffer s (tcgen05.st), the MMA's A operand (M = 128 lanes, K = 128); at
//     each segment start both widen the request's E4M3 queries to fp16 into a
//     128B-swizzled B tile (double buffered);
//   * warpgroup 3, and 4 when a request has 64 rows (epilogue, 200 / 104
//     registers): warp q owns page q (with two warpgroups warps q and q + 4
//     split its rows in two halves); it keeps the running max of the page's
//     tokens over the 4 slices for its rows, reduces it over its lanes
//     (butterfly shuffles that leave column k in lane k), and lane k inserts
//     the page score of its row into the row's running top-15 in registers;
//     at a segment end the four warps' lists of each row are merged.
//   The register figures are for 16 / 20 warps.
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

constexpr int kQuadSlots = 4;            // raw page ring: quad kq fills stages 4 * (kq % 4) + q
constexpr int kDecStages = 4 * kQuadSlots;
constexpr int kDecSlices = 4;            // slice s: A buffer s (columns [64s, 64s+64))
// One role per warpgroup, so that setmaxnreg can move registers between
// them: warpgroup 0 = warp 0 TMA, warps 1 / 2 MMA issue, warp 3 idle;
// warpgroups 1 / 2 dequant; then one epilogue warpgroup, or two when a
// request has 64 rows (each then takes half of every page's rows).
constexpr int kDqTid0 = 128, kEpTid0 = 384, kEpWarp0 = 12;
constexpr int kDecMaxThreads = 640;
template <int NQ>
struct DecRoles {
  static constexpr int kEpGroups = NQ == 64 ? 2 : 1;
  static constexpr int kThreads = 384 + 128 * kEpGroups;
  static constexpr int kEpThreads = 128 * kEpGroups;
  // 512 threads launch with 128 registers each, 640 with 96; the role
  // shares add up to at most the launch allocation:
  // 128 x 88 + 256 x 112 + 128 x 200 = 65536 = 512 x 128 and
  // 128 x 80 + 256 x 96 + 256 x 104 = 61440 = 640 x 96.
  static constexpr uint32_t kRegsLaunch = kEpGroups == 2 ? 96 : 128;
  static constexpr uint32_t kRegsCtl = kEpGroups == 2 ? 80 : 88;
  static constexpr uint32_t kRegsDq = kEpGroups == 2 ? 96 : 112;
  static constexpr uint32_t kRegsEpi = kEpGroups == 2 ? 104 : 200;
  static_assert(128 * kRegsCtl + 256 * kRegsDq + kEpThreads * kRegsEpi <= kThreads * kRegsLaunch,
                "setmaxnreg shares exceed the launch allocation");
};
constexpr uint32_t kDecTmemCols = 512;

// D buffers in tensor memory from column 256: for NQ <= 32 two sets of four
// 32-column buffers (quad kq uses set kq % 2, so the epilogue may lag the MMAs
// by a quad), for NQ = 64 one set of four 64-column buffers.
template <int NQ>
struct DecD {
  static constexpr int kSets = NQ <= 32 ? 2 : 1;
  static constexpr int kCols = NQ <= 32 ? 32 : 64;
  __device__ static __forceinline__ int set(int64_t kq) { return kSets == 2 ? (int)(kq & 1) : 0; }
  // parity of the epilogue's release of quad kq's D buffer
  __device__ static __forceinline__ uint32_t phase(int64_t kq) {
    return (uint32_t)((kSets == 2 ? (kq >> 1) : kq) & 1);
  }
  __device__ static __forceinline__ uint32_t col(int64_t kq, int sl) {
    return 256u + (uint32_t)((set(kq) * kDecSlices + sl) * kCols);
  }
};

template <int NQ, class PF>   // PF: page format (codec.cuh)
struct DecLayout {
  static constexpr uint32_t kQBytes = NQ * 256;                   // 16-bit [2][NQ][64], SW128
  static constexpr uint32_t kQOff = 0;                             // two query tiles
  static constexpr uint32_t kStageOff = 2 * kQBytes;               // multiple of 1024
  static constexpr uint32_t kListOff = kStageOff + kDecStages * PF::kPageBytes;  // [4 warps][64 rows][15] (score, id)
  static constexpr uint32_t kPreOff = kListOff + 4 * kMaxRows * kHistK * 8;
  // one CTA per SM: it holds all 512 tensor-memory columns
  static size_t bytes(int num_reqs) {
    const size_t b = 1024 + kPreOff + (size_t)(num_reqs + 1) * 4;
    return b < 120 * 1024 ? 120 * 1024 : b;
  }
};
static_assert(1024 + DecLayout<64, Nvfp4Pages>::kPreOff + (kMaxDecodeReqs + 1) * 4 + 1024 <= 227 * 1024 &&
                  1024 + DecLayout<64, Mxfp4Pages>::kPreOff + (kMaxDecodeReqs + 1) * 4 + 1024 <= 227 * 1024,
              "decode shared memory above the 227 KB a CTA may hold");

__device__ __forceinline__ int hist_pages(int seq_len, int pt_stride) {
  const int h = seq_len >= 1 ? (seq_len - 1) >> 7 : 0;
  return h > pt_stride ? 0 : h;   // a history wider than the table is finalised as bad by the merge
}

// First history page request r scores (0, or its context-parallel share's).
__device__ __forceinline__ int req_lo(const DecodeParams& p, int r) {
  return p.page_lo ? max(0, __ldg(p.page_lo + r)) : 0;
}
// Pages request r scores: its history, cut to [page_lo, page_hi) for a
// context-parallel share.
__device__ __forceinline__ int req_pages(const DecodeParams& p, int r) {
  const int h = hist_pages(__ldg(p.seq_lens + r), p.pt_stride);
  if (!p.page_lo) return h;
  const int hi = min(h, __ldg(p.page_hi + r));
  return max(0, hi - req_lo(p, r));
}

// A row's 15 candidates (score, page id), sorted, for a context-parallel
// merge; an unreadable request marks its list with id -2 first.
__device__ __forceinline__ void write_cand_row(float2* row, const float* s, const int* id, bool bad) {
#pragma unroll
  for (int k = 0; k < kHistK; ++k) {
    const int i = bad ? (k == 0 ? -2 : -1) : id[k];
    row[k] = make_float2(i >= 0 ? s[k] : 0.0f, __int_as_float(i));
  }
}

// CTA owning global page x when T pages are split over G CTAs.
__device__ __forceinline__ int cta_of(int64_t x, int64_t T, int G) {
  return (int)(((x + 1) * G - 1) / T);
}

// Column maxima over the warp's 32 lanes by butterfly transpose-reduction:
// at step H each lane keeps half of its columns, sends the other half to
// lane ^ H and takes the max with what it receives (H shuffles).  For N = 32
// columns, lane l ends with column l (31 shuffles in all, against 32
// warp-wide reductions column by column); for N = 16 (8), two (four) lanes
// finish each column with one (two) more shuffles, and lane l ends with
// column l & 15 (l & 7).  v is overwritten.
template <int H>
__device__ __forceinline__ void colmax_step(float* v, int lane) {
  const bool up = (lane & H) != 0;
#pragma unroll
  for (int i = 0; i < H; ++i) {
    const float keep = up ? v[i + H] : v[i];
    const float send = up ? v[i] : v[i + H];
    v[i] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, H));
  }
}
template <int N>
__device__ __forceinline__ float warp_colmax(float* v, int lane) {
  static_assert(N == 8 || N == 16 || N == 32, "8, 16 or 32 columns");
  if constexpr (N == 32) colmax_step<16>(v, lane);
  if constexpr (N >= 16) colmax_step<8>(v, lane);
  colmax_step<4>(v, lane);
  colmax_step<2>(v, lane);
  colmax_step<1>(v, lane);
  float m = v[0];
  if constexpr (N == 8) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
  if constexpr (N <= 16) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
  return m;
}

// Merge the four sorted lists of `row` ([4][64][15] in shared memory) into
// the top 15 by score, equal scores by lower id.
__device__ __forceinline__ void merge4_top15(const float2* lists, int row, float (&s)[kHistK],
                                             int (&id)[kHistK]) {
  int h[4] = {0, 0, 0, 0};
#pragma unroll
  for (int k = 0; k < kHistK; ++k) {
    float bs = -CUDART_INF_F;
    int bi = -1, bw = -1;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      if (h[w] < kHistK) {
        const float2 e = lists[(w * kMaxRows + row) * kHistK + h[w]];
        const int ei = __float_as_int(e.y);
        if (ei >= 0 && (bw < 0 || e.x > bs || (e.x == bs && ei < bi))) {
          bs = e.x;
          bi = ei;
          bw = w;
        }
      }
    }
    s[k] = bs;
    id[k] = bi;
#pragma unroll
    for (int w = 0; w < 4; ++w) h[w] += (bw == w) ? 1 : 0;
  }
}

// The CTA's walk over its page range, identical in every role.
struct SegWalk {
  const int32_t* pre;
  int NR;
  int64_t n;        // pages in the range
  int64_t g;        // pages walked
  int r, j;         // current request, page (logical id)
  __device__ __forceinline__ bool more() const { return g < n; }
  // pages [j, j_end) of request r form the current segment
  __device__ __forceinline__ int seg_end(const DecodeParams& p) const {
    const int end = req_lo(p, r) + (pre[r + 1] - pre[r]);
    const int64_t left = n - g;
    return (int)((int64_t)end < (int64_t)j + left ? (int64_t)end : (int64_t)j + left);
  }
  __device__ __forceinline__ void next_request(const DecodeParams& p) {
    ++r;
    while (r < NR && pre[r + 1] - pre[r] == 0) ++r;
    j = r < NR ? req_lo(p, r) : 0;
  }
};

// The rows of a segment whose scores a run-out wait left incomplete: -1
// rows for a request the CTA finalises, else a bad slot for the merge.  Out
// of line, so that the epilogue's loop keeps its code and registers.
__device__ __noinline__ void decode_segment_failed(const DecodeParams& p, const int32_t* pre, int64_t T, int G,
                                                   int r, int c, int ep, int R) {
  const int cf = cta_of(pre[r], T, G), cl = cta_of(pre[r + 1] - 1, T, G);
  if (cf == cl && ep < R) {
    const float zs[kHistK] = {};
    const int none[kHistK] = {-1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1};
    if (p.cand_out) write_cand_row(p.cand_out + ((int64_t)r * R + ep) * kHistK, zs, none, true);
    else write_out_row(p.out + ((int64_t)r * R + ep) * kTopK, none, -1, true);
  }
  if (ep == 0 && cf != cl) p.slot_bad[c + r] = 1;
}

template <int NQ, class PF>
__global__ void __launch_bounds__(DecRoles<NQ>::kThreads, 1) decode_score_kernel(const DecodeParams p) {
  using Lay = DecLayout<NQ, PF>;
  using Roles = DecRoles<NQ>;
  constexpr int kDecThreads = Roles::kThreads;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t raw_full[kDecStages], raw_empty[kDecStages];
  __shared__ __align__(8) uint64_t a_full[kDecSlices];
  // d_full[h][s]: MMAs of slice s of the quads kq with kq % 2 == h are done.
  // Split by quad parity so that every waiter takes each barrier's phases in
  // order (a parity wait on phase k passes wrongly at phase k - 1 and blocks
  // at phase k + 2): the epilogue waits d_full[kq % 2] at quad kq, and the
  // dequant group of quad kq (A buffer free) waits d_full[(kq - 1) % 2].
  __shared__ __align__(8) uint64_t d_full[2][kDecSlices], d_empty[2][kDecSlices];
  __shared__ __align__(8) uint64_t q_full[2], q_empty[2];
  __shared__ uint32_t tmem_base_s;
  __shared__ volatile int abort_s;
  __shared__ int warp_sum[kDecMaxThreads / 32];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint64_t lim = p.wait_ns;                    // limit of every bounded wait
  griddep_launch_dependents();                       // the merge kernel may be scheduled
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t sbase = (raw_u32 + 1023u) & ~1023u;
  uint8_t* const base = smem_raw + (sbase - raw_u32);
  int32_t* const pre = reinterpret_cast<int32_t*>(base + Lay::kPreOff);

  const int NR = p.num_reqs, R = p.R, c = blockIdx.x;
  constexpr int NW = kDecThreads / 32;

  // ---- 1. history pages per request -> exclusive prefix sums in smem
  {
    const int per = (NR + kDecThreads - 1) / kDecThreads;
    const int r0 = tid * per, r1 = min(NR, r0 + per);
    int sum = 0;
    for (int r = r0; r < r1; ++r) sum += req_pages(p, r);
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
      run += req_pages(p, r);
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
      mbar_init(smem_u32(&raw_empty[s]), 32);   // one dequant warp reads a page
    }
    // every thread of a role arrives for itself as soon as its own part is
    // done (one arrival per warp after a __syncwarp measured 2.5 us slower
    // per call on long_mixed)
    for (int b = 0; b < kDecSlices; ++b) {
      mbar_init(smem_u32(&a_full[b]), 128);     // the quad's dequant warpgroup
      mbar_init(smem_u32(&d_full[0][b]), 1);    // MMA commit
      mbar_init(smem_u32(&d_full[1][b]), 1);
      mbar_init(smem_u32(&d_empty[0][b]), Roles::kEpThreads);   // the epilogue warpgroup(s)
      mbar_init(smem_u32(&d_empty[1][b]), Roles::kEpThreads);
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
  SegWalk walk{pre, NR, n, 0, r_start, req_lo(p, r_start) + (int)(x0 - pre[r_start])};
  auto fail = [&]() {
    if (!abort_s) {
      abort_s = 1;
      atomicOr(p.status, kStatusTimeout);
    }
  };

  if (warp < 4) {
    // warpgroup 0 gives registers back to the epilogue (executed by all
    // four warps of the warpgroup, warp 3 has no other role)
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(Roles::kRegsCtl));
    if (warp == 0) {
      // ================================================= producer (TMA)
      // Quad kq fills stages 4 * (kq % 4) + q, q < 4; a page missing from a
      // partial quad gets an arrival without data.  So stage s is filled once
      // every four quads and read by one warp only (warp q of the dequant group
      // of parity kq % 2), which waits its phases in order (an mbarrier parity
      // wait cannot tell phase k from phase k + 2).  Up to four quads are in
      // the ring: two being dequantised, two in flight from memory.
      // The whole warp walks the range and reads page ids 32 at a time (one
      // coalesced load; 32 is a multiple of the quad); lane 0 issues.
      int64_t kq = 0;
      int64_t last = -1;                                // lane s < 16: last quad that filled stage s
      bool ok = true;
      while (walk.more() && ok) {
        const int je = walk.seg_end(p);
        const int32_t* row = p.page_table + (int64_t)walk.r * p.pt_stride;
        for (int jb = walk.j; jb < je && ok; jb += 32) {
          const int cnt = min(32, je - jb);
          const int my_phys = lane < cnt ? __ldg(row + jb + lane) : 0;
          for (int k = 0; k < cnt && ok; k += 4, ++kq) {
#pragma unroll 1
            for (int q = 0; q < 4; ++q) {
              const int phys = __shfl_sync(0xffffffffu, my_phys, (k + q) & 31);
              const int s = 4 * (int)(kq % kQuadSlots) + q;
              int issued = 1;
              if (lane == 0) {
                if (!mbar_wait_or_abort(smem_u32(&raw_empty[s]), (uint32_t)(((kq / kQuadSlots) & 1) ^ 1),
                                        &abort_s, lim)) {
                  fail();
                  issued = 0;
                } else {
                  const uint32_t fb = smem_u32(&raw_full[s]);
                  if (k + q >= cnt) {
                    mbar_arrive(fb);
                  } else if (phys < 0 || phys >= p.num_blocks) {
                    atomicOr(p.status, kStatusBadPage);
                    mbar_arrive(fb);
                  } else {
                    mbar_arrive_expect_tx(fb, PF::kPageBytes);
                    bulk_g2s(sbase + Lay::kStageOff + s * PF::kPageBytes, p.kv + (int64_t)phys * PF::kPageBytes,
                             PF::kPageBytes, fb);
                  }
                }
              }
              if (!__shfl_sync(0xffffffffu, issued, 0)) {
                ok = false;
                break;
              }
              if (lane == s) last = kq;
            }
          }
        }
        walk.g += je - walk.j;
        walk.j = je;
        if (ok && walk.more()) walk.next_request(p);
      }
      // wait for every copy this warp issued before the CTA may exit: the
      // readers of a stage stop waiting once another role's wait ran out
      if (lane < kDecStages && last >= 0)
        mbar_wait(smem_u32(&raw_full[lane]), (uint32_t)((last / kQuadSlots) & 1));
    } else if (warp == 1 || warp == 2) {
      // ================================================= MMA issuers
      // Issuer m takes slices m and m + 2 of every quad.
      if (lane == 0) {
        const int m = warp - 1;
        constexpr uint32_t idesc = idesc_f16_f32(128, NQ, PF::kBf16);
        int64_t kq = 0;
        uint32_t last_bar = 0, last_par = 0;
        int sq = 0;
        while (walk.more() && !abort_s) {
          const int je = walk.seg_end(p);
          const int qs = sq & 1;
          if (!mbar_wait_or_abort(smem_u32(&q_full[qs]), (uint32_t)((sq >> 1) & 1), &abort_s, lim)) { fail(); break; }
          const uint32_t qaddr = sbase + Lay::kQOff + qs * Lay::kQBytes;
          // B (query) descriptors of the 8 K steps of this segment
          uint64_t bd[8];
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            bd[kk] = desc_advance(smem_desc_sw128(qaddr), (uint32_t)((kk >> 2) * (NQ * 128) + (kk & 3) * 32));
          bool ok = true;
          for (; walk.j < je && ok; ++kq) {
            const int npq = min(4, je - walk.j);
            walk.j += npq;
            walk.g += npq;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int sl = m + 2 * h;
              if (!mbar_wait_or_abort(smem_u32(&a_full[sl]), (uint32_t)(kq & 1), &abort_s, lim) ||
                  !mbar_wait_or_abort(smem_u32(&d_empty[DecD<NQ>::set(kq)][sl]), DecD<NQ>::phase(kq) ^ 1u,
                                      &abort_s, lim)) {
                fail();
                ok = false;
                break;
              }
              tc_fence_after();
              const uint32_t d_t = tbase + DecD<NQ>::col(kq, sl);
              uint32_t at[8];
#pragma unroll
              for (int kk = 0; kk < 8; ++kk) at[kk] = tbase + sl * 64 + kk * 8;
              // the slice's 8 MMAs and one commit: d_full also tells the
              // dequant warps that A buffer sl is free
              mma8_f16_ts_commit(d_t, at, bd, idesc, smem_u32(&d_full[kq & 1][sl]));
              last_bar = smem_u32(&d_full[kq & 1][sl]);
              last_par = (uint32_t)((kq >> 1) & 1);
            }
          }
          if (!ok || abort_s) break;
          mma_commit(smem_u32(&q_empty[qs]));
          ++sq;
          if (walk.more()) walk.next_request(p);
        }
        // a commit covers every MMA issued before it: wait for the last one
        // before tensor memory may be freed (the epilogue stops waiting once
        // another role's wait ran out)
        if (last_bar != 0) mbar_wait(last_bar, last_par);
      }
    }
  } else if (warp < 12) {
    // ================================================= dequant warpgroups
    if constexpr (Roles::kRegsDq < Roles::kRegsLaunch)
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(Roles::kRegsDq));
    // Group grp takes the quads of parity grp; warp q (tensor-memory lanes
    // [32q, 32q+32)) dequantises page q of the quad, one 32-token slice at a
    // time, into its lane quarter of A buffer s.  A warp of a partial quad
    // with no page still takes part in every barrier (its lanes of the A
    // buffer then hold stale finite values whose scores nobody reads).
    const int grp = (warp - 4) >> 2;
    const int q = warp & 3;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    const int dq = tid - kDqTid0;                     // 0..255 (both groups share the query tile)
    int64_t kq = 0;
    int sq = 0;
    bool ok = true;
    while (walk.more() && ok) {
      const int je = walk.seg_end(p);
      const int qs = sq & 1;
      // the request's queries -> fp16 B tile (128B swizzle, K-major)
      if (!__all_sync(0xffffffffu, mbar_wait_or_abort(smem_u32(&q_empty[qs]),
                                                       (uint32_t)(((sq >> 1) & 1) ^ 1), &abort_s, lim))) {
        fail();
        break;
      }
      uint8_t* qt = base + Lay::kQOff + qs * Lay::kQBytes;
      for (int it = dq; it < NQ * 16; it += 256) {
        const int row = it >> 4, c8 = it & 15;
        uint4 o = make_uint4(0, 0, 0, 0);
        if (row < R) {
          const uint2 e = __ldg(reinterpret_cast<const uint2*>(p.q + ((int64_t)walk.r * R + row) * 128 + c8 * 8));
          o.x = PF::widen_q(e.x & 0xFFFFu);
          o.y = PF::widen_q(e.x >> 16);
          o.z = PF::widen_q(e.y & 0xFFFFu);
          o.w = PF::widen_q(e.y >> 16);
        }
        *reinterpret_cast<uint4*>(qt + (c8 >> 3) * (NQ * 128) + sw128_offset(row, c8 & 7)) = o;
      }
      fence_proxy_async_smem();
      mbar_arrive(smem_u32(&q_full[qs]));
      for (; walk.j < je && ok; ++kq) {
        const int npq = min(4, je - walk.j);
        walk.j += npq;
        walk.g += npq;
        if ((int)(kq & 1) != grp) continue;
        const bool has = q < npq;
        const int st = 4 * (int)(kq % kQuadSlots) + q;  // this warp's stage (see the producer)
        if (!__all_sync(0xffffffffu, mbar_wait_or_abort(smem_u32(&raw_full[st]),
                                                         (uint32_t)((kq / kQuadSlots) & 1), &abort_s, lim))) {
          fail();
          ok = false;
          break;
        }
        if (!has) mbar_arrive(smem_u32(&raw_empty[st]));
        const uint8_t* const page = base + Lay::kStageOff + st * PF::kPageBytes;
#pragma unroll 1
        for (int sl = 0; sl < kDecSlices; ++sl) {
          uint32_t a[64];
          if (has) {
            typename PF::Row row;
            PF::load(page, sl * 32 + lane, row);
            if (sl == kDecSlices - 1) mbar_arrive(smem_u32(&raw_empty[st]));
#pragma unroll
            for (int g8 = 0; g8 < 8; ++g8) PF::chunk16(row, g8, a + 8 * g8);
          }
          // A buffer sl is free once the MMAs of quad kq - 1 are done
          if (kq >= 1 &&
              !__all_sync(0xffffffffu, mbar_wait_or_abort(smem_u32(&d_full[(kq - 1) & 1][sl]),
                                                           (uint32_t)(((kq - 1) >> 1) & 1), &abort_s, lim))) {
            fail();
            ok = false;
            break;
          }
          if (has) {
            tc_fence_after();
            tmem_st_32x32b_x64(tbase + lane_base + sl * 64, a);
            tmem_wait_st();
          }
          tc_fence_before();
          mbar_arrive(smem_u32(&a_full[sl]));
        }
      }
      ++sq;
      if (ok && walk.more()) walk.next_request(p);
    }
  } else {
    // ================================================= epilogue warpgroup(s)
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(Roles::kRegsEpi));
    // Warp q of an epilogue warpgroup owns page q of every quad (tensor-
    // memory lanes [32q, 32q+32)); with two warpgroups, warps q and q + 4
    // split its NQ rows and half hf takes rows [hf * NH, (hf + 1) * NH).  Per
    // slice a warp loads its lanes' NH columns of D buffer s and keeps the
    // running max over slices; after the 4th slice a butterfly transpose-
    // reduction over the lanes gives the page score of each of its rows (row
    // hf * NH + k in lane k).  That lane keeps the running top-15 of its row
    // in registers; at a segment end the lists go through shared memory and
    // the four warps' lists of each row are merged.  The walk is never left
    // early, so every barrier is always reached.
    constexpr int NH = NQ / Roles::kEpGroups;         // rows per warp (<= 32)
    const int q = warp & 3;
    const int hf = (warp - kEpWarp0) >> 2;
    const int ep = tid - kEpTid0;                     // row owner at the merge
    const int myrow = hf * NH + (lane & (NH - 1));    // lanes < NH hold a distinct row
    const bool row_lane = lane < NH;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    float2* const lists = reinterpret_cast<float2*>(base + Lay::kListOff);   // [4][64][15]
    float2* const my = lists + (q * kMaxRows + myrow) * kHistK;
    constexpr int CW = Roles::kEpGroups == 2 ? 16 : NH;   // columns per load + max pass
    int64_t kq = 0;
    bool ok = true;                                   // uniform within the warp
    while (walk.more()) {
      const int je = walk.seg_end(p);
      const int r = walk.r;
      const int seq_r = __ldg(p.seq_lens + r);
      const int pos = seq_r - p.qlen + myrow / p.H;
      const int L = pos >= 0 ? (pos >> 7) : -1;
      // an unreadable page id anywhere in the segment: checked once, up front
      int seg_bad = 0;
      for (int jj = walk.j + ep; jj < je; jj += Roles::kEpThreads) {
        const int ph = __ldg(p.page_table + (int64_t)r * p.pt_stride + jj);
        seg_bad |= (ph < 0 || ph >= p.num_blocks);
      }
      TopK15 top;
      top.reset();
      for (; walk.j < je; ++kq) {
        const int npq = min(4, je - walk.j);
        const int jp = walk.j + q;                    // this warp's page
        const bool has = q < npq;
        walk.j += npq;
        walk.g += npq;
        float run[NH];
#pragma unroll
        for (int sl = 0; sl < kDecSlices; ++sl) {
          if (ok) {
            ok = __all_sync(0xffffffffu, mbar_wait_or_abort(smem_u32(&d_full[kq & 1][sl]),
                                                             (uint32_t)((kq >> 1) & 1), &abort_s, lim));
            if (!ok) fail();
          }
          if (ok) {
            tc_fence_after();
            if (has) {
              const uint32_t ta = tbase + lane_base + DecD<NQ>::col(kq, sl) + (uint32_t)(hf * NH);
              if (sl == 0) {
                tmem_ld_row<NH>(ta, run);
                tmem_wait_ld();
              } else {
#pragma unroll
                for (int ch = 0; ch < NH / CW; ++ch) {
                  float t[CW];
                  tmem_ld_row<CW>(ta + ch * CW, t);
                  tmem_wait_ld();
#pragma unroll
                  for (int i = 0; i < CW; ++i) run[ch * CW + i] = fmaxf(run[ch * CW + i], t[i]);
                }
              }
            }
            tc_fence_before();
            mbar_arrive(smem_u32(&d_empty[DecD<NQ>::set(kq)][sl]));
          }
        }
        if (ok && has) {
          // the warp's rows: max over its 32 token lanes
          const float m = canon_zero(warp_colmax<NH>(run, lane));
          if (row_lane && myrow < R && jp < L) {
            top.insert(m, jp);
            if (p.scores_dbg) p.scores_dbg[((int64_t)r * R + myrow) * p.dbg_stride + jp] = m;
          }
        }
      }
      // ---- merge the four warps' lists of each row, finalise the segment
      if (row_lane) {
#pragma unroll
        for (int k = 0; k < kHistK; ++k) my[k] = make_float2(top.s[k], __int_as_float(top.id[k]));
      }
      const int bad = named_bar_red_or(2, Roles::kEpThreads, seg_bad);
      const int failed = named_bar_red_or(3, Roles::kEpThreads, (!ok || abort_s) ? 1 : 0);
      if (!failed) {
        const int cf = cta_of(pre[r], T, G), cl = cta_of(pre[r + 1] - 1, T, G);
        if (ep < R) {
          float ts[kHistK];
          int ti[kHistK];
          merge4_top15(lists, ep, ts, ti);
          const int pe = seq_r - p.qlen + ep / p.H;
          if (cf == cl) {
            if (p.cand_out) write_cand_row(p.cand_out + ((int64_t)r * R + ep) * kHistK, ts, ti, bad != 0);
            else write_out_row(p.out + ((int64_t)r * R + ep) * kTopK, ti, pe >= 0 ? (pe >> 7) : -1, bad != 0);
          } else {
            float2* dst = p.cand + ((int64_t)(c + r) * R + ep) * kHistK;
#pragma unroll
            for (int k = 0; k < kHistK; ++k) dst[k] = make_float2(ts[k], __int_as_float(ti[k]));
          }
        }
        if (ep == 0 && cf != cl) p.slot_bad[c + r] = bad;
      } else {
        // a wait ran out: the scores are incomplete, so the segment's rows
        // become -1 (a request this CTA finalises) or its slot is flagged
        // bad, so that the merge writes -1 rows instead of reading
        // candidates this call never wrote
        decode_segment_failed(p, pre, T, G, r, c, ep, R);
      }
      named_bar_sync(2, Roles::kEpThreads);           // lists are read before the next reset
      if (walk.more()) walk.next_request(p);
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
// W warps per CTA; lane k holds kHeads lists, k + 32h (h < kHeads), and with
// more than 32 kHeads segments each of them is the top-15 of lists k + 32h,
// k + 32h + 32 kHeads, ... (ascending page ranges).  15 warp-wide rounds then
// take the best head (score desc, id asc) of all of them.  The quad kernel's
// requests (a few segments each) take <8, 1>; the small-row kernel's warps
// (dozens of segments per request) take <4, 2>.
template <int W, int kHeads>
__global__ void __launch_bounds__(W * 32) decode_merge_kernel(const DecodeParams p) {
  static_assert(kHeads == 1 || kHeads == 2, "one or two lists per lane");
  griddep_wait();                                    // the scoring grid's candidates are written
  constexpr int kLists = 32 * kHeads;
  __shared__ float2 lists[W][kLists][kHistK];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t gw = (int64_t)blockIdx.x * W + warp;
  if (gw >= (int64_t)p.num_reqs * p.R) return;
  const int r = (int)(gw / p.R), n = (int)(gw % p.R);
  const int seq = __ldg(p.seq_lens + r);
  const int2 info = p.req_info[r];                   // loaded with seq, not after it
  const int pos = seq - p.qlen + n / p.H;
  const int L = pos >= 0 ? (pos >> 7) : -1;
  const int hist = seq >= 1 ? (seq - 1) >> 7 : 0;
  int32_t* out_row = p.out + gw * kTopK;
  float2* cand_row = p.cand_out ? p.cand_out + gw * kHistK : nullptr;   // context-parallel share
  const int none[kHistK] = {-1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1};
  const float zs[kHistK] = {};
  auto finish = [&](const float* s, const int* id, bool bad) {   // lane 0
    if (cand_row) write_cand_row(cand_row, s, id, bad);
    else write_out_row(out_row, id, L, bad);
  };
  if (hist > p.pt_stride) {
    if (lane == 0) {
      finish(zs, none, true);
      atomicOr(p.status, kStatusBadTable);
    }
    return;
  }
  const int nseg = info.y;
  if (nseg == 1) return;                      // finalised by the scoring kernel
  if (nseg == 0) {                            // no history page (in the share): local page only
    if (lane == 0) finish(zs, none, false);
    return;
  }
  const int slot0 = info.x + r;
  // up to kLists lists: loaded into registers together with the segments'
  // bad flags (one memory latency, not two; dropped if a flag is set)
  float2 e[kHeads][kHistK];
  if (nseg <= kLists) {
#pragma unroll
    for (int hh = 0; hh < kHeads; ++hh) {
      const int li = lane + 32 * hh;
      if (li < nseg) {
        const float2* src = p.cand + ((int64_t)(slot0 + li) * p.R + n) * kHistK;
#pragma unroll
        for (int k = 0; k < kHistK; ++k) e[hh][k] = src[k];
      } else {
#pragma unroll
        for (int k = 0; k < kHistK; ++k) e[hh][k] = make_float2(0.0f, __int_as_float(-1));
      }
    }
  }
  int bad = 0;
  for (int k = lane; k < nseg; k += 32) bad |= p.slot_bad[slot0 + k];
  if (__any_sync(0xffffffffu, bad)) {
    if (lane == 0) finish(zs, none, true);
    return;
  }
#pragma unroll
  for (int hh = 0; hh < kHeads; ++hh) {
    const int li = lane + 32 * hh;
    float2(&mine)[kHistK] = lists[warp][li];
    if (nseg <= kLists) {
#pragma unroll
      for (int k = 0; k < kHistK; ++k) mine[k] = e[hh][k];
    } else {
      // lists li, li + kLists, ... cover ascending page ranges: inserted in
      // that order, an equal score always comes with a higher id
      TopK15 t;
      t.reset();
      for (int k = li; k < nseg; k += kLists) {
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
  }
  __syncwarp();
  int res[kHistK];
  float rs[kHistK];
  int h0 = 0, h1 = 0;                         // heads of lists lane and lane + 32
#pragma unroll
  for (int k = 0; k < kHistK; ++k) {
    const float2 e0 = h0 < kHistK ? lists[warp][lane][h0] : make_float2(0.0f, __int_as_float(-1));
    const int id0 = __float_as_int(e0.y);
    const uint32_t k0 = id0 >= 0 ? order_key(e0.x) : 0u;
    uint32_t key = k0;
    int id = id0;
    bool take1 = false;
    if constexpr (kHeads == 2) {
      const float2 e1 = h1 < kHistK ? lists[warp][lane + 32][h1] : make_float2(0.0f, __int_as_float(-1));
      const int id1 = __float_as_int(e1.y);
      const uint32_t k1 = id1 >= 0 ? order_key(e1.x) : 0u;
      take1 = k1 > k0 || (k1 == k0 && k1 != 0u && id1 < id0);
      key = take1 ? k1 : k0;
      id = take1 ? id1 : id0;
    }
    const uint32_t kmax = warp_max_u32(key);
    const uint32_t idmin = warp_min_u32(key == kmax && kmax != 0u ? (uint32_t)id : 0xFFFFFFFFu);
    if (kmax != 0u && key == kmax && (uint32_t)id == idmin) {
      if (take1) ++h1; else ++h0;
    }
    res[k] = kmax != 0u ? (int)idmin : -1;
    rs[k] = kmax != 0u ? key_to_float(kmax) : 0.0f;
  }
  if (lane == 0) finish(rs, res, false);
}

// One warp per (row, head): merge the `world` context-parallel ranks'
// candidate lists of the row (each sorted by score desc, id asc; the ranks'
// page ranges are disjoint) into its final row.  Lane k holds rank k's list
// (ranks k, k+32, ... folded in when world > 32).
__global__ void __launch_bounds__(256) cp_merge_kernel(const float2* __restrict__ cand_all, int world,
                                                       int num_reqs, int query_len, int H,
                                                       const int32_t* __restrict__ seq_lens,
                                                       int32_t* __restrict__ out, int32_t* status) {
  __shared__ float2 lists[8][32][kHistK];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t rows = (int64_t)num_reqs * query_len * H;
  const int64_t gw = (int64_t)blockIdx.x * 8 + warp;
  if (gw >= rows) return;
  const int t = (int)(gw / H);                          // query row
  const int r = t / query_len, i = t % query_len;
  const int pos = __ldg(seq_lens + r) - query_len + i;
  const int L = pos >= 0 ? (pos >> 7) : -1;
  int bad = 0;
  TopK15 tk;
  tk.reset();
  for (int k = lane; k < world; k += 32) {
    const float2* src = cand_all + ((int64_t)k * rows + gw) * kHistK;
    bad |= __float_as_int(src[0].y) == -2;
#pragma unroll
    for (int e = 0; e < kHistK; ++e) {
      const float2 v = src[e];
      if (__float_as_int(v.y) >= 0) tk.insert_any(v.x, __float_as_int(v.y));
    }
  }
  float2(&mine)[kHistK] = lists[warp][lane];
#pragma unroll
  for (int k = 0; k < kHistK; ++k) mine[k] = make_float2(tk.s[k], __int_as_float(tk.id[k]));
  __syncwarp();
  bad = __any_sync(0xffffffffu, bad);
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
  if (lane == 0) {
    write_out_row(out + gw * kTopK, res, L, bad != 0);
    if (bad && status) atomicOr(status, kStatusBadPage);
  }
}

cudaError_t launch_cp_merge(const float2* cand_all, int world, int num_reqs, int query_len, int H,
                            const int32_t* seq_lens, int32_t* out, int32_t* status, cudaStream_t stream) {
  const int64_t warps = (int64_t)num_reqs * query_len * H;
  if (warps <= 0) return cudaSuccess;
  cp_merge_kernel<<<(unsigned)((warps + 7) / 8), 256, 0, stream>>>(cand_all, world, num_reqs, query_len, H,
                                                                   seq_lens, out, status);
  return cudaGetLastError();
}

// ============================================================ small-R decode
// Requests of at most 8 rows (query_len x heads <= 8: decode_batch's 4, a
// single query of 1..8 heads) on NVFP4 pages.  The quad kernel above pays a
// chain of tensor-memory hand-offs per slice whatever the row count; here
// the contraction is small enough for the warp-level mma.sync tensor path
// (m16n8k16, f16 operands, f32 accumulation: the same exact products and
// fp32 sums), so every warp streams its own pages with no hand-off at all.
//   * the split unit is a warp: the T history pages are cut into G = min(16 x
//     grid, T) contiguous ranges, warp u of the grid takes range u, walks it
//     as segments (one per request) and keeps each row's top-15 in lane n
//     (n < R); a request inside one range is finalised by its warp, the
//     others leave 15 candidates per row in slot u + r for the merge kernel
//     (the same slots, request info and merge as the quad kernel, with warps
//     in place of CTAs), so no barrier joins the warps of a CTA;
//   * half pages (64 tokens) go through a 2-stage ring per warp (bulk
//     copies; lane 0 issues the copy of the half after next as soon as a
//     stage is read), 16 warps per CTA;
//   * per page 8 token tiles x 8 K steps of mma.sync, M = 16 tokens, N = 8
//     query rows (row n in lane group n, rows >= R zero), K = 16 dimensions
//     = one NVFP4 group: lane (g, c) dequantises its A fragment straight
//     from the raw page, the two code bytes 8kk + 2c, 8kk + 2c + 1 of tokens
//     g and g + 8 times the group's E4M3 scale (exact in f16).  The K order
//     inside a group is permuted alike for A and the query fragment B
//     (fragment columns 2c, 2c+1, 2c+8, 2c+9 <- dimensions 4c .. 4c+3), which
//     leaves every dot product unchanged;
//   * the row maxima over the 128 tokens: per lane over its two tokens of
//     each tile, then over the 8 lane groups by shuffles.
// Every wait is bounded; a wait that runs out gives the quad kernel's
// failure rows (-1 rows or a bad slot) and the copies in flight are drained.
constexpr int kSmWarps = 16, kSmStages = 2, kSmRows = 8;
constexpr uint32_t kSmHalf = 64 * 72;                 // a stage holds 64 tokens (half a page)
constexpr uint32_t kSmPageOff = 0;
constexpr uint32_t kSmPreOff = kSmWarps * kSmStages * kSmHalf;
static_assert(kSmPreOff + (kMaxDecodeReqs + 1) * 4 + 128 <= 227 * 1024, "small decode shared memory");

// Bytes 0 and 1 of w (two E2M1 codes each, low nibble first) -> two f16x2.
__device__ __forceinline__ void e2m1x4_lo2_to_f16x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

__device__ __forceinline__ void mma_m16n8k16_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                                 uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_m16n8k16_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                                  uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Split units of the decode launch: CTAs of the quad kernel, or warps of the
// small-row kernel (the candidate slots are indexed by unit + request).
int decode_split_units(int R, int page_format, int grid) {
  (void)page_format;                                 // both page formats
  return R <= kSmRows ? grid * kSmWarps : grid;
}

template <class PF>
__global__ void __launch_bounds__(kSmWarps * 32, 1) decode_small_kernel(const DecodeParams p) {
  // a stage: NVFP4, 64 token rows of 72 bytes; MXFP4, 64 rows of 64 code
  // bytes, then their 64 x 4 E8M0 scale bytes
  constexpr uint32_t kRow = PF::kBf16 ? 64u : 72u;
  constexpr uint32_t kStageBytes = PF::kBf16 ? 64u * 64u + 64u * 4u : kSmHalf;
  extern __shared__ __align__(128) uint8_t sm_raw[];
  __shared__ __align__(8) uint64_t pg_full[kSmWarps][kSmStages];
  __shared__ volatile int abort_s;
  __shared__ int warp_sum[kSmWarps];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int lg = lane >> 2, lc = lane & 3;            // mma fragment lane group / index in group
  const uint64_t lim = p.wait_ns;
  griddep_launch_dependents();                       // the merge kernel may be scheduled
  uint8_t* const base = sm_raw + ((128u - (smem_u32(sm_raw) & 127u)) & 127u);
  int32_t* const pre = reinterpret_cast<int32_t*>(base + kSmPreOff);
  const int NR = p.num_reqs, R = p.R;
  constexpr int kThreads = kSmWarps * 32;

  // ---- history pages per request -> exclusive prefix sums in smem
  {
    const int per = (NR + kThreads - 1) / kThreads;
    const int r0 = tid * per, r1 = min(NR, r0 + per);
    int sum = 0;
    for (int r = r0; r < r1; ++r) sum += req_pages(p, r);
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
      run += req_pages(p, r);
    }
    if (tid == kThreads - 1) {
      int tot = 0;
      for (int w = 0; w < kSmWarps; ++w) tot += warp_sum[w];
      pre[NR] = tot;
    }
    if (tid == 0) {
      for (int w = 0; w < kSmWarps; ++w)
        for (int st = 0; st < kSmStages; ++st) mbar_init(smem_u32(&pg_full[w][st]), 1);
      abort_s = 0;
      fence_mbar_init();
    }
    __syncthreads();
  }
  const int64_t T = pre[NR];
  const int G = (int)min((int64_t)gridDim.x * kSmWarps, T);
  if (blockIdx.x == 0) {
    for (int r = tid; r < NR; r += kThreads) {
      const int h = pre[r + 1] - pre[r];
      int2 info = make_int2(0, 0);
      if (h > 0) {
        const int cf = cta_of(pre[r], T, G), cl = cta_of(pre[r + 1] - 1, T, G);
        info = make_int2(cf, cl - cf + 1);
      }
      p.req_info[r] = info;
    }
  }
  const int u = blockIdx.x * kSmWarps + warp;        // this warp's split unit
  if (u >= G) return;
  const int64_t x0 = (int64_t)u * T / G, x1 = (int64_t)(u + 1) * T / G;

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
  SegWalk walk{pre, NR, x1 - x0, 0, r_start, req_lo(p, r_start) + (int)(x0 - pre[r_start])};
  uint8_t* const ring = base + kSmPageOff + (uint32_t)warp * kSmStages * kSmHalf;
  int64_t kw = 0;                                    // pages of this warp so far (ring position)
  int64_t last_k[kSmStages] = {-1, -1};              // the last page issued into each stage
  bool ok = true;                                    // uniform within the warp

  while (walk.more()) {
    const int je = walk.seg_end(p);
    const int r = walk.r, js = walk.j;
    const int seq_r = __ldg(p.seq_lens + r);
    const int32_t* const pt_row = p.page_table + (int64_t)r * p.pt_stride;
    const int npw = je - js;                          // this segment's pages, all this warp's
    const int nh = 2 * npw;                           // and their halves: half h of page i is item 2i + h
    const int64_t k0 = kw;
    // the copy of item x (page js + x / 2, tokens 64 (x % 2) ..) into stage
    // (k0 + x) % 2; false: unreadable page
    auto issue = [&](int x) {
      const int64_t k = k0 + x;
      const int st = (int)(k & 1);
      int phys = 0;
      if (lane == 0) phys = __ldg(pt_row + js + (x >> 1));
      phys = __shfl_sync(0xffffffffu, phys, 0);
      const bool good = phys >= 0 && phys < p.num_blocks;
      if (lane == 0) {
        const uint32_t fb = smem_u32(&pg_full[warp][st]);
        if (good) {
          mbar_arrive_expect_tx(fb, kStageBytes);
          const uint8_t* const page = p.kv + (int64_t)phys * PF::kPageBytes;
          if constexpr (PF::kBf16) {
            bulk_g2s(smem_u32(ring + st * kSmHalf), page + (x & 1) * 4096, 4096u, fb);
            bulk_g2s(smem_u32(ring + st * kSmHalf + 4096), page + 8192 + (x & 1) * 256, 256u, fb);
          } else {
            bulk_g2s(smem_u32(ring + st * kSmHalf), page + (x & 1) * kSmHalf, kSmHalf, fb);
          }
        } else {
          if (!(x & 1)) atomicOr(p.status, kStatusBadPage);
          mbar_arrive(fb);                           // nothing to copy: the stage's phase completes empty
        }
      }
      last_k[st] = k;
      return good;
    };
    bool good0 = true, good1 = true;                 // the item in stage 0 / 1 was readable
    for (int x = 0; ok && x < nh && x < kSmStages; ++x) {
      const bool gd = issue(x);
      if ((k0 + x) & 1) good1 = gd; else good0 = gd;
    }
    // the request's queries as mma B fragments: row n = lg, dimensions
    // 16kk + 4lc .. 16kk + 4lc + 3 (rows >= R zero)
    uint32_t bq[8][2];
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      uint32_t w4 = 0;
      if (lg < R) w4 = __ldg(reinterpret_cast<const uint32_t*>(p.q + ((int64_t)r * R + lg) * 128 + 16 * kk + 4 * lc));
      bq[kk][0] = PF::widen_q(w4 & 0xFFFFu);
      bq[kk][1] = PF::widen_q(w4 >> 16);
    }
    const int pos = seq_r - p.qlen + lane / p.H;       // row `lane` (lanes < R)
    const int L = pos >= 0 ? (pos >> 7) : -1;
    TopK15 top;
    top.reset();
    int seg_bad = 0;
    float rm0 = -CUDART_INF_F, rm1 = -CUDART_INF_F;  // rows 2lc, 2lc + 1, over the page's items so far
    for (int x = 0; x < nh; ++x) {
      const int64_t k = k0 + x;
      const int st = (int)(k & 1);
      const int j = js + (x >> 1);
      if (ok) {
        ok = __all_sync(0xffffffffu, mbar_wait_or_abort(smem_u32(&pg_full[warp][st]), (uint32_t)((k >> 1) & 1),
                                                        &abort_s, lim));
        if (!ok && lane == 0 && !abort_s) {
          abort_s = 1;
          atomicOr(p.status, kStatusTimeout);
        }
      }
      const bool good = st ? good1 : good0;
      seg_bad |= good ? 0 : 1;
      if (ok && good) {
        const uint8_t* const pg = ring + st * kSmHalf;
#pragma unroll 1
        for (int mt = 0; mt < 4; ++mt) {
          const uint8_t* const t0 = pg + (16 * mt + lg) * kRow;
          const uint8_t* const t1 = t0 + 8 * kRow;
          float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
          if constexpr (PF::kBf16) {
            // the two tokens' 4 E8M0 scales, one per 32 dimensions = K steps
            // 2j, 2j + 1, as bf16x2 broadcasts
            const uint32_t sa = *reinterpret_cast<const uint32_t*>(pg + 4096 + (16 * mt + lg) * 4);
            const uint32_t sb = *reinterpret_cast<const uint32_t*>(pg + 4096 + (16 * mt + lg + 8) * 4);
            uint32_t s2a[4], s2b[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint32_t ba = (sa >> (8 * j)) & 0xFFu, bb = (sb >> (8 * j)) & 0xFFu;
              s2a[j] = e8m0x2_to_bf16x2(ba | (ba << 8));
              s2b[j] = e8m0x2_to_bf16x2(bb | (bb << 8));
            }
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint32_t wa = *reinterpret_cast<const uint16_t*>(t0 + 8 * kk + 2 * lc);
              const uint32_t wb = *reinterpret_cast<const uint16_t*>(t1 + 8 * kk + 2 * lc);
              uint32_t ca0, ca2, cb0, cb2;
              e2m1x4_lo2_to_f16x2(wa, ca0, ca2);
              e2m1x4_lo2_to_f16x2(wb, cb0, cb2);
              const uint32_t sA = s2a[kk >> 1], sB = s2b[kk >> 1];
              mma_m16n8k16_bf16(d, bmul2_u32(f16x2_to_bf16x2(ca0), sA), bmul2_u32(f16x2_to_bf16x2(cb0), sB),
                                bmul2_u32(f16x2_to_bf16x2(ca2), sA), bmul2_u32(f16x2_to_bf16x2(cb2), sB),
                                bq[kk][0], bq[kk][1]);
            }
          } else {
            // the two tokens' 8 scales, f16x2 pairs {group 2i, group 2i + 1}
            const uint2 sa = *reinterpret_cast<const uint2*>(t0 + 64);
            const uint2 sb = *reinterpret_cast<const uint2*>(t1 + 64);
            const uint32_t sca[4] = {e4m3x2_to_f16x2(sa.x & 0xFFFFu), e4m3x2_to_f16x2(sa.x >> 16),
                                     e4m3x2_to_f16x2(sa.y & 0xFFFFu), e4m3x2_to_f16x2(sa.y >> 16)};
            const uint32_t scb[4] = {e4m3x2_to_f16x2(sb.x & 0xFFFFu), e4m3x2_to_f16x2(sb.x >> 16),
                                     e4m3x2_to_f16x2(sb.y & 0xFFFFu), e4m3x2_to_f16x2(sb.y >> 16)};
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              // the code bytes 8kk + 2lc, 8kk + 2lc + 1 of the two tokens
              const uint32_t wa = *reinterpret_cast<const uint16_t*>(t0 + 8 * kk + 2 * lc);
              const uint32_t wb = *reinterpret_cast<const uint16_t*>(t1 + 8 * kk + 2 * lc);
              const uint32_t s2a = (kk & 1) ? f16x2_bcast_hi(sca[kk >> 1]) : f16x2_bcast_lo(sca[kk >> 1]);
              const uint32_t s2b = (kk & 1) ? f16x2_bcast_hi(scb[kk >> 1]) : f16x2_bcast_lo(scb[kk >> 1]);
              uint32_t ca0, ca2, cb0, cb2;
              e2m1x4_lo2_to_f16x2(wa, ca0, ca2);
              e2m1x4_lo2_to_f16x2(wb, cb0, cb2);
              mma_m16n8k16_f16(d, hmul2_u32(ca0, s2a), hmul2_u32(cb0, s2b), hmul2_u32(ca2, s2a),
                               hmul2_u32(cb2, s2b), bq[kk][0], bq[kk][1]);
            }
          }
          rm0 = fmaxf(rm0, fmaxf(d[0], d[2]));
          rm1 = fmaxf(rm1, fmaxf(d[1], d[3]));
        }
      }
      // the stage is read: the item after next goes into it
      if (ok && x + kSmStages < nh) {
        __syncwarp();
        fence_proxy_async_smem();
        const bool gd = issue(x + kSmStages);
        if (st) good1 = gd; else good0 = gd;
      }
      if (x & 1) {                                    // the page's second half: its score
        if (ok && good) {
          // over the 8 lane groups (tokens lg, lg + 8 of every tile)
#pragma unroll
          for (int o = 4; o < 32; o <<= 1) {
            rm0 = fmaxf(rm0, __shfl_xor_sync(0xffffffffu, rm0, o));
            rm1 = fmaxf(rm1, __shfl_xor_sync(0xffffffffu, rm1, o));
          }
          // row `lane`'s score sits in lane lane / 2 (rm0 for even rows, rm1 for odd)
          const float v0 = __shfl_sync(0xffffffffu, rm0, (lane >> 1) & 3);
          const float v1 = __shfl_sync(0xffffffffu, rm1, (lane >> 1) & 3);
          const float m = canon_zero((lane & 1) ? v1 : v0);
          if (lane < R && j < L) {
            top.insert(m, j);
            if (p.scores_dbg) p.scores_dbg[((int64_t)r * R + lane) * p.dbg_stride + j] = m;
          }
        }
        rm0 = -CUDART_INF_F;
        rm1 = -CUDART_INF_F;
      }
    }
    kw = k0 + nh;

    // ---- the segment's rows: final (a request inside this range) or candidates
    const int cf = cta_of(pre[r], T, G), cl = cta_of(pre[r + 1] - 1, T, G);
    const bool bad = __any_sync(0xffffffffu, seg_bad != 0);
    if (ok && !abort_s) {
      if (lane < R) {
        const int pe = seq_r - p.qlen + lane / p.H;
        if (cf == cl) {
          if (p.cand_out) write_cand_row(p.cand_out + ((int64_t)r * R + lane) * kHistK, top.s, top.id, bad);
          else write_out_row(p.out + ((int64_t)r * R + lane) * kTopK, top.id, pe >= 0 ? (pe >> 7) : -1, bad);
        } else {
          float2* dst = p.cand + ((int64_t)(u + r) * R + lane) * kHistK;
#pragma unroll
          for (int kq = 0; kq < kHistK; ++kq) dst[kq] = make_float2(top.s[kq], __int_as_float(top.id[kq]));
        }
      }
      if (lane == 0 && cf != cl) p.slot_bad[u + r] = bad ? 1 : 0;
    } else {
      // a wait ran out: -1 rows for a request this warp finalises, else a bad slot
      if (cf == cl && lane < R) {
        const float zs[kHistK] = {};
        const int none[kHistK] = {-1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1, -1};
        if (p.cand_out) write_cand_row(p.cand_out + ((int64_t)r * R + lane) * kHistK, zs, none, true);
        else write_out_row(p.out + ((int64_t)r * R + lane) * kTopK, none, -1, true);
      }
      if (lane == 0 && cf != cl) p.slot_bad[u + r] = 1;
    }
    walk.g += je - walk.j;
    walk.j = je;
    if (walk.more()) walk.next_request(p);
  }
  // copies still in flight (after a wait ran out) land before the warp leaves
#pragma unroll
  for (int st = 0; st < kSmStages; ++st)
    if (last_k[st] >= 0) mbar_wait(smem_u32(&pg_full[warp][st]), (uint32_t)((last_k[st] >> 1) & 1));
}

template <int NQ, class PF>
static cudaError_t launch_decode_nq(const DecodeParams& p, int grid, cudaStream_t stream) {
  const size_t smem = DecLayout<NQ, PF>::bytes(p.num_reqs);
  cudaError_t e = cudaFuncSetAttribute(decode_score_kernel<NQ, PF>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  decode_score_kernel<NQ, PF><<<grid, DecRoles<NQ>::kThreads, smem, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t warps = (int64_t)p.num_reqs * p.R;
  return launch_dependent(decode_merge_kernel<8, 1>, (unsigned)((warps + 7) / 8), 256u, 0, stream, p);
}

template <class PF>
static cudaError_t launch_decode_small(const DecodeParams& p, int grid, cudaStream_t stream) {
  const size_t smem = 128 + kSmPreOff + (size_t)(p.num_reqs + 1) * 4;   // grid CTAs = 8 x grid split units
  cudaError_t e =
      cudaFuncSetAttribute(decode_small_kernel<PF>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  decode_small_kernel<PF><<<grid, kSmWarps * 32, smem, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t warps = (int64_t)p.num_reqs * p.R;
  return launch_dependent(decode_merge_kernel<4, 2>, (unsigned)((warps + 3) / 4), 128u, 0, stream, p);
}

template <class PF>
static cudaError_t launch_decode_pf(const DecodeParams& p, int grid, cudaStream_t stream) {
  if (p.R <= kSmRows) return launch_decode_small<PF>(p, grid, stream);
  switch (decode_nq(p.R)) {
    case 16: return launch_decode_nq<16, PF>(p, grid, stream);
    case 32: return launch_decode_nq<32, PF>(p, grid, stream);
    default: return launch_decode_nq<64, PF>(p, grid, stream);
  }
}

cudaError_t launch_decode(const DecodeParams& p, int grid, cudaStream_t stream) {
  return p.page_format == kPagesMxfp4 ? launch_decode_pf<Mxfp4Pages>(p, grid, stream)
                                      : launch_decode_pf<Nvfp4Pages>(p, grid, stream);
}

}  // namespace nvfp4idx
