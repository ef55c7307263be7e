// prefill.cu -- prefill indexer: a dense Q.K^T per page on the tensor cores,
// row max per page, fused top-15 with the causal clamp.
//
// Follows MiniMaxM3IndexerNvfp4Impl._prefill of
// vllm.models.minimax_m3.nvidia.indexer_nvfp4 in what it computes, with the
// per-token causal clamp of vllm.models.minimax_m3.nvidia.indexer_flashinfer
// (valid pages = pos/128 + 1).  Instead of the pages' FP8 gather workspace
// (a lossy extra HBM pass), each NVFP4 page is dequantised exactly to fp16
// straight into shared memory.
//
// Tiling.  A tile is 128 query rows = (128/H tokens) x H heads of one
// request (the last tile of a request may be ragged).  A work unit is a PAIR
// of consecutive tiles of one request (tiles ntile-1-2k and ntile-2-2k) or,
// for the tile left over in a request with an odd number of tiles, a single
// tile; a unit walks the pages of its later tile, which has the most: every
// page is dequantised once and multiplied against both tiles, so the
// CUDA-core work per unit of tensor work is halved.  Units are ordered pairs
// first (requests in order, last tiles first), then singles.
//
// Balance.  The pages of all units, weighted by their measured cost (a page
// of a pair 17, of a single 10, plus 96 per unit for the switch to its
// queries), are split evenly over the CTAs (one per SM): a CTA walks a
// contiguous range of (unit, page), so no CTA waits for a long request's
// last tiles while others idle.  A unit cut by a CTA boundary leaves, per
// CTA, its rows' top-15 candidates in plan scratch (two slots per CTA: its
// first and its last unit), and prefill_merge_kernel merges them in page
// order.
// Warp roles, one per warpgroup (setmaxnreg moves registers between them),
// linked by mbarrier rings:
//   * warpgroup 0 (56 registers): warp 0 has the TMA unit copy each raw
//     9216-byte page into a 6-stage shared ring; warps 1 / 2 issue the 8
//     tcgen05.mma of every page for tile A / tile B (both operands in shared
//     memory: the tile's queries, M = 128, and the page, N = 128; K = 16),
//     D[row][token] in fp32 in tensor memory, two accumulators per tile;
//     warp 3 idles;
//   * warpgroups 1 / 2 (88 registers, pages of even / odd index): thread t
//     dequantises token t to fp16 into the group's own 128B-swizzled K-major
//     B tile [128 tokens x 128];
//   * warpgroups 3 / 4 (120 registers, tile A / tile B), thread = query row:
//     at a unit start widen the tile's E4M3 queries into a 128B-swizzled
//     fp16 A tile in shared memory; per page take the row's max over the 128
//     tokens with four load-and-reduce tensor-memory reads (tcgen05.ld.red,
//     32 columns each: no CUDA-core instruction per score) and update the
//     row's top-15 if the page is a history page of its token; write the row
//     (or its candidates) at the end of the unit.
#include <cstdint>
#include <cuda_runtime.h>

#include "codec.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "topk.cuh"

namespace nvfp4idx {

constexpr int kPreStages = 6;              // raw page ring (even: pages of one parity per stage)
constexpr int kPreThreads = 640;           // 5 warpgroups
// 4 x 56 + 8 x 88 + 8 x 120 = 1888 registers per lane slot <= 640 x 96 / 32
constexpr uint32_t kRegsCtl = 56, kRegsDq = 88, kRegsEpi = 120;
constexpr uint32_t kPreTmemCols = 512;     // tile A: D [0,128), [128,256); tile B: [256,384), [384,512)
constexpr uint32_t kTileBytes = 128 * 256; // fp16 [2 K-blocks][128 rows][64], 128B swizzle

template <class PF>   // page format (codec.cuh)
struct PreLayout {
  static constexpr uint32_t kQOff = 0;                           // A tiles of tile A and tile B
  static constexpr uint32_t kBOff = 2 * kTileBytes;              // B tiles of dequant groups 0 and 1
  static constexpr uint32_t kStageOff = kBOff + 2 * kTileBytes;
  static constexpr uint32_t kTpreOff = kStageOff + kPreStages * PF::kPageBytes;
  // two prefix arrays per request: tiles and possible pairs
  static size_t bytes(int num_reqs) { return 1024 + kTpreOff + (size_t)(num_reqs + 1) * 8; }
};
static_assert(1024 + PreLayout<Nvfp4Pages>::kTpreOff + (kMaxPrefillReqs + 1) * 8 + 1024 <= 227 * 1024 &&
                  1024 + PreLayout<Mxfp4Pages>::kTpreOff + (kMaxPrefillReqs + 1) * 8 + 1024 <= 227 * 1024,
              "prefill shared memory above the 227 KB a CTA may hold");

// Byte offset of K step kk (16 elements) inside a 128B-swizzled K-major tile
// of 128 rows: two K-blocks of 64 elements, 32 bytes per step within one.
__host__ __device__ constexpr uint32_t kstep_bytes(int kk) {
  return (uint32_t)(kk >> 2) * (128u * 128u) + (uint32_t)(kk & 3) * 32u;
}

struct TileRows {
  int t0, nt, row0;   // first token of the tile within the request, tokens, first q row
};

struct PairInfo {
  int r, ctx, L_max;  // request, context length, pages walked (those of tile A)
  bool table_bad;
  TileRows tile[2];   // tile A (the later one) and tile B (nt = 0 when absent)
};

// The work schedule, identical in every thread: tpre[r] / fpre[r] = tiles /
// possible pairs of the requests before r; P pairs are formed (requests in
// order, each request's last tiles first), the remaining tiles are singles.
struct Sched {
  const int32_t* tpre;
  const int32_t* fpre;
  int NR, P;
  __device__ __forceinline__ int pairs_before(int r) const { return min(fpre[r], P); }
  __device__ __forceinline__ int singles_before(int r) const { return tpre[r] - 2 * pairs_before(r); }
};

template <int H>
__device__ __forceinline__ PairInfo prefill_pair(const PrefillParams& p, const Sched& sc, int u) {
  constexpr int TQ = 128 / H;
  const bool is_pair = u < sc.P;
  const int key = is_pair ? u : u - sc.P;
  int lo = 0, hi = sc.NR - 1;                        // last request whose prefix <= key
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((is_pair ? sc.fpre[mid] : sc.singles_before(mid)) <= key) lo = mid; else hi = mid - 1;
  }
  PairInfo pi;
  pi.r = lo;
  const int cu0 = __ldg(p.cu_seqlens_q + lo);
  const int ql = __ldg(p.cu_seqlens_q + lo + 1) - cu0;
  const int ntile = (ql + TQ - 1) / TQ;
  int la;                                            // tile A; tile B = la - 1 for a pair
  if (is_pair) {
    la = ntile - 1 - 2 * (key - sc.fpre[lo]);
  } else {
    const int pairs_r = sc.pairs_before(lo + 1) - sc.pairs_before(lo);
    la = ntile - 1 - 2 * pairs_r - (key - sc.singles_before(lo));
  }
#pragma unroll
  for (int x = 0; x < 2; ++x) {
    const int lt = (x == 0 || is_pair) ? la - x : -1;
    TileRows& tr = pi.tile[x];
    tr.t0 = lt >= 0 ? lt * TQ : 0;
    tr.nt = lt >= 0 ? min(TQ, ql - tr.t0) : 0;
    tr.row0 = cu0 + tr.t0;
  }
  const int seq = __ldg(p.seq_lens + lo);
  pi.ctx = seq - ql;
  const int hist = seq >= 1 ? (seq - 1) >> 7 : 0;
  pi.table_bad = hist > p.pt_stride;
  const int pos_last = pi.ctx + pi.tile[0].t0 + pi.tile[0].nt - 1;
  pi.L_max = (pos_last >= 0 && !pi.table_bad) ? (pos_last >> 7) : 0;
  return pi;
}

// weighted cost of one page of unit u (pair 17, single 10); a unit with pages
// also costs kUnitOverhead before its first page (the switch to its queries
// drains the MMA pipeline; measured: about five and a half pages of a pair)
__device__ __forceinline__ int unit_weight(const Sched& sc, int u) { return u < sc.P ? 17 : 10; }
constexpr int kUnitOverhead = 96;
__device__ __forceinline__ long long unit_cost(int w, int L) {
  return L > 0 ? kUnitOverhead + (long long)w * L : 0;
}

// Pages [ja, jb) of a unit of L pages whose weighted range starts at U that
// fall in the CTA range [A, B) (last: B is the end of all work): page j sits
// at U + w j.
__device__ __forceinline__ void seg_pages(long long U, int w, int L, long long A, long long B, bool last,
                                          int& ja, int& jb) {
  ja = 0;
  jb = L;
  if (U < A) ja = (int)min((long long)L, (A - U + w - 1) / w);
  if (!last && U + (long long)w * L > B) jb = (int)min((long long)L, max(0ll, (B - U + w - 1) / w));
  jb = max(jb, ja);   // none here: ja == jb (also for a unit of no pages)
}

// CTA owning weighted position x when [0, W) is split over G CTAs at
// floor(c W / G).
__device__ __forceinline__ int split_cta(long long x, long long W, int G) {
  return (int)(((x + 1) * G - 1) / W);
}

// This CTA's share of the work (in shared memory: every role reads it).
struct PreRange {
  long long A, B, W;   // weighted range [A, B) of [0, W)
  long long Uua;       // weighted start of unit ua
  int ua, ub;          // units walked
  int last;            // the last CTA (takes everything up to W)
};

// The CTA's walk over units ua..ub, identical in every role: for each unit its
// description and the pages [ja, jb) of it that fall in this CTA's range.
struct PreWalk {
  const PreRange* rg;
  int u;
  long long U;         // weighted start of unit u
  __device__ __forceinline__ explicit PreWalk(const PreRange* r) : rg(r), u(r->ua), U(r->Uua) {}
  __device__ __forceinline__ bool more() const { return u <= rg->ub; }
  template <int H>
  __device__ __forceinline__ void get(const PrefillParams& p, const Sched& sc, PairInfo& pi, int& w, int& ja,
                                      int& jb) const {
    pi = prefill_pair<H>(p, sc, u);
    w = unit_weight(sc, u);
    seg_pages(U + kUnitOverhead, w, pi.L_max, rg->A, rg->B, rg->last != 0, ja, jb);
  }
  __device__ __forceinline__ void next(int w, int L) {
    U += unit_cost(w, L);
    ++u;
  }
};

template <int H, class PF>
__global__ void __launch_bounds__(kPreThreads, 1) prefill_kernel(const PrefillParams p) {
  using PreLayout = nvfp4idx::PreLayout<PF>;
  constexpr int TQ = 128 / H;     // tokens per tile
  // Waits that sleep inside mbarrier.try_wait (up to 1 ms) leave their
  // schedulers' issue slots to the dequant and epilogue warps: NVFP4 pages
  // gain; MXFP4 pages, whose dequantisation costs 2.5 times the
  // instructions, measured slower with them.
  constexpr bool kSleep = !PF::kBf16;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t raw_full[kPreStages], raw_empty[kPreStages];
  // B tile h is free again once both tiles' MMAs of its last page are done,
  // which d_full[0][h] and d_full[1][h] tell: no separate release barrier
  __shared__ __align__(8) uint64_t b_full[2];                      // B tile of dequant group h
  __shared__ __align__(8) uint64_t d_full[2][2], d_empty[2][2];    // [tile][accumulator]
  __shared__ __align__(8) uint64_t q_full[2], q_empty;             // A tiles (queries)
  __shared__ uint32_t tmem_base_s;
  __shared__ volatile int abort_s;
  __shared__ int warp_sum[kPreThreads / 32], warp_sum2[kPreThreads / 32];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint64_t lim = p.wait_ns;                    // limit of every bounded wait
  griddep_launch_dependents();                       // the merge kernel may be scheduled
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t sbase = (raw_u32 + 1023u) & ~1023u;
  uint8_t* const base = smem_raw + (sbase - raw_u32);
  int32_t* const tpre = reinterpret_cast<int32_t*>(base + PreLayout::kTpreOff);
  const int NR = p.num_reqs, G = gridDim.x, c = blockIdx.x;
  constexpr int NW = kPreThreads / 32;

  // ---- tiles and possible pairs per request -> exclusive prefix sums
  int32_t* const fpre = tpre + (NR + 1);
  {
    const int per = (NR + kPreThreads - 1) / kPreThreads;
    const int r0 = tid * per, r1 = min(NR, r0 + per);
    auto tiles = [&](int r) {
      const int ql = __ldg(p.cu_seqlens_q + r + 1) - __ldg(p.cu_seqlens_q + r);
      return ql > 0 ? (ql + TQ - 1) / TQ : 0;
    };
    int st = 0, sp = 0;
    for (int r = r0; r < r1; ++r) {
      const int nt = tiles(r);
      st += nt;
      sp += nt >> 1;
    }
    int it = st, ipp = sp;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int a1 = __shfl_up_sync(0xffffffffu, it, o), a2 = __shfl_up_sync(0xffffffffu, ipp, o);
      if (lane >= o) {
        it += a1;
        ipp += a2;
      }
    }
    if (lane == 31) warp_sum[warp] = it, warp_sum2[warp] = ipp;
    __syncthreads();
    int ot = 0, op = 0;
    for (int w = 0; w < warp; ++w) ot += warp_sum[w], op += warp_sum2[w];
    int rt = ot + it - st, rp = op + ipp - sp;
    for (int r = r0; r < r1; ++r) {
      tpre[r] = rt;
      fpre[r] = rp;
      const int nt = tiles(r);
      rt += nt;
      rp += nt >> 1;
    }
    if (tid == kPreThreads - 1) {
      int tt = 0, tp = 0;
      for (int w = 0; w < NW; ++w) tt += warp_sum[w], tp += warp_sum2[w];
      tpre[NR] = tt;
      fpre[NR] = tp;
    }
    __syncthreads();
  }
  // every possible pair is formed (the split below balances the CTAs)
  Sched sched{tpre, fpre, NR, fpre[NR]};
  const int NU = tpre[NR] - sched.P;                 // P pairs + the singles

  // ---- this CTA's share of the weighted pages: [A, B) of [0, W), walked as
  // the units ua..ub (64-bit block scan over per-thread chunks of units)
  __shared__ PreRange rg;
  {
    __shared__ long long cs_warp[kPreThreads / 32];
    __shared__ int ua_s, ub_s;
    __shared__ long long uua_s;
    const int k = (NU + kPreThreads - 1) / kPreThreads;
    const int u0 = min(NU, tid * k), u1 = min(NU, u0 + k);
    long long sum = 0;
    for (int u = u0; u < u1; ++u)
      sum += unit_cost(unit_weight(sched, u), prefill_pair<H>(p, sched, u).L_max);
    long long incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane == 31) cs_warp[warp] = incl;
    if (tid == 0) {
      ua_s = NU;
      ub_s = -1;
      uua_s = 0;
    }
    __syncthreads();
    long long off = 0, W = 0;
    for (int w = 0; w < NW; ++w) {
      if (w < warp) off += cs_warp[w];
      W += cs_warp[w];
    }
    const long long A = (long long)c * W / G;
    const long long B = (c == G - 1) ? W : (long long)(c + 1) * W / G;
    long long U = off + incl - sum;
    int my_a = NU, my_b = -1;
    for (int u = u0; u < u1; ++u) {
      const long long cu = unit_cost(unit_weight(sched, u), prefill_pair<H>(p, sched, u).L_max);
      // first unit: overlaps [A, ...) (a unit of no pages: sits at or after A)
      if (my_a == NU && (cu > 0 ? (U + cu > A) : (U >= A))) my_a = u;
      if (c == G - 1 || U < B) my_b = u;
      U += cu;
    }
    if (my_a < NU) atomicMin(&ua_s, my_a);
    if (my_b >= 0) atomicMax(&ub_s, my_b);
    __syncthreads();
    if (ua_s >= u0 && ua_s < u1) {
      long long V = off + incl - sum;
      for (int u = u0; u < ua_s; ++u) V += unit_cost(unit_weight(sched, u), prefill_pair<H>(p, sched, u).L_max);
      uua_s = V;
    }
    // both scratch slots of this CTA start empty
    if (tid < 2) p.pslot[(2 * c + tid) * kPreSlotInts] = -1;
    __syncthreads();
    if (tid == 0) {
      rg.A = A;
      rg.B = B;
      rg.W = W;
      rg.Uua = uua_s;
      rg.ua = ua_s;
      rg.ub = ub_s;
      rg.last = (c == G - 1) ? 1 : 0;
    }
    __syncthreads();
  }
  if (rg.ua > rg.ub) return;                        // no work for this CTA

  // ---- tensor memory, barriers
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_base_s), kPreTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int s = 0; s < kPreStages; ++s) {
      mbar_init(smem_u32(&raw_full[s]), 1);
      mbar_init(smem_u32(&raw_empty[s]), 128);  // the page's dequant group
    }
    for (int h = 0; h < 2; ++h) {
      mbar_init(smem_u32(&b_full[h]), 128);     // dequant group h
      for (int d = 0; d < 2; ++d) {
        mbar_init(smem_u32(&d_full[h][d]), 1);    // MMA issuer of tile h commits
        mbar_init(smem_u32(&d_empty[h][d]), 128); // epilogue of tile h
      }
      mbar_init(smem_u32(&q_full[h]), 128);     // epilogue of tile h writes its A tile
    }
    mbar_init(smem_u32(&q_empty), 2);           // both MMA issuers commit per pair
    abort_s = 0;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_base_s;
  auto fail = [&]() {
    if (!abort_s) {
      abort_s = 1;
      atomicOr(p.status, kStatusTimeout);
    }
  };

  if (warp < 4) {
    // warpgroup 0 gives registers back to the epilogues (executed by all four
    // warps of the warpgroup; warp 3 has no other role)
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsCtl));
    if (warp == 0) {
      // ================================================= producer (TMA)
      if (lane == 0) {
        int64_t g = 0;
        for (PreWalk sw(&rg); sw.more() && !abort_s;) {
          PairInfo pi;
          int w, ja, jb;
          sw.get<H>(p, sched, pi, w, ja, jb);
          sw.next(w, pi.L_max);
          for (int j = ja; j < jb; ++j, ++g) {
            const int s = (int)(g % kPreStages);
            if (!mbar_wait_or_abort<kSleep>(smem_u32(&raw_empty[s]), (uint32_t)(((g / kPreStages) & 1) ^ 1),
                                    &abort_s, lim)) {
              fail();
              break;
            }
            const uint32_t fb = smem_u32(&raw_full[s]);
            const int phys = __ldg(p.page_table + (int64_t)pi.r * p.pt_stride + j);
            if (phys < 0 || phys >= p.num_blocks) {
              mbar_arrive(fb);
            } else {
              mbar_arrive_expect_tx(fb, PF::kPageBytes);
              bulk_g2s(sbase + PreLayout::kStageOff + s * PF::kPageBytes, p.kv + (int64_t)phys * PF::kPageBytes,
                       PF::kPageBytes, fb);
            }
          }
        }
        // wait for every copy issued before the CTA may exit: the readers of
        // a stage stop waiting once another role's wait ran out
        for (int64_t k = (g > kPreStages ? g - kPreStages : 0); k < g; ++k)
          mbar_wait(smem_u32(&raw_full[k % kPreStages]), (uint32_t)((k / kPreStages) & 1));
      }
    } else if (warp == 1 || warp == 2) {
      // ================================================= MMA issuers
      // Issuer x multiplies every page against tile x's queries.
      if (lane == 0) {
        const int x = warp - 1;
        constexpr uint32_t idesc = idesc_f16_f32(128, 128, PF::kBf16);
        const uint32_t qaddr = sbase + PreLayout::kQOff + (uint32_t)x * kTileBytes;
        // operand descriptors of every K step, computed once
        uint64_t ad[8];
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) ad[kk] = desc_advance(smem_desc_sw128(qaddr), kstep_bytes(kk));
        const uint64_t bdesc_t0 = smem_desc_sw128(sbase + PreLayout::kBOff);
        const uint64_t bdesc_t1 = smem_desc_sw128(sbase + PreLayout::kBOff + kTileBytes);
        int64_t g = 0;
        int ip = 0;                                   // pairs with pages so far
        uint32_t last_bar = 0, last_par = 0;
        for (PreWalk sw(&rg); sw.more() && !abort_s;) {
          PairInfo pi;
          int w, ja, jb;
          sw.get<H>(p, sched, pi, w, ja, jb);
          sw.next(w, pi.L_max);
          if (jb <= ja) continue;                     // no pages of this unit here
          if (!mbar_wait_or_abort<kSleep>(smem_u32(&q_full[x]), (uint32_t)(ip & 1), &abort_s, lim)) { fail(); break; }
          bool ok = true;
          for (int j = ja; j < jb; ++j, ++g) {
            const int b = (int)(g & 1);
            const uint32_t par = (uint32_t)((g >> 1) & 1);
            if (!mbar_wait_or_abort<kSleep>(smem_u32(&b_full[b]), par, &abort_s, lim) ||
                !mbar_wait_or_abort<kSleep>(smem_u32(&d_empty[x][b]), par ^ 1u, &abort_s, lim)) {
              fail();
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t dt = tbase + (uint32_t)(x * 256 + b * 128);
            const uint64_t bdesc = b ? bdesc_t1 : bdesc_t0;     // B tile of the page's dequant group
            uint64_t bd[8];
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) bd[kk] = desc_advance(bdesc, kstep_bytes(kk));
            // the page's 8 MMAs and one commit: d_full[x][b] also tells
            // dequant group b that tile x is done with its B tile
            mma8_f16_ss_commit(dt, ad, bd, idesc, smem_u32(&d_full[x][b]));
            last_bar = smem_u32(&d_full[x][b]);
            last_par = par;
          }
          if (!ok || abort_s) break;
          mma_commit(smem_u32(&q_empty));
          ++ip;
        }
        // a commit covers every MMA issued before it: wait for the last one
        // before tensor memory may be freed (the epilogues stop waiting once
        // another role's wait ran out)
        if (last_bar != 0) mbar_wait(last_bar, last_par);
      }
    }
  } else if (warp < 12) {
    // ================================================= dequant warpgroups
    // Group grp takes the pages of parity grp and owns B tile grp, so each of
    // its barriers has one waiter that takes the phases in order.  These
    // waits are on every page's critical path and spin without the 1 ms
    // sleep limit the other roles' waits ask for (measured: 1.5 % slower
    // with it; the MMA issuers' sleep is where the gain comes from).
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsDq));
    const int grp = (warp - 4) >> 2;
    const int tok = ((warp & 3) << 5) | lane;        // token row of the page / of the B tile
    uint8_t* const bt = base + PreLayout::kBOff + grp * kTileBytes;
    int64_t g = 0;
    bool ok = true;
    for (PreWalk sw(&rg); sw.more() && ok;) {
      PairInfo pi;
      int w, ja, jb;
      sw.get<H>(p, sched, pi, w, ja, jb);
      sw.next(w, pi.L_max);
      for (int j = ja; j < jb; ++j, ++g) {
        if ((int)(g & 1) != grp) continue;
        const int s = (int)(g % kPreStages);
        if (!__all_sync(0xffffffffu, mbar_wait_or_abort(smem_u32(&raw_full[s]),
                                                         (uint32_t)((g / kPreStages) & 1), &abort_s, lim))) {
          fail();
          ok = false;
          break;
        }
        typename PF::Row row;
        PF::load(base + PreLayout::kStageOff + s * PF::kPageBytes, tok, row);
        mbar_arrive(smem_u32(&raw_empty[s]));
        // the B tile is free once both tiles' MMAs of page g - 2 are done:
        // phase (g - 2) / 2 of d_full[0][grp] and d_full[1][grp] (this group
        // waits on each of them at every one of its pages, in order; the next
        // phase needs this page)
        const uint32_t fpar = (uint32_t)((((g >> 1) - 1)) & 1);
        if (g >= 2 &&
            !__all_sync(0xffffffffu, mbar_wait_or_abort(smem_u32(&d_full[0][grp]), fpar, &abort_s, lim) &&
                                         mbar_wait_or_abort(smem_u32(&d_full[1][grp]), fpar, &abort_s, lim))) {
          fail();
          ok = false;
          break;
        }
#pragma unroll
        for (int g8 = 0; g8 < 8; ++g8) {
          uint32_t o[8];
          PF::chunk16(row, g8, o);
          // elements 16*g8 .. +15 = 16-byte chunks 2*g8, 2*g8+1 of the row
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int c16 = 2 * g8 + h;
            *reinterpret_cast<uint4*>(bt + (c16 >> 3) * (128 * 128) + sw128_offset(tok, c16 & 7)) =
                make_uint4(o[4 * h], o[4 * h + 1], o[4 * h + 2], o[4 * h + 3]);
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(smem_u32(&b_full[grp]));
      }
    }
  } else {
    // ================================================= epilogue warpgroups
    // Warpgroup x handles tile x of every pair; thread = query row.
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsEpi));
    const int x = (warp - 12) >> 2;
    const int n = ((warp & 3) << 5) | lane;          // query row = tensor-memory lane
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t bar_id = 2 + x;                   // named barrier of this warpgroup
    uint8_t* const qt = base + PreLayout::kQOff + x * kTileBytes;
    TopK15 top;
    bool ok = true;
    int64_t g = 0;
    int ip = 0;
    for (PreWalk sw(&rg); sw.more();) {
      // every warp of the group takes the same decision (a barrier it skipped
      // would otherwise hold the others): once a wait has run out, the walk
      // goes on without waiting, only to mark the remaining rows as failed
      if (named_bar_red_or(bar_id, 128, (!ok || abort_s) ? 1 : 0)) ok = false;
      PairInfo pi;
      int w, ja, jb;
      sw.get<H>(p, sched, pi, w, ja, jb);
      const int u = sw.u;
      sw.next(w, pi.L_max);
      if (jb <= ja && pi.L_max > 0) continue;        // none of this unit's pages here
      const TileRows tr = x ? pi.tile[1] : pi.tile[0];
      const int rows = tr.nt * H;
      const int pos = pi.ctx + tr.t0 + n / H;
      const int L = (n < rows && pos >= 0 && !pi.table_bad) ? (pos >> 7) : -1;
      if (jb > ja) {
        // this tile's queries -> fp16 A tile, once the MMAs of the previous
        // unit are done with it
        if (ok && ip > 0 && !__all_sync(0xffffffffu, mbar_wait_or_abort<kSleep>(smem_u32(&q_empty),
                                                                    (uint32_t)((ip - 1) & 1), &abort_s, lim))) {
          fail();
          ok = false;
        }
        if (ok) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            uint4 e = make_uint4(0, 0, 0, 0);
            if (n < rows) e = __ldg(reinterpret_cast<const uint4*>(p.q + ((int64_t)tr.row0 * H + n) * 128) + i);
            const uint32_t ew[4] = {e.x, e.y, e.z, e.w};
            uint32_t a[8];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              a[2 * k] = PF::widen_q(ew[k] & 0xFFFFu);
              a[2 * k + 1] = PF::widen_q(ew[k] >> 16);
            }
            // 16 query bytes = elements 16i .. 16i+15 = 16-byte chunks 2i, 2i+1
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int c16 = 2 * i + h;
              *reinterpret_cast<uint4*>(qt + (c16 >> 3) * (128 * 128) + sw128_offset(n, c16 & 7)) =
                  make_uint4(a[4 * h], a[4 * h + 1], a[4 * h + 2], a[4 * h + 3]);
            }
          }
          fence_proxy_async_smem();
          mbar_arrive(smem_u32(&q_full[x]));
        }
        ++ip;
      }
      // a request with an unreadable history page gets all -1 rows
      int tile_bad = pi.table_bad ? 1 : 0;
      if (!pi.table_bad) {
        const int seq = __ldg(p.seq_lens + pi.r);
        const int hist = seq >= 1 ? (seq - 1) >> 7 : 0;
        for (int jj = n; jj < hist; jj += 128) {
          const int ph = __ldg(p.page_table + (int64_t)pi.r * p.pt_stride + jj);
          tile_bad |= (ph < 0 || ph >= p.num_blocks);
        }
      }
      tile_bad = named_bar_red_or(bar_id, 128, tile_bad);
      if (n == 0 && tile_bad && rows > 0) atomicOr(p.status, pi.table_bad ? kStatusBadTable : kStatusBadPage);
      top.reset();
      for (int j = ja; j < jb; ++j, ++g) {
        const int b = (int)(g & 1);
        if (!ok) continue;
        if (!__all_sync(0xffffffffu, mbar_wait_or_abort<kSleep>(smem_u32(&d_full[x][b]), (uint32_t)((g >> 1) & 1),
                                                         &abort_s, lim))) {
          fail();
          ok = false;
          continue;
        }
        tc_fence_after();
        const uint32_t dt = tbase + lane_base + (uint32_t)(x * 256 + b * 128);
        // the row's maximum over the page's 128 tokens: the tensor-memory
        // loads reduce 32 columns each
        float m = -CUDART_INF_F;
#pragma unroll 1
        for (int c = 0; c < 128; c += 32) {
          float v[32];
          const float r = tmem_ld_red_max_32x32b_x32(dt + (uint32_t)c, v);
          tmem_wait_ld();
          m = fmaxf(m, r);
        }
        m = canon_zero(m);
        tc_fence_before();
        mbar_arrive(smem_u32(&d_empty[x][b]));
        if (j < L) {
          top.insert(m, j);
          if (p.scores_dbg) p.scores_dbg[((int64_t)tr.row0 * H + n) * p.dbg_stride + j] = m;
        }
      }
      // after a wait ran out the unit's rows are -1: written here, or by the
      // merge for a unit cut by a CTA boundary (its slot says so, for the
      // whole tile: the warps' outcomes are combined first)
      const bool tile_failed = named_bar_red_or(bar_id, 128, ok ? 0 : 1) != 0;
      if (ja == 0 && jb == pi.L_max) {
        if (n < rows)
          write_out_row(p.out + ((int64_t)tr.row0 * H + n) * kTopK, top.id, L, tile_bad != 0 || !ok);
      } else {
        // cut by a CTA boundary: this CTA's candidates go to its slot of the
        // unit (2c for its first unit, 2c + 1 for its last) and
        // prefill_merge_kernel writes the rows
        const int slot = 2 * c + (u == rg.ua ? 0 : 1);
        float2* dst = p.pcand + (((int64_t)slot * 2 + x) * 128 + n) * kHistK;
        if (!tile_failed) {
#pragma unroll
          for (int k = 0; k < kHistK; ++k) dst[k] = make_float2(top.s[k], __int_as_float(top.id[k]));
        }
        if (n == 0) p.pslot[slot * kPreSlotInts + 19 + x] = tile_failed ? 1 : 0;
        if (x == 0 && n == 0) {
          int32_t* m = p.pslot + slot * kPreSlotInts;
          m[1] = ja;
          m[2] = jb;
          m[3] = pi.L_max;
          m[4] = pi.r;
          m[5] = pi.ctx;
#pragma unroll
          for (int y = 0; y < 2; ++y) {
            m[6 + 3 * y] = pi.tile[y].t0;
            m[7 + 3 * y] = pi.tile[y].nt;
            m[8 + 3 * y] = pi.tile[y].row0;
          }
          m[12] = tile_bad;
          m[13] = w;
          // weighted position of page 0 (the walk has moved past the unit)
          const long long U0 = sw.U - unit_cost(w, pi.L_max) + kUnitOverhead;
          m[14] = (int32_t)(uint32_t)(U0 & 0xFFFFFFFFll);
          m[15] = (int32_t)(U0 >> 32);
          m[16] = (int32_t)(uint32_t)(rg.W & 0xFFFFFFFFll);
          m[17] = (int32_t)(rg.W >> 32);
          m[18] = pi.table_bad ? 1 : 0;
          m[0] = u;
        }
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tbase, kPreTmemCols);
}

// Merge the sorted candidate list b (15 (score, id) entries from another
// CTA, id < 0 = none) into the top 15 (s, id): the result is the first 15 of
// both by (score descending, id ascending); the lists hold disjoint ids and
// their empty entries come last.  With both lists padded to 16 entries and
// an empty entry keyed (-inf, INT_MAX), c_i = the better of a_i and b_(15-i)
// holds the 16 best of both as a bitonic sequence (a descending, then b
// ascending), which four rounds of compare-exchange, 8 / 4 / 2 / 1 apart,
// sort (Batcher's bitonic merge): 48 compare-exchanges.
__device__ __forceinline__ bool cand_better(float s1, int i1, float s2, int i2) {
  return s1 > s2 || (s1 == s2 && i1 < i2);
}
__device__ __forceinline__ void merge_top15_list(float (&s)[kHistK], int (&id)[kHistK], const float2* b) {
  constexpr int kNone = 0x7FFFFFFF;
  float2 bb[kHistK];
#pragma unroll
  for (int k = 0; k < kHistK; ++k) bb[k] = b[k];
  float cs[16];
  int ci[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float as = i < kHistK && id[i] >= 0 ? s[i] : -CUDART_INF_F;
    const int ai = i < kHistK && id[i] >= 0 ? id[i] : kNone;
    const int jb = 15 - i;                           // b_(15 - i); b_15 is the padding
    const int bi0 = jb < kHistK ? __float_as_int(bb[jb < kHistK ? jb : 0].y) : -1;
    const float bs = bi0 >= 0 ? bb[jb < kHistK ? jb : 0].x : -CUDART_INF_F;
    const int bi = bi0 >= 0 ? bi0 : kNone;
    const bool ta = cand_better(as, ai, bs, bi);
    cs[i] = ta ? as : bs;
    ci[i] = ta ? ai : bi;
  }
#pragma unroll
  for (int d = 8; d >= 1; d >>= 1) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (i & d) continue;
      const bool sw = cand_better(cs[i + d], ci[i + d], cs[i], ci[i]);
      const float ts = sw ? cs[i + d] : cs[i], us = sw ? cs[i] : cs[i + d];
      const int ti = sw ? ci[i + d] : ci[i], ui = sw ? ci[i] : ci[i + d];
      cs[i] = ts;
      ci[i] = ti;
      cs[i + d] = us;
      ci[i + d] = ui;
    }
  }
#pragma unroll
  for (int k = 0; k < kHistK; ++k) {
    s[k] = ci[k] != kNone ? cs[k] : -CUDART_INF_F;
    id[k] = ci[k] != kNone ? ci[k] : -1;
  }
}

// Rows of the units cut by CTA boundaries: block c takes each unit whose first
// page lies in CTA c's range and that goes on past it, merges the candidate
// lists that the CTAs holding its pages left (in page order, so equal scores
// keep the lower page id first) and writes the unit's rows; thread = row of
// tile (t / 128).
template <int H>
__global__ void __launch_bounds__(256) prefill_merge_kernel(const PrefillParams p) {
  griddep_wait();                                    // the scoring grid's candidates are written
  const int c = blockIdx.x, G = gridDim.x;
  const int x = threadIdx.x >> 7, n = threadIdx.x & 127;
  for (int sh = 0; sh < 2; ++sh) {
    const int slot = 2 * c + sh;
    const int32_t* m = p.pslot + slot * kPreSlotInts;
    const int u = m[0];
    if (u < 0 || m[1] != 0) continue;                // empty, or begun in an earlier CTA
    const int L = m[3], w = m[13];
    const long long U = (long long)(uint32_t)m[14] | ((long long)m[15] << 32);
    const long long W = (long long)(uint32_t)m[16] | ((long long)m[17] << 32);
    const int cl = split_cta(U + (long long)w * (L - 1), W, G);   // CTA of its last page
    const int t0 = m[6 + 3 * x], nt = m[7 + 3 * x], row0 = m[8 + 3 * x];
    if (n >= nt * H) continue;
    float s[kHistK];
    int id[kHistK];
    // m[19 + x]: tile x's candidates are incomplete (a wait ran out)
    bool failed = m[19 + x] != 0;
    {
      const float2* own = p.pcand + (((int64_t)slot * 2 + x) * 128 + n) * kHistK;
      for (int k = 0; k < kHistK; ++k) {
        s[k] = own[k].x;
        id[k] = __float_as_int(own[k].y);
      }
    }
    for (int cc = c + 1; cc <= cl && cc < G; ++cc) {
      if (p.pslot[(2 * cc) * kPreSlotInts] != u) continue;   // none of the unit's pages there
      if (p.pslot[(2 * cc) * kPreSlotInts + 19 + x]) failed = true;
      else merge_top15_list(s, id, p.pcand + (((int64_t)(2 * cc) * 2 + x) * 128 + n) * kHistK);
    }
    const int pos = m[5] + t0 + n / H;
    const int Lrow = (pos >= 0 && !m[18]) ? (pos >> 7) : -1;
    write_out_row(p.out + ((int64_t)row0 * H + n) * kTopK, id, Lrow, m[12] != 0 || failed);
  }
}

template <int H, class PF>
static cudaError_t launch_prefill_h(const PrefillParams& p, int grid, cudaStream_t stream) {
  const size_t smem = PreLayout<PF>::bytes(p.num_reqs);   // > 114 KB: one CTA per SM
  cudaError_t e = cudaFuncSetAttribute(prefill_kernel<H, PF>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  prefill_kernel<H, PF><<<grid, kPreThreads, smem, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_dependent(prefill_merge_kernel<H>, (unsigned)grid, 256u, 0, stream, p);
}

template <class PF>
static cudaError_t launch_prefill_pf(const PrefillParams& p, int grid, cudaStream_t stream) {
  switch (p.H) {
    case 1: return launch_prefill_h<1, PF>(p, grid, stream);
    case 2: return launch_prefill_h<2, PF>(p, grid, stream);
    case 4: return launch_prefill_h<4, PF>(p, grid, stream);
    default: return launch_prefill_h<8, PF>(p, grid, stream);
  }
}

cudaError_t launch_prefill(const PrefillParams& p, int grid, cudaStream_t stream) {
  return p.page_format == kPagesMxfp4 ? launch_prefill_pf<Mxfp4Pages>(p, grid, stream)
                                      : launch_prefill_pf<Nvfp4Pages>(p, grid, stream);
}

}  // namespace nvfp4idx
