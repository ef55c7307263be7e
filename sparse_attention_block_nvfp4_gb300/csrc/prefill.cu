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
// request (the last tile of a request may be ragged).  A CTA takes a PAIR of
// consecutive tiles of one request (tiles ntile-1-2k and ntile-2-2k) and
// walks the pages of the later one, which has the most: every page is
// dequantised once and multiplied against both tiles, so the CUDA-core work
// per unit of tensor work is halved.  Work units are dealt round-robin to the
// CTAs (one per SM): first the pairs (requests in order, last tiles first),
// then the tiles left over as singles (a pair whose second tile is empty).
// How many pairs to form is chosen so that the slowest CTA finishes first:
// all possible pairs, or only whole rounds of pairs (one per CTA) with the
// rest as singles, whichever gives the smaller estimated makespan (a pair
// costs about 1.7 singles).
// Warp roles, one per warpgroup (setmaxnreg moves registers between them),
// linked by mbarrier rings:
//   * warpgroup 0 (40 registers): warp 0 has the TMA unit copy each raw
//     9216-byte page into a 6-stage shared ring; warps 1 / 2 issue the 8
//     tcgen05.mma of every page for tile A / tile B (both operands in shared
//     memory: the tile's queries, M = 128, and the page, N = 128; K = 16),
//     D[row][token] in fp32 in tensor memory, two accumulators per tile;
//     warp 3 idles;
//   * warpgroups 1 / 2 (88 registers, pages of even / odd index): thread t
//     dequantises token t to fp16 into the group's own 128B-swizzled K-major
//     B tile [128 tokens x 128];
//   * warpgroups 3 / 4 (128 registers, tile A / tile B), thread = query row:
//     at a pair start widen the tile's E4M3 queries into a 128B-swizzled
//     fp16 A tile in shared memory; per page load the row of D (16 columns
//     per tcgen05.ld), take the max over the 128 tokens and update the row's
//     top-15 if the page is a history page of its token; write the row at the
//     end of the pair.
#include <cstdint>
#include <cuda_runtime.h>

#include "codec.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "topk.cuh"

namespace nvfp4idx {

constexpr int kPreStages = 6;              // raw page ring (even: pages of one parity per stage)
constexpr int kPreThreads = 640;           // 5 warpgroups
// 4 x 40 + 8 x 88 + 8 x 128 = 1888 registers per lane slot <= 640 x 96 / 32
constexpr uint32_t kRegsCtl = 40, kRegsDq = 88, kRegsEpi = 128;
constexpr uint32_t kPreTmemCols = 512;     // tile A: D [0,128), [128,256); tile B: [256,384), [384,512)
constexpr uint32_t kTileBytes = 128 * 256; // fp16 [2 K-blocks][128 rows][64], 128B swizzle

struct PreLayout {
  static constexpr uint32_t kQOff = 0;                           // A tiles of tile A and tile B
  static constexpr uint32_t kBOff = 2 * kTileBytes;              // B tiles of dequant groups 0 and 1
  static constexpr uint32_t kStageOff = kBOff + 2 * kTileBytes;
  static constexpr uint32_t kTpreOff = kStageOff + kPreStages * kPageBytes;
  // two prefix arrays per request: tiles and possible pairs
  static size_t bytes(int num_reqs) { return 1024 + kTpreOff + (size_t)(num_reqs + 1) * 8; }
};
static_assert(1024 + PreLayout::kTpreOff + (kMaxPrefillReqs + 1) * 8 + 1024 <= 227 * 1024,
              "prefill shared memory above the 227 KB a CTA may hold");

// Three-input maximum (one instruction on sm_100 and later).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// max of 64 floats: four independent chains of three-input maxima (one
// dependent chain of 64 maxima would be the epilogue's critical path)
__device__ __forceinline__ float max64(const float (&v)[64]) {
  float ma = fmax3(v[0], v[1], v[2]), mb = fmax3(v[3], v[4], v[5]), mc = fmax3(v[6], v[7], v[8]),
        md = fmax3(v[9], v[10], v[11]);
#pragma unroll
  for (int i = 12; i < 60; i += 8) {
    ma = fmax3(ma, v[i], v[i + 1]);
    mb = fmax3(mb, v[i + 2], v[i + 3]);
    mc = fmax3(mc, v[i + 4], v[i + 5]);
    md = fmax3(md, v[i + 6], v[i + 7]);
  }
  ma = fmax3(ma, v[60], v[61]);
  mb = fmax3(mb, v[62], v[63]);
  return fmaxf(fmaxf(ma, mb), fmaxf(mc, md));
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

template <int H>
__global__ void __launch_bounds__(kPreThreads, 1) prefill_kernel(const PrefillParams p) {
  constexpr int TQ = 128 / H;     // tokens per tile
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
  // how many pairs: all possible ones, or whole rounds of G pairs and the
  // rest as singles, whichever finishes sooner (pair ~ 17, single ~ 10)
  Sched sched{tpre, fpre, NR, 0};
  int NU;
  {
    const int NT = tpre[NR], Pall = fpre[NR];
    const int Sall = NT - 2 * Pall;
    const int Pr = min(Pall, (NT / (2 * G)) * G);
    const int Sr = NT - 2 * Pr;
    const long long cost_all = (long long)((Pall + G - 1) / G) * 17 + (long long)((Sall + G - 1) / G) * 10;
    const long long cost_rounds = (long long)((Pr + G - 1) / G) * 17 + (long long)((Sr + G - 1) / G) * 10;
    sched.P = cost_rounds < cost_all ? Pr : Pall;
    NU = NT - sched.P;                               // P pairs + (NT - 2P) singles
  }
  if (c >= NU) return;

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
        for (int t = c; t < NU && !abort_s; t += G) {
          const PairInfo pi = prefill_pair<H>(p, sched, t);
          for (int j = 0; j < pi.L_max; ++j, ++g) {
            const int s = (int)(g % kPreStages);
            if (!mbar_wait_or_abort(smem_u32(&raw_empty[s]), (uint32_t)(((g / kPreStages) & 1) ^ 1),
                                    &abort_s)) {
              fail();
              break;
            }
            const uint32_t fb = smem_u32(&raw_full[s]);
            const int phys = __ldg(p.page_table + (int64_t)pi.r * p.pt_stride + j);
            if (phys < 0 || phys >= p.num_blocks) {
              mbar_arrive(fb);
            } else {
              mbar_arrive_expect_tx(fb, kPageBytes);
              bulk_g2s(sbase + PreLayout::kStageOff + s * kPageBytes, p.kv + (int64_t)phys * kPageBytes,
                       kPageBytes, fb);
            }
          }
        }
        if (abort_s) {   // drain issued copies before the CTA may exit
          for (int64_t k = (g > kPreStages ? g - kPreStages : 0); k < g; ++k)
            mbar_wait(smem_u32(&raw_full[k % kPreStages]), (uint32_t)((k / kPreStages) & 1));
        }
      }
    } else if (warp == 1 || warp == 2) {
      // ================================================= MMA issuers
      // Issuer x multiplies every page against tile x's queries.
      if (lane == 0) {
        const int x = warp - 1;
        constexpr uint32_t idesc = idesc_f16_f32(128, 128);
        const uint32_t qaddr = sbase + PreLayout::kQOff + (uint32_t)x * kTileBytes;
        int64_t g = 0;
        int ip = 0;                                   // pairs with pages so far
        uint32_t last_bar = 0, last_par = 0;
        for (int t = c; t < NU && !abort_s; t += G) {
          const PairInfo pi = prefill_pair<H>(p, sched, t);
          if (pi.L_max == 0) continue;
          if (!mbar_wait_or_abort(smem_u32(&q_full[x]), (uint32_t)(ip & 1), &abort_s)) { fail(); break; }
          bool ok = true;
          for (int j = 0; j < pi.L_max; ++j, ++g) {
            const int b = (int)(g & 1);
            const uint32_t par = (uint32_t)((g >> 1) & 1);
            if (!mbar_wait_or_abort(smem_u32(&b_full[b]), par, &abort_s) ||
                !mbar_wait_or_abort(smem_u32(&d_empty[x][b]), par ^ 1u, &abort_s)) {
              fail();
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t bt = sbase + PreLayout::kBOff + (uint32_t)b * kTileBytes;
            const uint32_t dt = tbase + (uint32_t)(x * 256 + b * 128);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint32_t koff = (kk >> 2) * (128 * 128) + (kk & 3) * 32;
              mma_f16_ss(dt, smem_desc_sw128(qaddr + koff), smem_desc_sw128(bt + koff), idesc,
                         kk > 0 ? 1u : 0u);
            }
            // one commit per page: d_full[x][b] also tells dequant group b
            // that tile x is done with its B tile
            mma_commit(smem_u32(&d_full[x][b]));
            last_bar = smem_u32(&d_full[x][b]);
            last_par = par;
          }
          if (!ok || abort_s) break;
          mma_commit(smem_u32(&q_empty));
          ++ip;
        }
        // a commit covers every MMA issued before it: drain the last one
        // before tensor memory is freed
        if (abort_s && last_bar != 0) mbar_wait(last_bar, last_par);
      }
    }
  } else if (warp < 12) {
    // ================================================= dequant warpgroups
    // Group grp takes the pages of parity grp and owns B tile grp, so each of
    // its barriers has one waiter that takes the phases in order.
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsDq));
    const int grp = (warp - 4) >> 2;
    const int tok = ((warp & 3) << 5) | lane;        // token row of the page / of the B tile
    uint8_t* const bt = base + PreLayout::kBOff + grp * kTileBytes;
    int64_t g = 0;
    bool ok = true;
    for (int t = c; t < NU && ok; t += G) {
      const PairInfo pi = prefill_pair<H>(p, sched, t);
      for (int j = 0; j < pi.L_max; ++j, ++g) {
        if ((int)(g & 1) != grp) continue;
        const int s = (int)(g % kPreStages);
        if (!__all_sync(0xffffffffu, mbar_wait_or_abort(smem_u32(&raw_full[s]),
                                                         (uint32_t)((g / kPreStages) & 1), &abort_s))) {
          fail();
          ok = false;
          break;
        }
        uint32_t w[18];
        {
          const uint2* src = reinterpret_cast<const uint2*>(base + PreLayout::kStageOff + s * kPageBytes + tok * kRowBytes);
#pragma unroll
          for (int i = 0; i < 9; ++i) {
            const uint2 t2 = src[i];
            w[2 * i] = t2.x;
            w[2 * i + 1] = t2.y;
          }
        }
        mbar_arrive(smem_u32(&raw_empty[s]));
        // the B tile is free once both tiles' MMAs of page g - 2 are done:
        // phase (g - 2) / 2 of d_full[0][grp] and d_full[1][grp] (this group
        // waits on each of them at every one of its pages, in order; the next
        // phase needs this page)
        const uint32_t fpar = (uint32_t)((((g >> 1) - 1)) & 1);
        if (g >= 2 &&
            !__all_sync(0xffffffffu, mbar_wait_or_abort(smem_u32(&d_full[0][grp]), fpar, &abort_s) &&
                                         mbar_wait_or_abort(smem_u32(&d_full[1][grp]), fpar, &abort_s))) {
          fail();
          ok = false;
          break;
        }
        const uint32_t sc[4] = {e4m3x2_to_f16x2(w[16] & 0xFFFFu), e4m3x2_to_f16x2(w[16] >> 16),
                                e4m3x2_to_f16x2(w[17] & 0xFFFFu), e4m3x2_to_f16x2(w[17] >> 16)};
#pragma unroll
        for (int g8 = 0; g8 < 8; ++g8) {
          const uint32_t s2 = (g8 & 1) ? f16x2_bcast_hi(sc[g8 >> 1]) : f16x2_bcast_lo(sc[g8 >> 1]);
          uint32_t o[8];
          dequant16(w[2 * g8], w[2 * g8 + 1], s2, o);
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
    for (int t = c; t < NU; t += G) {
      // every warp of the group takes the same decision to stop (a barrier it
      // skipped would otherwise hold the others)
      if (named_bar_red_or(bar_id, 128, (!ok || abort_s) ? 1 : 0)) break;
      const PairInfo pi = prefill_pair<H>(p, sched, t);
      const TileRows tr = x ? pi.tile[1] : pi.tile[0];
      const int rows = tr.nt * H;
      const int pos = pi.ctx + tr.t0 + n / H;
      const int L = (n < rows && pos >= 0 && !pi.table_bad) ? (pos >> 7) : -1;
      if (pi.L_max > 0) {
        // this tile's queries -> fp16 A tile, once the MMAs of the previous
        // pair are done with it
        if (ip > 0 && !__all_sync(0xffffffffu, mbar_wait_or_abort(smem_u32(&q_empty),
                                                                    (uint32_t)((ip - 1) & 1), &abort_s))) {
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
              a[2 * k] = e4m3x2_to_f16x2(ew[k] & 0xFFFFu);
              a[2 * k + 1] = e4m3x2_to_f16x2(ew[k] >> 16);
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
      for (int j = 0; j < pi.L_max; ++j, ++g) {
        const int b = (int)(g & 1);
        if (!ok) continue;
        if (!__all_sync(0xffffffffu, mbar_wait_or_abort(smem_u32(&d_full[x][b]), (uint32_t)((g >> 1) & 1),
                                                         &abort_s))) {
          fail();
          ok = false;
          continue;
        }
        tc_fence_after();
        const uint32_t dt = tbase + lane_base + (uint32_t)(x * 256 + b * 128);
        float v[64];
#pragma unroll
        for (int c16 = 0; c16 < 64; c16 += 16) tmem_ld_32x32b_x16(dt + c16, v + c16);
        tmem_wait_ld();
        const float m0 = max64(v);
#pragma unroll
        for (int c16 = 0; c16 < 64; c16 += 16) tmem_ld_32x32b_x16(dt + 64 + c16, v + c16);
        tmem_wait_ld();
        const float m = canon_zero(fmaxf(m0, max64(v)));
        tc_fence_before();
        mbar_arrive(smem_u32(&d_empty[x][b]));
        if (j < L) {
          top.insert(m, j);
          if (p.scores_dbg) p.scores_dbg[((int64_t)tr.row0 * H + n) * p.dbg_stride + j] = m;
        }
      }
      if (ok && n < rows) write_out_row(p.out + ((int64_t)tr.row0 * H + n) * kTopK, top.id, L, tile_bad != 0);
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tbase, kPreTmemCols);
}

template <int H>
static cudaError_t launch_prefill_h(const PrefillParams& p, int grid, cudaStream_t stream) {
  const size_t smem = PreLayout::bytes(p.num_reqs);   // > 114 KB: one CTA per SM
  cudaError_t e = cudaFuncSetAttribute(prefill_kernel<H>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  prefill_kernel<H><<<grid, kPreThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_prefill(const PrefillParams& p, int grid, cudaStream_t stream) {
  switch (p.H) {
    case 1: return launch_prefill_h<1>(p, grid, stream);
    case 2: return launch_prefill_h<2>(p, grid, stream);
    case 4: return launch_prefill_h<4>(p, grid, stream);
    default: return launch_prefill_h<8>(p, grid, stream);
  }
}

}  // namespace nvfp4idx
