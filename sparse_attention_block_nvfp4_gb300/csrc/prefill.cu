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
// request (the last tile of a request may be ragged); its rows sit in tensor
// memory as the MMA's A operand (M = 128, K = 128).  Tiles of a request are
// visited last-first (they hold the most pages) and dealt round-robin to the
// CTAs, one CTA per SM.  Warp roles, linked by mbarrier rings, one role per
// warpgroup so that registers can move between them (setmaxnreg):
//   * warpgroup 0 (40 registers): warp 0 has the TMA unit copy each raw
//     9216-byte page into a 6-stage shared ring; warps 1 and 2 take alternate
//     pages, one thread each issuing 8 tcgen05.mma per page, D[row][token] =
//     Q . K^T in fp32, 3 accumulators deep; warp 3 idles;
//   * warpgroups 1 and 2 (dequant, alternating pages): thread t dequantises
//     token t to fp16 into a 128B-swizzled K-major B tile [128 tokens x 128]
//     (4 tiles deep);
//   * warpgroup 3 (epilogue, 208 registers), thread = query row: widens the
//     next tile's queries into tensor memory (2 buffers), loads its whole
//     128-column row of D per page in one round trip, takes the max over the
//     tokens and updates its running top-15 if the page is a history page of
//     its token; writes the row at the end of the tile.
#include <cstdint>
#include <cuda_runtime.h>

#include "codec.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "topk.cuh"

namespace nvfp4idx {

constexpr int kPreStages = 6;              // raw page ring
constexpr int kPreB = 4;                   // dequantised B tiles
constexpr int kPreD = 3;                   // accumulators: columns [128 + 128d, 256 + 128d)
// warpgroup 0: warp 0 TMA, warps 1 / 2 MMA issue, warp 3 idle (registers
// lowered to 40); warpgroups 1 / 2: dequant (128); warpgroup 3: epilogue
// (raised to 208, so a thread holds its whole 128-column row of D).
// 4 x 40 + 8 x 128 + 4 x 208 registers x 32 lanes = 64512 <= 512 x 128.
constexpr int kPreThreads = 512;
constexpr uint32_t kRegsCtl = 40, kRegsEpi = 208;
constexpr uint32_t kPreTmemCols = 512;     // queries [0,64) and [64,128), accumulators [128,512)
constexpr uint32_t kBTileBytes = 128 * 256;  // fp16 [2 K-blocks][128 tokens][64]

struct PreLayout {
  static constexpr uint32_t kBOff = 0;
  static constexpr uint32_t kStageOff = kPreB * kBTileBytes;
  static constexpr uint32_t kTpreOff = kStageOff + kPreStages * kPageBytes;
  static size_t bytes(int num_reqs) { return 1024 + kTpreOff + (size_t)(num_reqs + 1) * 4; }
};

// Three-input maximum (one instruction on sm_100 and later).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

struct TileInfo {
  int r, t0, nt, L_max, ctx, row0;   // row0 = first token (q row) of the tile
  bool table_bad;
};

template <int H>
__device__ __forceinline__ TileInfo prefill_tile(const PrefillParams& p, const int32_t* tpre, int t) {
  constexpr int TQ = 128 / H;
  int lo = 0, hi = p.num_reqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (tpre[mid] <= t) lo = mid; else hi = mid - 1;
  }
  TileInfo ti;
  ti.r = lo;
  const int cu0 = __ldg(p.cu_seqlens_q + lo);
  const int ql = __ldg(p.cu_seqlens_q + lo + 1) - cu0;
  const int ntile = (ql + TQ - 1) / TQ;
  const int lt = ntile - 1 - (t - tpre[lo]);        // last tile first
  ti.t0 = lt * TQ;
  ti.nt = min(TQ, ql - ti.t0);
  const int seq = __ldg(p.seq_lens + lo);
  ti.ctx = seq - ql;
  ti.row0 = cu0 + ti.t0;
  const int hist = seq >= 1 ? (seq - 1) >> 7 : 0;
  ti.table_bad = hist > p.pt_stride;
  const int pos_last = ti.ctx + ti.t0 + ti.nt - 1;
  ti.L_max = (pos_last >= 0 && !ti.table_bad) ? (pos_last >> 7) : 0;
  return ti;
}

template <int H>
__global__ void __launch_bounds__(kPreThreads, 1) prefill_kernel(const PrefillParams p) {
  constexpr int TQ = 128 / H;     // tokens per tile
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t raw_full[kPreStages], raw_empty[kPreStages];
  __shared__ __align__(8) uint64_t b_full[kPreB], b_empty[kPreB];
  __shared__ __align__(8) uint64_t d_full[kPreD], d_empty[kPreD];
  __shared__ __align__(8) uint64_t q_full[2], q_empty[2];
  __shared__ uint32_t tmem_base_s;
  __shared__ volatile int abort_s;
  __shared__ int warp_sum[kPreThreads / 32];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t sbase = (raw_u32 + 1023u) & ~1023u;
  uint8_t* const base = smem_raw + (sbase - raw_u32);
  int32_t* const tpre = reinterpret_cast<int32_t*>(base + PreLayout::kTpreOff);
  const int NR = p.num_reqs, G = gridDim.x, c = blockIdx.x;
  constexpr int NW = kPreThreads / 32;

  // ---- tiles per request -> exclusive prefix sums
  {
    const int per = (NR + kPreThreads - 1) / kPreThreads;
    const int r0 = tid * per, r1 = min(NR, r0 + per);
    int sum = 0;
    for (int r = r0; r < r1; ++r) {
      const int ql = __ldg(p.cu_seqlens_q + r + 1) - __ldg(p.cu_seqlens_q + r);
      sum += ql > 0 ? (ql + TQ - 1) / TQ : 0;
    }
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
      tpre[r] = run;
      const int ql = __ldg(p.cu_seqlens_q + r + 1) - __ldg(p.cu_seqlens_q + r);
      run += ql > 0 ? (ql + TQ - 1) / TQ : 0;
    }
    if (tid == kPreThreads - 1) {
      int tot = 0;
      for (int w = 0; w < NW; ++w) tot += warp_sum[w];
      tpre[NR] = tot;
    }
    __syncthreads();
  }
  const int NT = tpre[NR];
  if (c >= NT) return;

  // ---- tensor memory, barriers
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_base_s), kPreTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int s = 0; s < kPreStages; ++s) {
      mbar_init(smem_u32(&raw_full[s]), 1);
      mbar_init(smem_u32(&raw_empty[s]), 128);
    }
    for (int b = 0; b < kPreB; ++b) {
      mbar_init(smem_u32(&b_full[b]), 128);
      mbar_init(smem_u32(&b_empty[b]), 1);
    }
    for (int d = 0; d < kPreD; ++d) {
      mbar_init(smem_u32(&d_full[d]), 1);
      mbar_init(smem_u32(&d_empty[d]), 128);
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(smem_u32(&q_full[k]), 128);
      mbar_init(smem_u32(&q_empty[k]), 2);   // both MMA issuers commit
    }
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
    // warpgroup 0 gives registers back to the epilogue (executed by all
    // four warps of the warpgroup, warp 3 has no other role)
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsCtl));
    if (warp == 0) {
      // ================================================= producer (TMA)
      if (lane == 0) {
        int64_t g = 0;
        for (int t = c; t < NT && !abort_s; t += G) {
          const TileInfo ti = prefill_tile<H>(p, tpre, t);
          for (int j = 0; j < ti.L_max; ++j, ++g) {
            const int s = (int)(g % kPreStages);
            if (!mbar_wait_or_abort(smem_u32(&raw_empty[s]), (uint32_t)(((g / kPreStages) & 1) ^ 1), &abort_s)) {
              fail();
              break;
            }
            const uint32_t fb = smem_u32(&raw_full[s]);
            const int phys = __ldg(p.page_table + (int64_t)ti.r * p.pt_stride + j);
            if (phys < 0 || phys >= p.num_blocks) {
              mbar_arrive(fb);
            } else {
              mbar_arrive_expect_tx(fb, kPageBytes);
              bulk_g2s(sbase + PreLayout::kStageOff + s * kPageBytes, p.kv + (int64_t)phys * kPageBytes,
                       kPageBytes, fb);
            }
          }
        }
        if (abort_s) {
          for (int64_t k = (g > kPreStages ? g - kPreStages : 0); k < g; ++k)
            mbar_wait(smem_u32(&raw_full[k % kPreStages]), (uint32_t)((k / kPreStages) & 1));
        }
      }
    } else if (warp == 1 || warp == 2) {
      // ================================================= MMA issuers
      // Two issuing threads take alternate pages, so that one thread's commits
      // and waits overlap the other's MMAs and the tensor core stays busy.
      if (lane == 0) {
        const int mgrp = warp - 1;
        constexpr uint32_t idesc = idesc_f16_f32(128, 128);
        int64_t g = 0, g_last = -1;
        int kq = 0;
        for (int t = c; t < NT && !abort_s; t += G) {
          const TileInfo ti = prefill_tile<H>(p, tpre, t);
          if (ti.L_max == 0) continue;
          const int qb = kq & 1;
          if (!mbar_wait_or_abort(smem_u32(&q_full[qb]), (uint32_t)((kq >> 1) & 1), &abort_s)) { fail(); break; }
          for (int j = 0; j < ti.L_max; ++j, ++g) {
            if ((int)(g & 1) != mgrp) continue;
            const int nb = (int)(g % kPreB), d = (int)(g % kPreD);
            if (!mbar_wait_or_abort(smem_u32(&b_full[nb]), (uint32_t)((g / kPreB) & 1), &abort_s)) { fail(); break; }
            if (!mbar_wait_or_abort(smem_u32(&d_empty[d]), (uint32_t)(((g / kPreD) & 1) ^ 1), &abort_s)) { fail(); break; }
            tc_fence_after();
            const uint32_t bt = sbase + PreLayout::kBOff + (uint32_t)nb * kBTileBytes;
  #pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint64_t bdesc = smem_desc_sw128(bt + (kk >> 2) * (128 * 128) + (kk & 3) * 32);
              mma_f16_tmemA(tbase + 128 + d * 128, tbase + qb * 64 + kk * 8, bdesc, idesc, kk > 0 ? 1u : 0u);
            }
            mma_commit(smem_u32(&b_empty[nb]));
            mma_commit(smem_u32(&d_full[d]));
            g_last = g;
          }
          if (abort_s) break;
          mma_commit(smem_u32(&q_empty[qb]));
          ++kq;
        }
        if (abort_s && g_last >= 0) {
          const int64_t k = g_last;
          mbar_wait(smem_u32(&d_full[k % kPreD]), (uint32_t)((k / kPreD) & 1));
        }
      }
    }
  } else if (warp < 12) {
    // ================================================= dequant warpgroups
    const int grp = (warp - 4) >> 2;                 // 0 or 1: takes pages with g % 2 == grp
    const int tok = ((warp & 3) << 5) | lane;        // token row of the page / of the B tile
    int64_t g = 0;
    bool ok = true;
    for (int t = c; t < NT && ok; t += G) {
      const TileInfo ti = prefill_tile<H>(p, tpre, t);
      for (int j = 0; j < ti.L_max; ++j, ++g) {
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
        const int nb = (int)(g % kPreB);
        if (!__all_sync(0xffffffffu, mbar_wait_or_abort(smem_u32(&b_empty[nb]),
                                                         (uint32_t)(((g / kPreB) & 1) ^ 1), &abort_s))) {
          fail();
          ok = false;
          break;
        }
        uint8_t* bt = base + PreLayout::kBOff + nb * kBTileBytes;
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
        mbar_arrive(smem_u32(&b_full[nb]));
      }
    }
  } else {
    // ================================================= epilogue warpgroup
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsEpi));
    const int n = ((warp & 3) << 5) | lane;          // query row = tensor-memory lane
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    TopK15 top;
    bool ok = true;
    // widen tile t's queries into tensor-memory buffer qb (thread = row)
    auto load_q = [&](const TileInfo& ti, int qb) {
      uint32_t a[64];
      if (n < ti.nt * H) {
        const uint4* src = reinterpret_cast<const uint4*>(p.q + ((int64_t)ti.row0 * H + n) * 128);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint4 e = __ldg(src + i);
          const uint32_t ew[4] = {e.x, e.y, e.z, e.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            a[8 * i + 2 * k] = e4m3x2_to_f16x2(ew[k] & 0xFFFFu);
            a[8 * i + 2 * k + 1] = e4m3x2_to_f16x2(ew[k] >> 16);
          }
        }
      } else {
#pragma unroll
        for (int i = 0; i < 64; ++i) a[i] = 0u;
      }
      tc_fence_after();
      tmem_st_32x32b_x64(tbase + lane_base + qb * 64, a);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(smem_u32(&q_full[qb]));
    };
    // the k-th tile of this CTA that has pages (the MMA's tile sequence)
    auto next_mma_tile = [&](int from) {
      for (int t = from; t < NT; t += G)
        if (prefill_tile<H>(p, tpre, t).L_max > 0) return t;
      return NT;
    };
    int t_next_q = next_mma_tile(c);      // next tile whose queries are not loaded yet
    int kq_loaded = 0;
    if (t_next_q < NT) {
      load_q(prefill_tile<H>(p, tpre, t_next_q), 0);
      kq_loaded = 1;
      t_next_q = next_mma_tile(t_next_q + G);
    }
    int64_t g = 0;
    for (int t = c; t < NT; t += G) {
      // every epilogue warp takes the same decision to stop (a barrier it
      // skipped would otherwise hold the others)
      if (named_bar_red_or(2, 128, (!ok || abort_s) ? 1 : 0)) break;
      const TileInfo ti = prefill_tile<H>(p, tpre, t);
      const int rows = ti.nt * H;
      const int pos = ti.ctx + ti.t0 + n / H;
      const int L = (n < rows && pos >= 0) ? (pos >> 7) : -1;
      if (ti.L_max > 0 && t_next_q < NT) {
        // one tile ahead: queries of the next tile with pages
        const int qb = kq_loaded & 1;
        if (__all_sync(0xffffffffu, mbar_wait_or_abort(smem_u32(&q_empty[qb]),
                                                        (uint32_t)(((kq_loaded >> 1) & 1) ^ 1), &abort_s))) {
          load_q(prefill_tile<H>(p, tpre, t_next_q), qb);
        } else {
          fail();
          ok = false;
        }
        ++kq_loaded;
        t_next_q = next_mma_tile(t_next_q + G);
      }
      // a request with an unreadable history page gets all -1 rows
      int tile_bad = ti.table_bad ? 1 : 0;
      if (!ti.table_bad) {
        const int seq = __ldg(p.seq_lens + ti.r);
        const int hist = seq >= 1 ? (seq - 1) >> 7 : 0;
        for (int jj = n; jj < hist; jj += 128) {
          const int ph = __ldg(p.page_table + (int64_t)ti.r * p.pt_stride + jj);
          tile_bad |= (ph < 0 || ph >= p.num_blocks);
        }
      }
      tile_bad = named_bar_red_or(2, 128, tile_bad);
      if (n == 0 && tile_bad) atomicOr(p.status, ti.table_bad ? kStatusBadTable : kStatusBadPage);
      top.reset();
      for (int j = 0; j < ti.L_max; ++j, ++g) {
        const int d = (int)(g % kPreD);
        if (!ok) continue;
        if (!__all_sync(0xffffffffu, mbar_wait_or_abort(smem_u32(&d_full[d]),
                                                         (uint32_t)((g / kPreD) & 1), &abort_s))) {
          fail();
          ok = false;
          continue;
        }
        tc_fence_after();
        const uint32_t dt = tbase + lane_base + 128 + d * 128;
        float v[128];
#pragma unroll
        for (int c16 = 0; c16 < 128; c16 += 16) tmem_ld_32x32b_x16(dt + c16, v + c16);
        tmem_wait_ld();
        float ma = fmax3(v[0], v[1], v[2]), mb = fmax3(v[3], v[4], v[5]), mc = fmax3(v[6], v[7], v[8]),
              md = fmax3(v[9], v[10], v[11]);
#pragma unroll
        for (int i = 12; i < 124; i += 8) {
          ma = fmax3(ma, v[i], v[i + 1]);
          mb = fmax3(mb, v[i + 2], v[i + 3]);
          mc = fmax3(mc, v[i + 4], v[i + 5]);
          md = fmax3(md, v[i + 6], v[i + 7]);
        }
        ma = fmax3(ma, v[124], v[125]);
        mb = fmax3(mb, v[126], v[127]);
        float m = fmaxf(fmaxf(ma, mb), fmaxf(mc, md));
        tc_fence_before();
        mbar_arrive(smem_u32(&d_empty[d]));
        m = canon_zero(m);
        if (j < L) {
          top.insert(m, j);
          if (p.scores_dbg) p.scores_dbg[((int64_t)ti.row0 * H + n) * p.dbg_stride + j] = m;
        }
      }
      if (ok && n < rows) write_out_row(p.out + ((int64_t)ti.row0 * H + n) * kTopK, top.id, L, tile_bad != 0);
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
