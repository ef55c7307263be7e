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
// request (the last tile of a request may be ragged).  Its rows go into
// tensor memory once (E4M3 widened exactly to fp16) and serve as the A
// operand, M = 128, K = 128.  For every history page of the tile:
//   * the TMA unit copies the raw 9216-byte page into a shared stage;
//   * thread t dequantises token t to fp16 and writes it into a 128B-swizzled
//     K-major B tile [128 tokens x 128] (double buffered);
//   * one thread issues 8 tcgen05.mma: D[row][token] = Q . K^T in fp32;
//   * while that runs, each thread (= one query row) loads the previous
//     page's D row from tensor memory, takes the max over the 128 tokens and
//     updates its running top-15 if the page is a history page of its token.
// Tiles of a request are visited last-first (they hold the most pages) and
// dealt round-robin to the CTAs.
#include <cstdint>
#include <cuda_runtime.h>

#include "codec.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "topk.cuh"

namespace nvfp4idx {

constexpr int kPreStages = 4;
constexpr int kPreThreads = 128;
constexpr uint32_t kPreTmemCols = 256;     // Q [0,64), D [128,256)
constexpr uint32_t kBTileBytes = 128 * 256;  // fp16 [2 K-blocks][128 tokens][64]

struct PreLayout {
  static constexpr uint32_t kBOff = 0;                                  // 2 x 32 KB
  static constexpr uint32_t kStageOff = 2 * kBTileBytes;
  static constexpr uint32_t kTpreOff = kStageOff + kPreStages * kPageBytes;
  static size_t bytes(int num_reqs) { return 1024 + kTpreOff + (size_t)(num_reqs + 1) * 4; }
};

struct TileInfo {
  int r, t0, nt, L_max, ctx, row0;   // row0 = first q row of the tile (token index)
  bool table_bad;
};

template <int H>
__global__ void __launch_bounds__(kPreThreads, 2) prefill_kernel(const PrefillParams p) {
  constexpr int TQ = 128 / H;     // tokens per tile
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[kPreStages];
  __shared__ __align__(8) uint64_t mma_bar;
  __shared__ int stage_bad[kPreStages];
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_s;
  __shared__ int warp_sum[4];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t sbase = (raw_u32 + 1023u) & ~1023u;
  uint8_t* const base = smem_raw + (sbase - raw_u32);
  int32_t* const tpre = reinterpret_cast<int32_t*>(base + PreLayout::kTpreOff);
  const int NR = p.num_reqs, G = gridDim.x, c = blockIdx.x;

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
    if (tid == kPreThreads - 1) tpre[NR] = off + incl;
    __syncthreads();
  }
  const int NT = tpre[NR];
  if (c >= NT) return;

  auto tile_info = [&](int t) {
    int lo = 0, hi = NR - 1;
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
  };

  // ---- tensor memory, barriers
  if (warp == 0) {
    tmem_alloc(smem_u32(&tmem_base_s), kPreTmemCols);
    tmem_relinquish();
  }
  if (tid == 32) {
    for (int s = 0; s < kPreStages; ++s) mbar_init(smem_u32(&full_bar[s]), 1);
    mbar_init(smem_u32(&mma_bar), 1);
    abort_s = 0;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tmem_base_s;
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;

  // ---- producer (thread 0): walks (tile, page) in the consumers' order
  int p_tile = c;               // tile index
  int p_j = 0;                  // page within tile
  TileInfo p_ti;
  int64_t issued = 0;
  if (tid == 0) {
    p_ti = tile_info(p_tile);
    while (p_tile < NT && p_ti.L_max == 0) {
      p_tile += G;
      if (p_tile < NT) p_ti = tile_info(p_tile);
    }
  }
  auto produce = [&]() {
    const int stage = (int)(issued % kPreStages);
    const uint32_t fb = smem_u32(&full_bar[stage]);
    const int phys = __ldg(p.page_table + (int64_t)p_ti.r * p.pt_stride + p_j);
    if (phys < 0 || phys >= p.num_blocks) {
      stage_bad[stage] = 1;
      mbar_arrive(fb);
    } else {
      stage_bad[stage] = 0;
      mbar_arrive_expect_tx(fb, kPageBytes);
      bulk_g2s(sbase + PreLayout::kStageOff + stage * kPageBytes, p.kv + (int64_t)phys * kPageBytes,
               kPageBytes, fb);
    }
    ++issued;
    if (++p_j >= p_ti.L_max) {
      p_j = 0;
      do {
        p_tile += G;
        if (p_tile < NT) p_ti = tile_info(p_tile);
      } while (p_tile < NT && p_ti.L_max == 0);
    }
  };
  if (tid == 0) {
    for (int s = 0; s < kPreStages && p_tile < NT; ++s) produce();
  }

  constexpr uint32_t idesc = idesc_f16_f32(128, 128);
  bool ok = true;
  auto fail = [&]() {
    if (ok) {
      ok = false;
      abort_s = 1;
      atomicOr(p.status, kStatusTimeout);
    }
  };

  TopK15 top;
  int64_t g = 0;            // pages consumed
  int64_t mma_issued = 0;
  float v[128];

  for (int t = c; t < NT; t += G) {
    const TileInfo ti = tile_info(t);
    const int rows = ti.nt * H;
    const int n = tid;                                // this thread's query row
    const int pos = ti.ctx + ti.t0 + n / H;
    const int L = (n < rows && pos >= 0) ? (pos >> 7) : -1;

    // query rows -> tensor memory (A operand)
    {
      uint32_t a[64];
      if (n < rows) {
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
      tmem_st_32x32b_x64(tbase + lane_base + 0, a);
      tmem_wait_st();
      tc_fence_before();
    }
    // a request with an unreadable history page gets all -1 rows
    int bad_local = ti.table_bad ? 1 : 0;
    if (!ti.table_bad) {
      const int seq = __ldg(p.seq_lens + ti.r);
      const int hist = seq >= 1 ? (seq - 1) >> 7 : 0;
      for (int jj = tid; jj < hist; jj += kPreThreads) {
        const int ph = __ldg(p.page_table + (int64_t)ti.r * p.pt_stride + jj);
        bad_local |= (ph < 0 || ph >= p.num_blocks);
      }
    }
    const int tile_bad = __syncthreads_or(bad_local);
    if (tid == 0 && tile_bad) atomicOr(p.status, ti.table_bad ? kStatusBadTable : kStatusBadPage);
    top.reset();

    for (int j = 0; j < ti.L_max; ++j, ++g) {
      const int stage = (int)(g % kPreStages);
      if (ok && !abort_s) {
        if (!mbar_wait(smem_u32(&full_bar[stage]), (uint32_t)((g / kPreStages) & 1))) fail();
      }
      uint32_t w[18];
      {
        const uint2* src = reinterpret_cast<const uint2*>(base + PreLayout::kStageOff + stage * kPageBytes + tid * kRowBytes);
#pragma unroll
        for (int i = 0; i < 9; ++i) {
          const uint2 t2 = src[i];
          w[2 * i] = t2.x;
          w[2 * i + 1] = t2.y;
        }
      }
      named_bar_sync(1, kPreThreads);
      if (tid == 0 && p_tile < NT && !abort_s) produce();

      // dequantise token `tid` into row `tid` of the B tile (SW128, K-major)
      {
        uint8_t* bt = base + PreLayout::kBOff + (g & 1) * kBTileBytes;
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
            *reinterpret_cast<uint4*>(bt + (c16 >> 3) * (128 * 128) + sw128_offset(tid, c16 & 7)) =
                make_uint4(o[4 * h], o[4 * h + 1], o[4 * h + 2], o[4 * h + 3]);
          }
        }
      }
      fence_proxy_async_smem();
      if (j > 0) {       // previous page's scores -> registers
        if (ok && !abort_s) {
          if (!mbar_wait(smem_u32(&mma_bar), (uint32_t)((g - 1) & 1))) fail();
        }
        tc_fence_after();
        tmem_ld_row<128>(tbase + lane_base + 128, v);
        tmem_wait_ld();
        tc_fence_before();
      }
      named_bar_sync(1, kPreThreads);
      if (tid == 0 && !abort_s) {
        tc_fence_after();
        const uint32_t bt = sbase + PreLayout::kBOff + (uint32_t)(g & 1) * kBTileBytes;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t bdesc = smem_desc_sw128(bt + (kk >> 2) * (128 * 128) + (kk & 3) * 32);
          mma_f16_tmemA(tbase + 128, tbase + kk * 8, bdesc, idesc, kk > 0 ? 1u : 0u);
        }
        mma_commit(smem_u32(&mma_bar));
        ++mma_issued;
      }
      if (j > 0) {
        float m = v[0];
#pragma unroll
        for (int i = 1; i < 128; ++i) m = fmaxf(m, v[i]);
        m = canon_zero(m);
        if (j - 1 < L) {
          top.insert(m, j - 1);
          if (p.scores_dbg) p.scores_dbg[((int64_t)ti.row0 * H + n) * p.dbg_stride + (j - 1)] = m;
        }
      }
    }
    if (ti.L_max > 0) {   // last page of the tile
      if (ok && !abort_s) {
        if (!mbar_wait(smem_u32(&mma_bar), (uint32_t)((g - 1) & 1))) fail();
      }
      tc_fence_after();
      tmem_ld_row<128>(tbase + lane_base + 128, v);
      tmem_wait_ld();
      tc_fence_before();
      float m = v[0];
#pragma unroll
      for (int i = 1; i < 128; ++i) m = fmaxf(m, v[i]);
      m = canon_zero(m);
      const int jl = ti.L_max - 1;
      if (jl < L) {
        top.insert(m, jl);
        if (p.scores_dbg) p.scores_dbg[((int64_t)ti.row0 * H + n) * p.dbg_stride + jl] = m;
      }
    }
    if (n < rows) write_out_row(p.out + ((int64_t)ti.row0 * H + n) * kTopK, top.id, L, tile_bad != 0);
    named_bar_sync(1, kPreThreads);      // tensor memory Q free for the next tile
  }

  __syncthreads();
  if (tid == 0 && abort_s) {
    for (int64_t k = (issued > kPreStages ? issued - kPreStages : 0); k < issued; ++k)
      mbar_wait(smem_u32(&full_bar[k % kPreStages]), (uint32_t)((k / kPreStages) & 1));
    if (mma_issued > 0) mbar_wait(smem_u32(&mma_bar), (uint32_t)((mma_issued - 1) & 1));
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tbase, kPreTmemCols);
}

template <int H>
static cudaError_t launch_prefill_h(const PrefillParams& p, int grid, cudaStream_t stream) {
  const size_t smem = PreLayout::bytes(p.num_reqs);
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
