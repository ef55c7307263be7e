// topk.cuh -- per-row running top-15 in registers, and the ordering helpers.
//
// Selection rule (vllm.models.minimax_m3.nvidia.indexer_nvfp4, module
// description: 15 score-ranked history pages, local page last): pages ranked
// by score, descending; equal scores rank the lower page id first.  Callers
// feed pages in ascending id order, so "strictly greater" comparisons give
// exactly that total order.
#pragma once
#include <cstdint>
#include <math_constants.h>

namespace nvfp4idx {

struct TopK15 {
  float s[15];
  int id[15];

  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int i = 0; i < 15; ++i) {
      s[i] = -CUDART_INF_F;
      id[i] = -1;
    }
  }

  // Insert (v, j); j must exceed every id inserted before with the same score.
  // Every entry computes its new value independently: entries scoring >= v
  // stay (equal scores keep the earlier, lower id ahead), the first entry
  // below v takes (v, j), the rest move down one place.
  __device__ __forceinline__ void insert(float v, int j) {
    if (v > s[14]) {
      bool ge[15];
#pragma unroll
      for (int i = 0; i < 15; ++i) ge[i] = s[i] >= v;
#pragma unroll
      for (int i = 14; i > 0; --i) {
        const bool here = !ge[i] && ge[i - 1];
        const float si = ge[i] ? s[i] : (here ? v : s[i - 1]);
        const int ii = ge[i] ? id[i] : (here ? j : id[i - 1]);
        s[i] = si;
        id[i] = ii;
      }
      if (!ge[0]) {
        s[0] = v;
        id[0] = j;
      }
    }
  }

  // Insert (v, j) in any id order: equal scores rank the lower id first
  // (for merging lists that were built over different pages).
  __device__ __forceinline__ void insert_any(float v, int j) {
    if (v > s[14] || (v == s[14] && (id[14] < 0 || j < id[14]))) {
      bool ge[15];
#pragma unroll
      for (int i = 0; i < 15; ++i) ge[i] = s[i] > v || (s[i] == v && id[i] >= 0 && id[i] < j);
#pragma unroll
      for (int i = 14; i > 0; --i) {
        const bool here = !ge[i] && ge[i - 1];
        const float si = ge[i] ? s[i] : (here ? v : s[i - 1]);
        const int ii = ge[i] ? id[i] : (here ? j : id[i - 1]);
        s[i] = si;
        id[i] = ii;
      }
      if (!ge[0]) {
        s[0] = v;
        id[0] = j;
      }
    }
  }
};

// -0.0 -> +0.0 so that equal scores compare equal in the integer key below.
__device__ __forceinline__ float canon_zero(float v) { return v + 0.0f; }

// Monotone map of finite floats (and -inf) to unsigned keys; 0 = "none".
__device__ __forceinline__ uint32_t order_key(float v) {
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_to_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

__device__ __forceinline__ uint32_t warp_max_u32(uint32_t v) {
  uint32_t r;
  asm volatile("redux.sync.max.u32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(v));
  return r;
}
__device__ __forceinline__ uint32_t warp_min_u32(uint32_t v) {
  uint32_t r;
  asm volatile("redux.sync.min.u32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(v));
  return r;
}

// Write one output row: m = min(15, L) ranked ids, then L, then -1.
// L < 0 or `bad` -> all -1.
__device__ __forceinline__ void write_out_row(int32_t* row, const int* ids, int L, bool bad) {
  int v[16];
  const int m = L < 15 ? L : 15;
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    int x = -1;
    if (!bad && L >= 0) {
      if (k < m) x = ids[k];
      else if (k == m) x = L;
    }
    v[k] = x;
  }
  int4* o = reinterpret_cast<int4*>(row);
#pragma unroll
  for (int k = 0; k < 4; ++k) o[k] = make_int4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
}

}  // namespace nvfp4idx
