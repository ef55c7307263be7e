// api.cu -- the C ABI (include/nvfp4_indexer.h): argument checks, the plan
// object and its device scratch, launches on the caller's stream.
#include <cmath>
#include <cstdarg>
#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <string>

#include <cuda_runtime.h>

#include "../../include/nvfp4_indexer.h"
#include "internal.h"

using namespace nvfp4idx;

namespace {

thread_local std::string g_last_error;

int set_err(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int cuda_err(cudaError_t e, const char* what) {
  return set_err(IDX_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool valid_heads(int h) { return h == 1 || h == 2 || h == 4 || h == 8; }

}  // namespace

namespace nvfp4idx {
// Error text for entry points defined in other translation units.
void set_last_error_text(const char* msg) { g_last_error = msg ? msg : ""; }
}  // namespace nvfp4idx

struct indexer_plan_s {
  int device = 0;
  int num_sms = 0;
  int num_heads = 0, max_reqs = 0, max_query_len = 0, max_pages = 0;
  int max_prefill_tokens = 0, max_prefill_reqs = 0;
  int decode_grid = 0;
  uint64_t wait_ns = kWaitLimitNs;   // limit of each bounded wait inside the kernels
  float2* cand = nullptr;      // [(split units + max_reqs) slots][R rows][15]
  int32_t* slot_bad = nullptr; // [16 * decode_grid + max_reqs]
  int2* req_info = nullptr;    // [max_reqs]
  int32_t* status = nullptr;   // 1 word
  float2* pcand = nullptr;     // [2 * num_sms][2][128][15]: prefill units cut by a CTA boundary
  int32_t* pslot = nullptr;    // [2 * num_sms][kPreSlotInts]
};

// One body per entry point family; page_format picks the page codec.
static int decode_impl(const char* fn, int page_format, indexer_plan_t plan, const uint8_t* q,
                       const uint8_t* kv_pages, int num_blocks, const int32_t* page_table, int pt_stride,
                       const int32_t* seq_lens, int num_reqs, int query_len, int32_t* out,
                       float* scores_dbg, int dbg_stride, cudaStream_t stream,
                       const int32_t* page_lo = nullptr, const int32_t* page_hi = nullptr,
                       float* cand_out = nullptr) {
  g_last_error.clear();
  if (!plan) return set_err(IDX_EINVAL, "%s: plan is NULL", fn);
  if (page_format != kPagesNvfp4 && page_format != kPagesMxfp4)
    return set_err(IDX_EUNSUPPORTED, "%s: page_format=%d", fn, page_format);
  if (!q || !kv_pages || !page_table || !seq_lens || (!out && !cand_out))
    return set_err(IDX_EINVAL, "%s: NULL array argument", fn);
  if (cand_out && (!page_lo || !page_hi)) return set_err(IDX_EINVAL, "%s: page_lo / page_hi are NULL", fn);
  if (!aligned16(q) || !aligned16(kv_pages) || (out && !aligned16(out)) || (cand_out && !aligned16(cand_out)))
    return set_err(IDX_EINVAL, "%s: q, kv_pages and out must be 16-byte aligned", fn);
  if (query_len < 1 || query_len > 8)
    return set_err(IDX_EUNSUPPORTED, "%s: query_len=%d, supported 1..8", fn, query_len);
  if (query_len > plan->max_query_len)
    return set_err(IDX_ENOSPACE, "%s: query_len=%d > plan max %d", fn, query_len, plan->max_query_len);
  if (num_reqs < 1 || num_reqs > plan->max_reqs)
    return set_err(IDX_ENOSPACE, "%s: num_reqs=%d outside 1..%d", fn, num_reqs, plan->max_reqs);
  if (num_blocks < 1) return set_err(IDX_EINVAL, "%s: num_blocks=%d", fn, num_blocks);
  if (pt_stride < 1 || pt_stride > plan->max_pages)
    return set_err(IDX_ENOSPACE, "%s: pt_stride=%d outside 1..%d", fn, pt_stride, plan->max_pages);
  if (scores_dbg && dbg_stride < pt_stride)
    return set_err(IDX_EINVAL, "%s: dbg_stride=%d < pt_stride=%d", fn, dbg_stride, pt_stride);
  int dev = -1;
  cudaGetDevice(&dev);
  if (dev != plan->device)
    return set_err(IDX_EINVAL, "%s: current device %d, plan made on %d", fn, dev, plan->device);

  DecodeParams p{};
  p.q = q;
  p.kv = kv_pages;
  p.page_table = page_table;
  p.seq_lens = seq_lens;
  p.out = out;
  p.scores_dbg = scores_dbg;
  p.cand = plan->cand;
  p.slot_bad = plan->slot_bad;
  p.req_info = plan->req_info;
  p.status = plan->status;
  p.num_blocks = num_blocks;
  p.pt_stride = pt_stride;
  p.num_reqs = num_reqs;
  p.qlen = query_len;
  p.H = plan->num_heads;
  p.R = query_len * plan->num_heads;
  p.dbg_stride = dbg_stride;
  p.page_format = page_format;
  p.page_lo = page_lo;
  p.page_hi = page_hi;
  p.cand_out = reinterpret_cast<float2*>(cand_out);
  p.wait_ns = plan->wait_ns;
  cudaError_t e = launch_decode(p, plan->decode_grid, stream);
  if (e != cudaSuccess) return set_err(IDX_ECUDA, "%s: launch: %s", fn, cudaGetErrorString(e));
  return IDX_OK;
}

static int prefill_impl(const char* fn, int page_format, indexer_plan_t plan, const uint8_t* q,
                        const int32_t* cu_seqlens_q, int num_reqs, int total_q, int max_seqlen_q,
                        const uint8_t* kv_pages, int num_blocks, const int32_t* page_table, int pt_stride,
                        const int32_t* seq_lens, int32_t* out, float* scores_dbg, int dbg_stride,
                        cudaStream_t stream) {
  g_last_error.clear();
  if (!plan) return set_err(IDX_EINVAL, "%s: plan is NULL", fn);
  if (!q || !cu_seqlens_q || !kv_pages || !page_table || !seq_lens || !out)
    return set_err(IDX_EINVAL, "%s: NULL array argument", fn);
  if (!aligned16(q) || !aligned16(kv_pages) || !aligned16(out))
    return set_err(IDX_EINVAL, "%s: q, kv_pages and out must be 16-byte aligned", fn);
  if (num_reqs < 1 || num_reqs > plan->max_prefill_reqs)
    return set_err(IDX_ENOSPACE, "%s: num_reqs=%d outside 1..%d", fn, num_reqs, plan->max_prefill_reqs);
  if (total_q < 0 || total_q > plan->max_prefill_tokens)
    return set_err(IDX_ENOSPACE, "%s: total_q=%d outside 0..%d", fn, total_q, plan->max_prefill_tokens);
  if (max_seqlen_q < 0 || max_seqlen_q > total_q)
    return set_err(IDX_EINVAL, "%s: max_seqlen_q=%d outside 0..total_q", fn, max_seqlen_q);
  if (num_blocks < 1) return set_err(IDX_EINVAL, "%s: num_blocks=%d", fn, num_blocks);
  if (pt_stride < 1 || pt_stride > plan->max_pages)
    return set_err(IDX_ENOSPACE, "%s: pt_stride=%d outside 1..%d", fn, pt_stride, plan->max_pages);
  if (scores_dbg && dbg_stride < pt_stride)
    return set_err(IDX_EINVAL, "%s: dbg_stride=%d < pt_stride=%d", fn, dbg_stride, pt_stride);
  int dev = -1;
  cudaGetDevice(&dev);
  if (dev != plan->device)
    return set_err(IDX_EINVAL, "%s: current device %d, plan made on %d", fn, dev, plan->device);
  if (total_q == 0) return IDX_OK;

  PrefillParams p{};
  p.q = q;
  p.kv = kv_pages;
  p.page_table = page_table;
  p.seq_lens = seq_lens;
  p.cu_seqlens_q = cu_seqlens_q;
  p.out = out;
  p.scores_dbg = scores_dbg;
  p.status = plan->status;
  p.num_blocks = num_blocks;
  p.pt_stride = pt_stride;
  p.num_reqs = num_reqs;
  p.total_q = total_q;
  p.H = plan->num_heads;
  p.dbg_stride = dbg_stride;
  p.pcand = plan->pcand;
  p.pslot = plan->pslot;
  const int grid = plan->num_sms;   // one prefill CTA per SM; the work is split evenly by pages
  p.page_format = page_format;
  p.wait_ns = plan->wait_ns;
  cudaError_t e = launch_prefill(p, grid, stream);
  if (e != cudaSuccess) return set_err(IDX_ECUDA, "%s: launch: %s", fn, cudaGetErrorString(e));
  return IDX_OK;
}

static int insert_impl(const char* fn, int page_format, const uint16_t* k_bf16, const int64_t* slot_mapping,
                       int n, uint8_t* kv_pages, int num_blocks, int32_t* status, cudaStream_t stream) {
  g_last_error.clear();
  if (n < 0) return set_err(IDX_EINVAL, "%s: n=%d", fn, n);
  if (n == 0) return IDX_OK;
  if (!k_bf16 || !slot_mapping || !kv_pages)
    return set_err(IDX_EINVAL, "%s: NULL array argument", fn);
  if (!aligned16(k_bf16) || !aligned16(kv_pages) || (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
    return set_err(IDX_EINVAL, "%s: k_bf16 and kv_pages must be 16-byte aligned, slot_mapping 8", fn);
  if (num_blocks < 1) return set_err(IDX_EINVAL, "%s: num_blocks=%d", fn, num_blocks);
  cudaError_t e = page_format == kPagesMxfp4
                      ? launch_insert_mxfp4(k_bf16, slot_mapping, n, kv_pages, num_blocks, status, stream)
                      : launch_insert(k_bf16, slot_mapping, n, kv_pages, num_blocks, status, stream);
  if (e != cudaSuccess) return set_err(IDX_ECUDA, "%s: launch: %s", fn, cudaGetErrorString(e));
  return IDX_OK;
}

extern "C" {

const char* indexer_version(void) { return "nvfp4_indexer 0.1 sm_103a"; }

const char* indexer_last_error(void) { return g_last_error.c_str(); }

int indexer_plan(indexer_plan_t* plan, int num_heads, int max_reqs, int max_query_len,
                 int max_pages_per_req, int max_prefill_tokens, int max_prefill_reqs) {
  g_last_error.clear();
  if (!plan) return set_err(IDX_EINVAL, "indexer_plan: plan is NULL");
  *plan = nullptr;
  if (!valid_heads(num_heads))
    return set_err(IDX_EUNSUPPORTED, "indexer_plan: num_heads=%d, supported 1, 2, 4, 8", num_heads);
  if (max_query_len < 1 || max_query_len > 8)
    return set_err(IDX_EUNSUPPORTED, "indexer_plan: max_query_len=%d, supported 1..8", max_query_len);
  if (max_reqs < 0 || max_reqs > kMaxDecodeReqs)
    return set_err(IDX_EINVAL, "indexer_plan: max_reqs=%d outside 0..%d", max_reqs, kMaxDecodeReqs);
  if (max_pages_per_req < 1 || max_pages_per_req > (1 << 20))
    return set_err(IDX_EINVAL, "indexer_plan: max_pages_per_req=%d outside 1..2^20", max_pages_per_req);
  if (max_prefill_tokens < 0 || max_prefill_reqs < 0 || max_prefill_reqs > kMaxPrefillReqs)
    return set_err(IDX_EINVAL, "indexer_plan: bad prefill limits (%d tokens, %d requests)",
                   max_prefill_tokens, max_prefill_reqs);

  indexer_plan_s* pl = new indexer_plan_s();
  cudaError_t e = cudaGetDevice(&pl->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&pl->num_sms, cudaDevAttrMultiProcessorCount, pl->device);
  if (e != cudaSuccess) {
    delete pl;
    return cuda_err(e, "indexer_plan: device query");
  }
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, pl->device);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, pl->device);
  if (major != 10 || minor != 3) {
    delete pl;
    return set_err(IDX_EUNSUPPORTED, "indexer_plan: device is sm_%d%d, the kernels are built for sm_103a",
                   major, minor);
  }
  pl->num_heads = num_heads;
  pl->max_reqs = max_reqs;
  pl->max_query_len = max_query_len;
  pl->max_pages = max_pages_per_req;
  pl->max_prefill_tokens = max_prefill_tokens;
  pl->max_prefill_reqs = max_prefill_reqs;
  pl->decode_grid = pl->num_sms;   // one decode CTA per SM
  // candidate slots = split units + requests: CTAs of the quad kernel (up to
  // 64 rows each), or warps of the small-row kernel (up to 8 rows each)
  const size_t slots = (size_t)pl->decode_grid + (size_t)max_reqs;
  const size_t bad_slots = (size_t)decode_split_units(1, kPagesNvfp4, pl->decode_grid) + (size_t)max_reqs;
  const size_t cand_rows = std::max(slots * kMaxRows, bad_slots * 8);
  e = cudaMalloc(&pl->cand, cand_rows * kHistK * sizeof(float2));
  if (e == cudaSuccess) e = cudaMalloc(&pl->slot_bad, bad_slots * sizeof(int32_t));
  if (e == cudaSuccess) e = cudaMalloc(&pl->req_info, (size_t)(max_reqs > 0 ? max_reqs : 1) * sizeof(int2));
  if (e == cudaSuccess) e = cudaMalloc(&pl->status, sizeof(int32_t));
  if (e == cudaSuccess) e = cudaMemset(pl->status, 0, sizeof(int32_t));
  if (e == cudaSuccess) e = cudaMemset(pl->slot_bad, 0, bad_slots * sizeof(int32_t));
  if (e == cudaSuccess)
    e = cudaMalloc(&pl->pcand, (size_t)2 * pl->num_sms * 2 * 128 * kHistK * sizeof(float2));
  if (e == cudaSuccess) e = cudaMalloc(&pl->pslot, (size_t)2 * pl->num_sms * kPreSlotInts * sizeof(int32_t));
  if (e != cudaSuccess) {
    indexer_plan_destroy(pl);
    return cuda_err(e, "indexer_plan: allocation");
  }
  *plan = pl;
  return IDX_OK;
}

int indexer_plan_set_wait_limit(indexer_plan_t plan, uint64_t wait_ns) {
  g_last_error.clear();
  if (!plan) return set_err(IDX_EINVAL, "indexer_plan_set_wait_limit: plan is NULL");
  plan->wait_ns = wait_ns ? wait_ns : kWaitLimitNs;
  return IDX_OK;
}

int indexer_plan_destroy(indexer_plan_t plan) {
  if (!plan) return IDX_OK;
  cudaFree(plan->cand);
  cudaFree(plan->slot_bad);
  cudaFree(plan->req_info);
  cudaFree(plan->status);
  cudaFree(plan->pcand);
  cudaFree(plan->pslot);
  delete plan;
  return IDX_OK;
}




int indexer_decode(indexer_plan_t plan, const uint8_t* q, const uint8_t* kv_pages, int num_blocks,
                   const int32_t* page_table, int pt_stride, const int32_t* seq_lens, int num_reqs,
                   int query_len, int32_t* out, float* scores_dbg, int dbg_stride, cudaStream_t stream) {
  return decode_impl("indexer_decode", kPagesNvfp4, plan, q, kv_pages, num_blocks, page_table, pt_stride,
                     seq_lens, num_reqs, query_len, out, scores_dbg, dbg_stride, stream);
}

int indexer_decode_mxfp4(indexer_plan_t plan, const uint8_t* q, const uint8_t* pages, int num_blocks,
                         const int32_t* page_table, int pt_stride, const int32_t* seq_lens, int num_reqs,
                         int query_len, int32_t* out, float* scores_dbg, int dbg_stride,
                         cudaStream_t stream) {
  return decode_impl("indexer_decode_mxfp4", kPagesMxfp4, plan, q, pages, num_blocks, page_table,
                     pt_stride, seq_lens, num_reqs, query_len, out, scores_dbg, dbg_stride, stream);
}

int indexer_decode_partial(indexer_plan_t plan, int page_format, const uint8_t* q, const uint8_t* pages,
                           int num_blocks, const int32_t* page_table, int pt_stride, const int32_t* seq_lens,
                           const int32_t* page_lo, const int32_t* page_hi, int num_reqs, int query_len,
                           float* cand_out, cudaStream_t stream) {
  return decode_impl("indexer_decode_partial", page_format, plan, q, pages, num_blocks, page_table, pt_stride,
                     seq_lens, num_reqs, query_len, nullptr, nullptr, 0, stream, page_lo, page_hi, cand_out);
}

int indexer_merge_candidates(const float* cand_all, int world, int num_reqs, int query_len, int num_heads,
                             const int32_t* seq_lens, int32_t* out, int32_t* status, cudaStream_t stream) {
  g_last_error.clear();
  if (!cand_all || !seq_lens || !out) return set_err(IDX_EINVAL, "indexer_merge_candidates: NULL array argument");
  if (!aligned16(cand_all) || !aligned16(out))
    return set_err(IDX_EINVAL, "indexer_merge_candidates: cand_all and out must be 16-byte aligned");
  if (world < 1) return set_err(IDX_EINVAL, "indexer_merge_candidates: world=%d", world);
  if (!valid_heads(num_heads))
    return set_err(IDX_EUNSUPPORTED, "indexer_merge_candidates: num_heads=%d, supported 1, 2, 4, 8", num_heads);
  if (query_len < 1 || query_len > 8)
    return set_err(IDX_EUNSUPPORTED, "indexer_merge_candidates: query_len=%d, supported 1..8", query_len);
  if (num_reqs < 0) return set_err(IDX_EINVAL, "indexer_merge_candidates: num_reqs=%d", num_reqs);
  cudaError_t e = launch_cp_merge(reinterpret_cast<const float2*>(cand_all), world, num_reqs, query_len,
                                  num_heads, seq_lens, out, status, stream);
  if (e != cudaSuccess) return cuda_err(e, "indexer_merge_candidates: launch");
  return IDX_OK;
}

int indexer_prefill(indexer_plan_t plan, const uint8_t* q, const int32_t* cu_seqlens_q, int num_reqs,
                    int total_q, int max_seqlen_q, const uint8_t* kv_pages, int num_blocks,
                    const int32_t* page_table, int pt_stride, const int32_t* seq_lens, int32_t* out,
                    float* scores_dbg, int dbg_stride, cudaStream_t stream) {
  return prefill_impl("indexer_prefill", kPagesNvfp4, plan, q, cu_seqlens_q, num_reqs, total_q,
                      max_seqlen_q, kv_pages, num_blocks, page_table, pt_stride, seq_lens, out, scores_dbg,
                      dbg_stride, stream);
}

int indexer_prefill_mxfp4(indexer_plan_t plan, const uint8_t* q, const int32_t* cu_seqlens_q, int num_reqs,
                          int total_q, int max_seqlen_q, const uint8_t* pages, int num_blocks,
                          const int32_t* page_table, int pt_stride, const int32_t* seq_lens, int32_t* out,
                          float* scores_dbg, int dbg_stride, cudaStream_t stream) {
  return prefill_impl("indexer_prefill_mxfp4", kPagesMxfp4, plan, q, cu_seqlens_q, num_reqs, total_q,
                      max_seqlen_q, pages, num_blocks, page_table, pt_stride, seq_lens, out, scores_dbg,
                      dbg_stride, stream);
}

int nvfp4_insert(const uint16_t* k_bf16, const int64_t* slot_mapping, int n, uint8_t* kv_pages,
                 int num_blocks, int32_t* status, cudaStream_t stream) {
  return insert_impl("nvfp4_insert", kPagesNvfp4, k_bf16, slot_mapping, n, kv_pages, num_blocks, status,
                     stream);
}

int mxfp4_insert(const uint16_t* k_bf16, const int64_t* slot_mapping, int n, uint8_t* pages,
                 int num_blocks, int32_t* status, cudaStream_t stream) {
  return insert_impl("mxfp4_insert", kPagesMxfp4, k_bf16, slot_mapping, n, pages, num_blocks, status,
                     stream);
}

int nvfp4_insert_norm_rope(const uint16_t* k_bf16, const int64_t* positions, const int64_t* slot_mapping,
                           int n, const uint16_t* norm_weight, float eps, const float* cos_sin_cache,
                           int max_pos, int rotary_dim, int is_neox, uint8_t* kv_pages, int num_blocks,
                           int32_t* status, cudaStream_t stream) {
  g_last_error.clear();
  const char* fn = "nvfp4_insert_norm_rope";
  if (n < 0) return set_err(IDX_EINVAL, "%s: n=%d", fn, n);
  if (rotary_dim < 0 || rotary_dim > 128 || (rotary_dim & 1))
    return set_err(IDX_EINVAL, "%s: rotary_dim=%d (even, 0..128)", fn, rotary_dim);
  if (rotary_dim && is_neox && rotary_dim != 64 && rotary_dim != 128)
    return set_err(IDX_EUNSUPPORTED, "%s: NeoX rotary_dim=%d (64 or 128)", fn, rotary_dim);
  if (!(eps >= 0.0f) || !(eps < INFINITY)) return set_err(IDX_EINVAL, "%s: eps must be finite and >= 0", fn);
  if (n == 0) return IDX_OK;
  if (!k_bf16 || !slot_mapping || !norm_weight || !kv_pages)
    return set_err(IDX_EINVAL, "%s: NULL array argument", fn);
  if (rotary_dim && (!positions || !cos_sin_cache || max_pos < 1))
    return set_err(IDX_EINVAL, "%s: rotary_dim > 0 needs positions, cos_sin_cache and max_pos >= 1", fn);
  if (!aligned16(k_bf16) || !aligned16(norm_weight) || !aligned16(kv_pages) ||
      (reinterpret_cast<uintptr_t>(slot_mapping) & 7u) || (reinterpret_cast<uintptr_t>(positions) & 7u))
    return set_err(IDX_EINVAL, "%s: k_bf16, norm_weight and kv_pages must be 16-byte aligned, "
                               "slot_mapping and positions 8", fn);
  const uintptr_t cs_align = (is_neox || rotary_dim % 8 == 0) ? 16u : 4u;   // vector loads of the rows
  if (rotary_dim && (reinterpret_cast<uintptr_t>(cos_sin_cache) & (cs_align - 1)))
    return set_err(IDX_EINVAL, "%s: cos_sin_cache must be %d-byte aligned", fn, (int)cs_align);
  if (num_blocks < 1) return set_err(IDX_EINVAL, "%s: num_blocks=%d", fn, num_blocks);
  NormRopeArgs a;
  a.k = k_bf16;
  a.positions = positions;
  a.slots = slot_mapping;
  a.n = n;
  a.weight = norm_weight;
  a.eps = eps;
  a.cos_sin = cos_sin_cache;
  a.max_pos = max_pos;
  a.rotary_dim = rotary_dim;
  a.is_neox = is_neox ? 1 : 0;
  a.pages = kv_pages;
  a.num_slots = (int64_t)num_blocks * 128;
  a.status = status;
  cudaError_t e = launch_insert_norm_rope(a, stream);
  if (e != cudaSuccess) return set_err(IDX_ECUDA, "%s: launch: %s", fn, cudaGetErrorString(e));
  return IDX_OK;
}

int indexer_sparse_attend(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache, int num_blocks,
                          const int32_t* page_table, int pt_stride, int num_reqs, const int32_t* row_req,
                          const int32_t* row_pos, const int32_t* topk_ids, int num_rows, int num_kv_heads,
                          int q_per_kv, float scale, float* out, int32_t* status, cudaStream_t stream) {
  g_last_error.clear();
  const char* fn = "indexer_sparse_attend";
  if (num_rows < 0) return set_err(IDX_EINVAL, "%s: num_rows=%d", fn, num_rows);
  if (!valid_heads(num_kv_heads))
    return set_err(IDX_EUNSUPPORTED, "%s: num_kv_heads=%d, supported 1, 2, 4, 8", fn, num_kv_heads);
  if (!(q_per_kv == 1 || q_per_kv == 2 || q_per_kv == 4 || q_per_kv == 8))
    return set_err(IDX_EUNSUPPORTED, "%s: q_per_kv=%d, supported 1, 2, 4, 8", fn, q_per_kv);
  if (!(scale == scale) || scale == INFINITY || scale == -INFINITY)
    return set_err(IDX_EINVAL, "%s: scale must be finite", fn);
  if (num_rows == 0) return IDX_OK;
  if (!q || !k_cache || !v_cache || !page_table || !row_req || !row_pos || !topk_ids || !out)
    return set_err(IDX_EINVAL, "%s: NULL array argument", fn);
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
    return set_err(IDX_EINVAL, "%s: q, k_cache, v_cache and out must be 16-byte aligned", fn);
  if (num_blocks < 1 || pt_stride < 1 || num_reqs < 1)
    return set_err(IDX_EINVAL, "%s: num_blocks=%d pt_stride=%d num_reqs=%d", fn, num_blocks, pt_stride, num_reqs);
  AttendParams p{};
  p.q = q;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.page_table = page_table;
  p.row_req = row_req;
  p.row_pos = row_pos;
  p.ids = topk_ids;
  p.out = out;
  p.status = status;
  p.num_blocks = num_blocks;
  p.pt_stride = pt_stride;
  p.num_reqs = num_reqs;
  p.num_rows = num_rows;
  p.H = num_kv_heads;
  p.G = q_per_kv;
  p.scale = scale;
  cudaError_t e = launch_attend(p, stream);
  if (e != cudaSuccess) return set_err(IDX_ECUDA, "%s: launch: %s", fn, cudaGetErrorString(e));
  return IDX_OK;
}

int indexer_get_status(indexer_plan_t plan, cudaStream_t stream, int32_t* bits) {
  g_last_error.clear();
  if (!plan) return set_err(IDX_EINVAL, "indexer_get_status: plan is NULL");
  int32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, plan->status, sizeof(v), cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(plan->status, 0, sizeof(int32_t), stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_err(e, "indexer_get_status");
  if (bits) *bits = v;
  if (v != 0) return set_err(IDX_EDEVICE, "device status bits 0x%x", v);
  return IDX_OK;
}

}  // extern "C"
