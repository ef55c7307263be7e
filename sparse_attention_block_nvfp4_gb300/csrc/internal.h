// internal.h -- declarations shared by the library's translation units.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace nvfp4idx {

constexpr int kPage = 128;        // tokens per page
constexpr int kDim = 128;         // index head dim
constexpr int kRowBytes = 72;     // 64 B codes + 8 B scales
constexpr int kPageBytes = kPage * kRowBytes;   // 9216
constexpr int kTopK = 16;
constexpr int kHistK = 15;        // score-ranked history pages per row
constexpr int kMaxRows = 64;      // query_len (<= 8) x heads (<= 8) per request
constexpr int kMaxDecodeReqs = 4096;   // per-request prefix sums live in shared memory
constexpr int kMaxPrefillReqs = 4096;
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // default limit of a bounded wait: 2 s

// index-K page formats
constexpr int kPagesNvfp4 = 0;    // [num_blocks, 128, 72]: E2M1 codes + E4M3 scales per 16
constexpr int kPagesMxfp4 = 1;    // [num_blocks, 8704]: E2M1 codes, then E8M0 scales per 32

// device status bits (mirror IDX_STATUS_* in include/nvfp4_indexer.h)
constexpr int32_t kStatusBadPage = 1;
constexpr int32_t kStatusBadTable = 2;
constexpr int32_t kStatusTimeout = 4;
constexpr int32_t kStatusBadSlot = 8;
constexpr int32_t kStatusBadPosition = 16;

struct DecodeParams {
  const uint8_t* q;            // [num_reqs * qlen][H][128] e4m3
  const uint8_t* kv;           // [num_blocks][128][72]
  const int32_t* page_table;   // [num_reqs][pt_stride]
  const int32_t* seq_lens;     // [num_reqs]
  int32_t* out;                // [rows][H][16]
  float* scores_dbg;           // nullable
  float2* cand;                // [(split units + num_reqs) slots][R][15] (score, id bits)
  int32_t* slot_bad;           // [(split units + num_reqs)]
  int2* req_info;              // [num_reqs] (first split unit, number of segments)
  int32_t* status;
  int num_blocks, pt_stride, num_reqs, qlen, H, R, dbg_stride;
  int page_format;             // kPagesNvfp4 / kPagesMxfp4
  // a context-parallel rank's share (indexer_decode_partial): request r
  // scores only its history pages in [page_lo[r], page_hi[r]) (NULL: all)
  // and leaves each row's 15 candidates in cand_out instead of a final row
  const int32_t* page_lo;
  const int32_t* page_hi;
  float2* cand_out;            // [rows][15] (score, id); NULL = final rows in out
  uint64_t wait_ns;            // wall-time limit of each bounded wait
};

struct PrefillParams {
  const uint8_t* q;            // [total_q][H][128]
  const uint8_t* kv;
  const int32_t* page_table;
  const int32_t* seq_lens;
  const int32_t* cu_seqlens_q; // [num_reqs + 1]
  int32_t* out;                // [total_q][H][16]
  float* scores_dbg;
  int32_t* status;
  // units cut by a CTA boundary: slot 2c / 2c + 1 = the first / last unit of
  // CTA c; per slot the candidates [2 tiles][128 rows][15] and the unit's
  // description (kPreSlotInts ints, slot_meta[0] = unit id or -1)
  float2* pcand;
  int32_t* pslot;
  int num_blocks, pt_stride, num_reqs, total_q, H, dbg_stride;
  int page_format;             // kPagesNvfp4 / kPagesMxfp4
  uint64_t wait_ns;            // wall-time limit of each bounded wait
};
constexpr int kPreSlotInts = 21;

// Block-sparse attention over the selected pages (indexer_sparse_attend).
struct AttendParams {
  const uint16_t* q;           // bf16 [num_rows][H * G][128]
  const uint16_t* k_cache;     // bf16 [num_blocks][128][H][128]
  const uint16_t* v_cache;     // bf16 [num_blocks][128][H][128]
  const int32_t* page_table;   // [num_reqs][pt_stride]
  const int32_t* row_req;      // [num_rows] request of each row
  const int32_t* row_pos;      // [num_rows] position of each row
  const int32_t* ids;          // [num_rows][H][16] logical page ids, -1 = none
  float* out;                  // fp32 [num_rows][H * G][128]
  int32_t* status;             // nullable
  int num_blocks, pt_stride, num_reqs, num_rows, H, G;
  float scale;
};
cudaError_t launch_attend(const AttendParams& p, cudaStream_t stream);   // [19 + x]: tile x of the unit failed (a wait ran out)

// Launch `kernel` so that it may be scheduled while the kernel before it on
// the stream is still running (programmatic dependent launch); the kernel
// must call griddep_wait() before reading what its predecessor wrote.
template <typename... Args>
cudaError_t launch_dependent(void (*kernel)(Args...), unsigned grid, unsigned block, size_t smem,
                             cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Error text for entry points defined outside api.cu (read back by
// indexer_last_error()).
void set_last_error_text(const char* msg);

cudaError_t launch_insert(const uint16_t* k, const int64_t* slots, int n, uint8_t* pages,
                          int num_blocks, int32_t* status, cudaStream_t stream);
cudaError_t launch_insert_mxfp4(const uint16_t* k, const int64_t* slots, int n, uint8_t* pages,
                                int num_blocks, int32_t* status, cudaStream_t stream);
// Arguments of the fused qk-norm + RoPE + NVFP4 insert (all device pointers;
// positions and cos_sin unused when rotary_dim == 0).
struct NormRopeArgs {
  const uint16_t* k;          // bf16 [n][128]
  const int64_t* positions;   // [n]
  const int64_t* slots;       // [n], negative = skip
  int n;
  const uint16_t* weight;     // bf16 [128]
  float eps;
  const float* cos_sin;       // [max_pos][rotary_dim]: cosines, then sines
  int64_t max_pos;
  int rotary_dim;
  int is_neox;
  uint8_t* pages;             // [num_blocks][128][72]
  int64_t num_slots;          // num_blocks * 128
  int32_t* status;
};
cudaError_t launch_insert_norm_rope(const NormRopeArgs& a, cudaStream_t stream);
cudaError_t launch_decode(const DecodeParams& p, int grid, cudaStream_t stream);
// Split units of a decode launch of `grid` CTAs (the candidate slots are
// indexed by unit + request): the CTAs, or for requests of up to 8 rows on
// NVFP4 pages the small-row kernel's 16 warps per CTA.
int decode_split_units(int R, int page_format, int grid);
// Merge the candidate lists of `world` context-parallel ranks ([world][rows][15],
// rank-major) into final rows [rows][16].
cudaError_t launch_cp_merge(const float2* cand_all, int world, int num_reqs, int query_len, int H,
                            const int32_t* seq_lens, int32_t* out, int32_t* status, cudaStream_t stream);
cudaError_t launch_prefill(const PrefillParams& p, int grid, cudaStream_t stream);   // + the merge

// smallest power-of-two >= 16 that holds R rows (the MMA N dimension)
inline int decode_nq(int R) { return R <= 16 ? 16 : (R <= 32 ? 32 : 64); }

}  // namespace nvfp4idx
