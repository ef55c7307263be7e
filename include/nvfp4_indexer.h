/*
 * nvfp4_indexer.h -- C ABI of the GB300 (sm_103a) NVFP4 lightning indexer.
 *
 * The indexer selects, for every query token and every index head, the 16
 * pages of the paged KV cache that block-sparse attention will read: the 15
 * history pages whose best token scores highest against the query, then the
 * query's own (local) page, then -1.  Source pages:
 *   vllm.models.minimax_m3.nvidia.indexer_nvfp4 (module description; class
 *   MiniMaxM3IndexerNvfp4Impl, __init__ / forward / _prefill; class
 *   MiniMaxM3IndexerNvfp4MetadataBuilder, build / _build_prefill_chunks) and
 *   vllm.models.minimax_m3.nvidia.indexer_flashinfer (forward; builder build).
 *
 * Fixed configuration (MiniMaxM3IndexerNvfp4Impl.__init__ rejects anything
 * else): 128-token pages, index head dim 128, top-k 16, init_blocks 0,
 * local_blocks 1, "max" scoring.
 *
 * Data formats (indexer_nvfp4, module description):
 *   kv_pages  uint8 [num_blocks][128 tokens][72 B]; per token 64 B of E2M1
 *             codes (element e in byte e/2, low nibble for even e) then 8 E4M3
 *             scales, scale j for elements 16j..16j+15; no global scale.
 *   q         E4M3 bytes [rows][H][128], row-major.
 *   out       int32 [rows][H][16] logical page ids: up to 15 history pages by
 *             score (descending; equal scores: lower id first), the local page
 *             pos/128, then -1.  A row whose position is negative (a padding
 *             request) is all -1.
 *   page_table int32 [num_reqs][pt_stride] logical -> physical page.
 *   seq_lens  int32 [num_reqs], every token of the request including the
 *             queries; queries sit at the last positions (right-aligned).
 *
 * Conventions for every call:
 *   - All array arguments are DEVICE pointers unless stated; the caller owns
 *     them.  Calls never allocate, never synchronise the stream (except
 *     indexer_get_status) and read seq_lens / page_table / cu_seqlens_q in
 *     place, so indexer_decode can be captured in a CUDA graph.
 *   - kv_pages and q must be 16-byte aligned; out 16-byte aligned.
 *   - Arguments are checked on the host before any launch; a bad argument
 *     returns IDX_EINVAL / IDX_EUNSUPPORTED and launches nothing.  The text of
 *     the last error of the calling thread is in indexer_last_error().
 *   - Device-side bad data (a page id outside [0, num_blocks), a history that
 *     does not fit pt_stride) never traps: the affected request's rows are
 *     written as -1 and the plan's status word records it (indexer_get_status).
 *   - A CUDA launch error returns IDX_ECUDA.
 */
#ifndef NVFP4_INDEXER_H
#define NVFP4_INDEXER_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  IDX_OK = 0,
  IDX_EINVAL = -1,         /* bad pointer, size, alignment or stride           */
  IDX_EUNSUPPORTED = -2,   /* head count or query length outside the kernels   */
  IDX_ECUDA = -3,          /* CUDA runtime error                              */
  IDX_ENOSPACE = -4,       /* call exceeds the sizes the plan was made for     */
  IDX_EDEVICE = -5         /* a device-side check fired (indexer_get_status)   */
};

/* Status bits of the device status word. */
enum {
  IDX_STATUS_BAD_PAGE = 1,     /* a page id outside the cache; rows set to -1  */
  IDX_STATUS_BAD_TABLE = 2,    /* history wider than pt_stride; rows set to -1 */
  IDX_STATUS_TIMEOUT = 4,      /* a bounded wait gave up; unfinished rows -1   */
  IDX_STATUS_BAD_SLOT = 8,     /* an insert skipped a slot past the cache       */
  IDX_STATUS_BAD_POSITION = 16 /* nvfp4_insert_norm_rope skipped a token whose
                                  position lies outside the cos/sin table       */
};

/* Page formats (indexer_decode_partial). */
enum {
  IDX_PAGES_NVFP4 = 0,         /* [num_blocks][128][72]                         */
  IDX_PAGES_MXFP4 = 1          /* [num_blocks][8704]                            */
};

typedef struct indexer_plan_s* indexer_plan_t;

/*
 * indexer_plan -- create a plan on the current CUDA device.
 * Owns the device scratch of the decode split-merge (per-split top-15
 * candidates, per-request bookkeeping), that of the prefill split-merge (two
 * candidate slots per SM for the work units that straddle two CTAs: about
 * 9 MB on a 152-SM GPU) and the status word; sized here and never resized.  Mirrors MiniMaxM3IndexerNvfp4MetadataBuilder.__init__,
 * which sizes one decode score buffer for the largest batch and context.
 *   num_heads          index heads H; one of 1, 2, 4, 8 (the builder's
 *                      DECODE_NUM_HEADS check; read here as {1,2,4,8})
 *   max_reqs           largest num_reqs of any indexer_decode call
 *   max_query_len      largest decode query_len, 1..8 (the builder rejects
 *                      more than 8 decode queries per request)
 *   max_pages_per_req  largest page-table width a call may pass as pt_stride
 *   max_prefill_tokens largest total_q of any indexer_prefill call
 *   max_prefill_reqs   largest num_reqs of any indexer_prefill call, at most 4096
 * Returns IDX_OK and *plan, or an error (nothing allocated).
 */
int indexer_plan(indexer_plan_t* plan, int num_heads, int max_reqs, int max_query_len,
                 int max_pages_per_req, int max_prefill_tokens, int max_prefill_reqs);

/* Free the plan's device memory.  The caller must not have work using the
 * plan in flight.  NULL is accepted. */
int indexer_plan_destroy(indexer_plan_t plan);

/*
 * indexer_plan_set_wait_limit -- wall-time limit of every bounded wait
 * inside the decode and prefill kernels run with this plan (no counterpart
 * in the pages: failure detection of this library).  Each wait between the
 * kernels' roles (copy landed, operands ready, accumulator free) gives up
 * after wait_ns nanoseconds; the kernel then sets IDX_STATUS_TIMEOUT in the
 * plan's status word, stops issuing work, waits (bounded, 2 s) for its own
 * copies and tensor-core work in flight, frees its tensor memory and
 * returns; the rows whose scores it could not finish are written as -1
 * (decode and prefill alike), the others are exact.  wait_ns = 0 restores
 * the default of 2 s.  Applies to calls queued after it; the plan's other
 * state is unchanged.  IDX_EINVAL for a NULL plan.
 */
int indexer_plan_set_wait_limit(indexer_plan_t plan, uint64_t wait_ns);

/*
 * indexer_decode -- top-k pages for uniform decode batches
 * (MiniMaxM3IndexerNvfp4Impl.forward, decode branch; the Q8KV4 indexer reads
 * the 1..8 queries of each request in place and writes straight to out).
 *   q          E4M3 [num_reqs * query_len][H][128]; row r*query_len+i is query
 *              i of request r, at position seq_lens[r] - query_len + i
 *   kv_pages   [num_blocks][128][72]
 *   page_table [num_reqs][pt_stride], pt_stride <= plan max_pages_per_req
 *   seq_lens   [num_reqs]; a request with seq_lens < query_len pads a graph
 *              batch, its rows with negative position are all -1
 *   num_reqs   1..plan max_reqs (host scalar, fixed in a captured graph)
 *   query_len  1..plan max_query_len
 *   out        int32 [num_reqs * query_len][H][16]
 *   scores_dbg NULL, or fp32 [num_reqs * query_len][H][dbg_stride]: page
 *              scores of every history page j < pos/128 of the row (other
 *              entries untouched); dbg_stride >= pt_stride
 *   stream     the stream all work is queued on
 * Work: each history page is read from HBM once for all queries and heads of
 * its request, scored on the tensor cores, top-15 kept per row; requests
 * split across CTAs are merged by a second small kernel.
 */
int indexer_decode(indexer_plan_t plan, const uint8_t* q, const uint8_t* kv_pages, int num_blocks,
                   const int32_t* page_table, int pt_stride, const int32_t* seq_lens,
                   int num_reqs, int query_len, int32_t* out, float* scores_dbg, int dbg_stride,
                   cudaStream_t stream);

/*
 * indexer_prefill -- top-k pages for ragged prefill rows (MiniMaxM3Indexer-
 * Nvfp4Impl._prefill; per-token causal clamp = pos/128 + 1 valid pages, as
 * the flashinfer builder's num_valid_pages).  Scores the NVFP4 pages
 * directly (exact fp16 dequantisation in shared memory), without the pages'
 * FP8 gather workspace.
 *   q            E4M3 [total_q][H][128]
 *   cu_seqlens_q int32 [num_reqs + 1], cu[0] = 0, cu[num_reqs] = total_q;
 *                request r owns rows cu[r] .. cu[r+1]-1 at positions
 *                seq_lens[r] - (cu[r+1]-cu[r]) + i (context first)
 *   num_reqs     1..plan max_prefill_reqs;  total_q <= plan max_prefill_tokens
 *   max_seqlen_q host upper bound of cu[r+1]-cu[r]: checked to lie in
 *                0..total_q, otherwise advisory (the grid is one CTA per
 *                SM and the split of the work is computed on the device
 *                from cu_seqlens_q, so a captured graph stays valid)
 *   out          int32 [total_q][H][16] (pass decode out + num_decode_rows*H*16
 *                for a mixed step; decode rows come first, as in forward)
 *   scores_dbg   NULL, or fp32 [total_q][H][dbg_stride], dbg_stride >= pt_stride
 */
int indexer_prefill(indexer_plan_t plan, const uint8_t* q, const int32_t* cu_seqlens_q,
                    int num_reqs, int total_q, int max_seqlen_q, const uint8_t* kv_pages,
                    int num_blocks, const int32_t* page_table, int pt_stride,
                    const int32_t* seq_lens, int32_t* out, float* scores_dbg, int dbg_stride,
                    cudaStream_t stream);

/*
 * nvfp4_insert -- quantise bf16 index keys and write them into the pages
 * (the quantise-and-scatter half of the fused qk-norm/rope insert named in
 * the indexer_nvfp4 module description).  Per token and 16-element group:
 * scale byte = E4M3 round-to-nearest-even of amax/6 (saturating at 448);
 * code = E2M1 round-to-nearest-even of x/scale (saturating at 6, sign kept,
 * sign-only zero codes when the scale is 0).
 *   k_bf16       [n][128] bf16 bit patterns, 16-byte aligned
 *   slot_mapping int64 [n]: page * 128 + row; negative = skip
 *   n            tokens (0 is a no-op)
 *   kv_pages     [num_blocks][128][72]
 *   status       NULL, or a device int32 that gets IDX_STATUS_BAD_SLOT OR-ed
 *                in when a slot >= num_blocks*128 was skipped
 */
int nvfp4_insert(const uint16_t* k_bf16, const int64_t* slot_mapping, int n, uint8_t* kv_pages,
                 int num_blocks, int32_t* status, cudaStream_t stream);

/*
 * nvfp4_insert_norm_rope -- the fused insert that writes the index-K cache
 * (page vllm.models.minimax_m3.nvidia.indexer_nvfp4, module description:
 * "the fused qk-norm/rope insert"; the pages give no more, so this follows
 * vLLM's RMSNorm and rotary-embedding conventions).  Per token:
 *   y = x / sqrt(mean(x^2) + eps) * norm_weight            (RMSNorm, fp32)
 *   rotary pairs (y1, y2) -> (y1 cos - y2 sin, y2 cos + y1 sin), angles from
 *   row `position` of cos_sin_cache; elements past rotary_dim pass through;
 *   the result rounded to bf16, then quantised and written as nvfp4_insert.
 * fp32 order of this kernel: per 16-element group g, running sums e_g and
 * o_g of the even and odd elements' squares (one fused multiply-add per
 * step), t_g = e_g + o_g, ss = ((t0 + t1) + (t2 + t3)) + ((t4 + t5) +
 * (t6 + t7)); v = ss / 128 + eps; rs = 1 / sqrt(v), square root and
 * division correctly rounded; y = (x * rs) * w; every rotation product and
 * sum rounded separately (no fused multiply-add).  The bf16 keys are
 * therefore those of the exact RMSNorm + RoPE up to that fp32 error (an
 * element whose exact value lies that close to a bf16 rounding boundary
 * may round to the other neighbour).
 *   k_bf16         [n][128] bf16 bit patterns, 16-byte aligned (32-byte
 *                  aligned keys are read in 32-byte loads: the faster path)
 *   positions      int64 [n] (unused, may be NULL, when rotary_dim == 0)
 *   slot_mapping   int64 [n]: page * 128 + row; negative = skip
 *   norm_weight    bf16 [128], 16-byte aligned
 *   eps            finite, >= 0 (an all-zero key needs eps > 0)
 *   cos_sin_cache  fp32 [max_pos][rotary_dim]: rotary_dim/2 cosines, then
 *                  rotary_dim/2 sines (16-byte aligned for NeoX or when
 *                  rotary_dim % 8 == 0, else 4)
 *   rotary_dim     even, 0..128; 0 = norm only
 *   is_neox        non-zero: pairs (i, i + rotary_dim/2), rotary_dim 64 or
 *                  128 (others IDX_EUNSUPPORTED); zero: pairs (2i, 2i+1)
 *   kv_pages       [num_blocks][128][72]
 *   status         NULL, or a device int32 that gets IDX_STATUS_BAD_SLOT or
 *                  IDX_STATUS_BAD_POSITION OR-ed in for a skipped token
 */
int nvfp4_insert_norm_rope(const uint16_t* k_bf16, const int64_t* positions, const int64_t* slot_mapping,
                           int n, const uint16_t* norm_weight, float eps, const float* cos_sin_cache,
                           int max_pos, int rotary_dim, int is_neox, uint8_t* kv_pages, int num_blocks,
                           int32_t* status, cudaStream_t stream);

/*
 * MXFP4 index-K pages (page vllm.models.minimax_m3.amd.indexer_mxfp4: its
 * scorers read "e2m1 / e8m0 pages" [pages, 8704] uint8 and feed the same
 * top-k as indexer_nvfp4).  Layout, as this library reads the page's
 * mxfp4_page_views split: bytes 0..8191 hold the E2M1 codes of tokens
 * 0..127 in order (64 bytes per token, element e in byte e/2, low nibble for
 * even e); bytes 8192..8703 hold 4 E8M0 scales per token in token order,
 * scale j covering elements 32j..32j+31; value = code * 2^(scale - 127),
 * scale 0xFF = NaN.  The scorers compute the same scores, selection and
 * output as their NVFP4 counterparts; the pages are dequantised exactly to
 * bf16 (an E8M0 scale can leave fp16's range), queries are widened to bf16.
 */

/*
 * mxfp4_insert -- quantise bf16 index keys into MXFP4 pages.  Per token and
 * 32-element block (the OCP Microscaling Formats v1.0 conversion): shared
 * exponent E = floor(log2(amax)) - 2, clamped to [-127, 127] (amax = 0 gives
 * -127), scale byte = E + 127; code = E2M1 round-to-nearest-even of
 * x / 2^E, saturating at 6, sign kept.
 *   k_bf16       [n][128] bf16 bit patterns, 16-byte aligned
 *   slot_mapping int64 [n]: page * 128 + row; negative = skip
 *   n            tokens (0 is a no-op)
 *   pages        [num_blocks][8704], 16-byte aligned
 *   status       NULL, or a device int32 that gets IDX_STATUS_BAD_SLOT OR-ed
 *                in when a slot >= num_blocks*128 was skipped
 */
int mxfp4_insert(const uint16_t* k_bf16, const int64_t* slot_mapping, int n, uint8_t* pages,
                 int num_blocks, int32_t* status, cudaStream_t stream);

/*
 * indexer_decode_mxfp4 -- indexer_decode over MXFP4 pages [num_blocks][8704];
 * every other argument, the output and the errors as indexer_decode.
 */
int indexer_decode_mxfp4(indexer_plan_t plan, const uint8_t* q, const uint8_t* pages, int num_blocks,
                         const int32_t* page_table, int pt_stride, const int32_t* seq_lens,
                         int num_reqs, int query_len, int32_t* out, float* scores_dbg, int dbg_stride,
                         cudaStream_t stream);

/*
 * indexer_prefill_mxfp4 -- indexer_prefill over MXFP4 pages [num_blocks][8704];
 * every other argument, the output and the errors as indexer_prefill.
 */
int indexer_prefill_mxfp4(indexer_plan_t plan, const uint8_t* q, const int32_t* cu_seqlens_q,
                          int num_reqs, int total_q, int max_seqlen_q, const uint8_t* pages,
                          int num_blocks, const int32_t* page_table, int pt_stride,
                          const int32_t* seq_lens, int32_t* out, float* scores_dbg, int dbg_stride,
                          cudaStream_t stream);

/*
 * Decode context parallelism (page vllm.models.minimax_m3.nvidia.indexer_nvfp4:
 * the per-layer decode-CP buffers and decode_cp.forward, which the indexer
 * uses when the decode batch's history is spread over ranks).  Each rank holds
 * a share of every request's history pages, scores only those, and keeps each
 * row's 15 best (score, logical page id); one all-gather of 15 x 8 bytes per
 * (row, head) and a merge under the same order (score descending, page id
 * ascending) give exactly the rows indexer_decode computes over the whole
 * history.  This library reads the split as a contiguous page range per
 * request and rank (the pages do not show it).
 *
 * indexer_decode_partial -- one rank's share of a decode batch.
 *   page_format  IDX_PAGES_NVFP4 or IDX_PAGES_MXFP4 (the layout of `pages`)
 *   page_lo, page_hi  int32 [num_reqs]: the logical history pages this rank
 *                scores for request r are [page_lo[r], page_hi[r]) cut to the
 *                request's history; page_table[r][j] must map each such j to
 *                this rank's `pages`
 *   cand_out     float [num_reqs * query_len][H][15][2], 16-byte aligned:
 *                (score, page id as int32 bits) pairs sorted by score
 *                descending, page id ascending; id -1 = no candidate, id -2 in
 *                entry 0 = the request has an unreadable page in this share
 *   other arguments as indexer_decode (no scores_dbg); rows are not written.
 */
int indexer_decode_partial(indexer_plan_t plan, int page_format, const uint8_t* q, const uint8_t* pages,
                           int num_blocks, const int32_t* page_table, int pt_stride, const int32_t* seq_lens,
                           const int32_t* page_lo, const int32_t* page_hi, int num_reqs, int query_len,
                           float* cand_out, cudaStream_t stream);

/*
 * indexer_merge_candidates -- the final rows from `world` ranks' candidates.
 *   cand_all   float [world][num_reqs * query_len][num_heads][15][2], rank
 *              major (as an all-gather of every rank's cand_out lays them out),
 *              16-byte aligned; the ranks' page ranges must be disjoint
 *   seq_lens   int32 [num_reqs], as given to indexer_decode_partial
 *   out        int32 [num_reqs * query_len][num_heads][16]: the 15 best
 *              history pages over all ranks, the local page, then -1; all -1
 *              for a row with negative position or an unreadable page
 *   status     NULL, or a device int32 that gets IDX_STATUS_BAD_PAGE OR-ed in
 *              when a rank marked a request unreadable
 */
int indexer_merge_candidates(const float* cand_all, int world, int num_reqs, int query_len, int num_heads,
                             const int32_t* seq_lens, int32_t* out, int32_t* status, cudaStream_t stream);

/*
 * indexer_decode_noalloc -- indexer_decode for callers that cannot allocate
 * device memory.  (No counterpart in the source pages: an addition of this
 * library.)
 * Creating a plan calls cudaMalloc.  Some callers cannot do that: a custom-op
 * hook inside a serving engine that is handed only its input and output
 * buffers while the engine owns all device memory, or a latency-critical loop
 * that must never call cudaMalloc, which can synchronise the device.  This
 * call takes no plan and allocates nothing; it runs the same kernels as
 * indexer_decode with their scratch in a fixed 4 MiB array compiled into the
 * library (held on every device that loads the library until the process
 * exits).
 *   Arguments as indexer_decode, plus
 *   num_heads  H, one of 1, 2, 4, 8
 *   status     NULL, or a device int32 that gets IDX_STATUS_* bits OR-ed in
 *   (no scores_dbg output)
 * Limit: with R = query_len*num_heads, the call needs 256-byte-aligned
 * pieces of roughly 8*num_reqs + (U + num_reqs) * (4 + 120*R) bytes, where
 * U = SMs, or 16*SMs for R <= 8 (the small-row kernel splits the pages over
 * warps, not CTAs); a call that needs more than 4 MiB returns IDX_ENOSPACE
 * and launches nothing (about 390 requests at R = 64 on a 152-SM GPU).
 * The first call on a device looks up the array's device address with
 * cudaGetSymbolAddress (once per device, that device current) and checks
 * that the device is sm_103 (else IDX_EUNSUPPORTED): make that first call
 * before any stream capture.  The address is cached for the life of the
 * process; after cudaDeviceReset on a device, do not call this entry point
 * on it again.  All calls share the array, so calls whose kernels overlap
 * on the GPU race and must be serialised by the caller.  If a wait inside
 * the kernels runs out (2 s without progress), the affected rows are -1 and
 * IDX_STATUS_TIMEOUT goes to *status; with status NULL the rows are still
 * -1 but the reason is not reported anywhere.
 */
int indexer_decode_noalloc(const uint8_t* q, const uint8_t* kv_pages, int num_blocks,
                           const int32_t* page_table, int pt_stride, const int32_t* seq_lens,
                           int num_reqs, int query_len, int num_heads, int32_t* out,
                           int32_t* status, cudaStream_t stream);

/*
 * indexer_sparse_attend -- block-sparse attention over the selected pages,
 * the consumer of the [T, H, 16] id buffer (page
 * vllm.models.minimax_m3.nvidia.indexer_nvfp4, MiniMaxM3IndexerNvfp4Impl
 * .forward: the ids go "straight into the shared [T, H, 16] buffer the
 * attend reads"; page vllm.models.minimax_m3.nvidia.indexer_flashinfer,
 * forward: "The attend reads the shared buffer directly").  The pages do not
 * describe the attend; this library reads it as the usual paged sparse
 * attention: per row t and KV head hk (one per index head), query heads
 * hk*G .. hk*G+G-1 attend over the tokens of the pages ids[t][hk][0..15]
 * (-1 skipped; the pages form a set, so an id listed twice counts once)
 * whose position is at most the row's (causal cut inside the local
 * page): o = sum_s softmax_s(scale * q.k_s) v_s, in fp32 (bf16
 * products exact, exp2f on log2e-scaled scores, online softmax page by
 * page); a row with no visible token gets o = 0.
 *   q          bf16 [num_rows][num_kv_heads * q_per_kv][128], 16-byte aligned
 *   k_cache    bf16 [num_blocks][128][num_kv_heads][128] (token-major pages,
 *              logical page j of request r = block page_table[r][j]);
 *              16-byte aligned, and read in 32-byte loads (the faster path)
 *              when 32-byte aligned
 *   v_cache    same layout as k_cache
 *   page_table int32 [num_reqs][pt_stride] (the indexer's table)
 *   row_req    int32 [num_rows]: the request of each row
 *   row_pos    int32 [num_rows]: the position of each row (decode: seq_len
 *              - query_len + i; prefill: seq_len - new tokens + i)
 *   topk_ids   int32 [num_rows][num_kv_heads][16]: indexer output
 *   num_kv_heads 1, 2, 4 or 8; q_per_kv (G) 1, 2, 4 or 8
 *   scale      finite (1/sqrt(128) for the usual scaling)
 *   out        fp32 [num_rows][num_kv_heads * q_per_kv][128]
 *   status     NULL, or a device int32: IDX_STATUS_BAD_TABLE (a request
 *              outside 0..num_reqs-1, an id >= pt_stride) or
 *              IDX_STATUS_BAD_PAGE (a block outside the cache) is OR-ed in
 *              and that (row, head)'s output is all zeros
 * All pointers are device pointers; nothing is allocated; the call does
 * not synchronise.
 */
int indexer_sparse_attend(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache, int num_blocks,
                          const int32_t* page_table, int pt_stride, int num_reqs, const int32_t* row_req,
                          const int32_t* row_pos, const int32_t* topk_ids, int num_rows, int num_kv_heads,
                          int q_per_kv, float scale, float* out, int32_t* status, cudaStream_t stream);

/* Synchronise `stream`, read and clear the plan's device status word.
 * Returns IDX_OK, or IDX_EDEVICE with the IDX_STATUS_* bits in *bits. */
int indexer_get_status(indexer_plan_t plan, cudaStream_t stream, int32_t* bits);

/* Text of the calling thread's last error ("" if none). */
const char* indexer_last_error(void);

/* Library version string. */
const char* indexer_version(void);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4_INDEXER_H */
