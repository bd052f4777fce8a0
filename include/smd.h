/*
 * smd.h -- C ABI of libsmd: sparse MLA decode over a paged latent cache (fp8_ds_mla or
 * bf16 rows), hand-written CUDA for NVIDIA GB300 (sm_103a).
 *
 * One decode step, per query token t (one token per request), computes
 *
 *   1. index conversion: the token's request-local top-k indices and sliding-window
 *      indices become global cache slots through the block table
 *      (vLLM PR #41217 report, "关键源码片段", _convert_req_index_to_global_index_kernel;
 *      page-range guard as in vLLM PR #52212 report, "关键源码片段", cp-gather kernel);
 *   2. row gather + dequantisation of every valid slot into a 512-wide bf16 latent that
 *      serves as both K and V (SGLang PR #26208 report, "关键源码片段",
 *      _gather_dequant_dsv4_kernel and the DSV4 row constants);
 *   3. partial attention: one 512-wide QK dot for all heads, masking of invalid
 *      entries, softmax, PV over the same 512 dims (vLLM PR #52212 report, "实现拆解"
 *      item 1: 512-wide QK dot, 4 x 128 PV accumulators, masked tail, attention sink,
 *      invalid-index semantics);
 *   4. a workload-aware split-K selector, 1..32 splits (same report, "实现拆解" item 2);
 *   5. a log-sum-exp combine of split partials that also adds the per-head sink logit
 *      to the softmax denominator (same report, test symbol _launch_sparse_decode_reduce).
 *
 * Cache formats (smd_dims.cache_format).  Global slot g lives in page g / P at offset
 * g % P, P = block_size.
 *   SMD_CACHE_FP8_DS_MLA (0): a page is P * 584 bytes: first the P data rows of 576
 *     bytes (448 fp8 e4m3 NoPE values, then 64 little-endian bf16 RoPE values), then the
 *     P scale rows of 8 bytes (7 UE8M0 codes, one per 64 NoPE values, then one pad
 *     byte).  Latent element d < 448 is e4m3(byte d) * 2^(code[d/64] - 127); element
 *     448 + r is RoPE value r.
 *   SMD_CACHE_BF16 (1): a page is P * 1024 bytes, one row of 512 little-endian bf16
 *     latent values (NoPE then RoPE) per slot (vLLM PR #41217 report, the bf16-KV decode
 *     path _forward_bf16_kv; the pages print no layout, this is the plainest reading).
 * An element that is not finite once held as bf16 (NaN byte, code 255, non-finite bf16,
 * overflow) is replaced by 0: the cache is never trusted to be NaN-free (vLLM PR #52212
 * report, "实现拆解" item 3).
 *
 * Two scopes.  The top-k entries (the main scope) and the sliding-window entries attend
 * in one softmax.  By default both live in kv_cache under one block table; with
 * smd_decode_opts.swa_kv_cache the window entries live in a second cache of the same
 * format with its own block table, page size and page count (vLLM PR #52212 report,
 * "实现拆解" items 1 and 3: main and SWA scopes over the compressed and window caches).
 *
 * Semantics (float64 definition, up to bf16/fp32 rounding):
 *   s[h,e]  = scale * q[t,h,:] . k_e              over the valid entries e of token t
 *   den[h]  = sum_e exp(s[h,e]) + exp(sink[h])      (sink term absent if sink == NULL)
 *   out[t,h,:] = sum_e exp(s[h,e]) k_e / den[h]     (0 when den has no terms)
 *   lse[t,h]   = ln den[h]                           (-inf when den has no terms)
 * Entries count once per occurrence (no de-duplication across or within scopes).
 *
 * Conventions for every call:
 *   - All pointers except the dims structs and host outputs are DEVICE pointers of the
 *     current CUDA device; the caller owns every buffer.  Only smd_read_status
 *     synchronises; every other call is asynchronous on `stream` (NULL = legacy stream).
 *   - q, out, kv_cache, kv_out, o_part and workspace must be 16-byte aligned.
 *   - Bad argument VALUES of the inputs (indices -1 or out of range, block-table entries
 *     -1 or out of range, request ids out of range) are masked, never errors.
 *   - Errors: SMD_ERR_INVALID_ARG for bad shapes/pointers (nothing is launched),
 *     SMD_ERR_WORKSPACE for a too-small workspace, SMD_ERR_UNSUPPORTED for a shape the
 *     kernels do not cover, SMD_ERR_CUDA when a launch fails.  smd_last_error() then
 *     returns a message (thread-local, valid until the next call on this thread).
 */
#ifndef SMD_H_
#define SMD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SMD_API __attribute__((visibility("default")))

/* Same type as cudaStream_t. */
typedef struct CUstream_st *smd_stream_t;

enum {
  SMD_OK = 0,
  SMD_ERR_INVALID_ARG = -1,
  SMD_ERR_UNSUPPORTED = -2,
  SMD_ERR_WORKSPACE = -3,
  SMD_ERR_CUDA = -4,
  SMD_ERR_TIMEOUT = -5,
  SMD_ERR_DEVICE_CHECK = -6
};

enum { SMD_CACHE_FP8_DS_MLA = 0, SMD_CACHE_BF16 = 1 };

#define SMD_LATENT_DIM 512
#define SMD_ROW_BYTES 584      /* fp8_ds_mla bytes per slot */
#define SMD_ROW_BYTES_BF16 1024
#define SMD_MAX_HEADS 128
#define SMD_MAX_SPLITS 32

/* Shapes shared by the calls.  Counts are elements; strides are elements between rows. */
typedef struct smd_dims {
  int32_t num_tokens;          /* T in [0, 65535]: query tokens (one per request)       */
  int32_t num_heads;           /* H in [1, 128]: query heads; one shared latent KV head  */
  int32_t num_requests;        /* R >= 1: rows of block_table                           */
  int32_t max_blocks_per_req;  /* >= 1: valid columns of block_table                    */
  int64_t num_pages;           /* >= 1: pages in kv_cache; num_pages*block_size < 2^31   */
  int32_t block_size;          /* P >= 1: slots per page (64 for the DSV4 cache)         */
  int32_t topk;                /* K >= 0: top-k entries per token                       */
  int32_t swa;                 /* W >= 0: sliding-window entries per token              */
  int32_t cache_format;        /* SMD_CACHE_FP8_DS_MLA (0) or SMD_CACHE_BF16 (1)         */
  int64_t bt_stride;           /* >= max_blocks_per_req: block_table row stride         */
  int64_t topk_stride;         /* >= topk: topk_idx row stride                          */
  int64_t swa_stride;          /* >= swa: swa_idx row stride                            */
} smd_dims;

/*
 * Optional parts of a decode step (a NULL smd_decode_opts* means all off).  A zeroed
 * struct is "all off" too.
 *   swa_kv_cache     the window scope's own cache (format dims->cache_format), or NULL:
 *                    the window entries then use kv_cache, block_table and dims' P
 *   swa_block_table  i32 [R, swa_bt_stride]: its block table.  The decode takes both or
 *                    neither; the conversion reads only the block table (and the window
 *                    paging fields), the attention only the cache (swa_num_pages,
 *                    swa_block_size)
 *   swa_num_pages, swa_block_size, swa_max_blocks_per_req, swa_bt_stride: as in smd_dims,
 *                    for the window cache (num_pages * block_size < 2^31)
 *   topk_length      i32 [T] or NULL: top-k column k of token t is masked when
 *                    k >= topk_length[t] (SGLang PR #26208 report, "关键源码片段",
 *                    _gather_dequant_dsv4_kernel's HAS_TOPK_LENGTH branch; one query
 *                    token per sequence)
 *   compact          nonzero: the conversion packs each token's valid slots to the front
 *                    of its row and writes per-token counts, and the attention reads no
 *                    masked row (vLLM PR #41217 report, "实现拆解" item 2: sparse lengths
 *                    built before the decode).  Same results; fewer rows gathered when
 *                    many entries are masked.
 */
typedef struct smd_decode_opts {
  const uint8_t *swa_kv_cache;
  const int32_t *swa_block_table;
  int64_t swa_num_pages;
  int64_t swa_bt_stride;
  int32_t swa_block_size;
  int32_t swa_max_blocks_per_req;
  const int32_t *topk_length;
  int32_t compact;
  int32_t reserved_;           /* set to 0 */
} smd_decode_opts;

/*
 * Split selector (host only, no device call unless num_sms <= 0).  Returns the number of
 * split-K parts S the decode will use, or a negative status.  num_splits: 0 = automatic
 * with cap 32; n > 0 = automatic with cap n; n < 0 = exactly -n (1..32).  The automatic
 * choice depends only on the shapes and num_sms, so a captured CUDA graph stays valid:
 * the S in 1..cap that minimises waves x (tiles per split + 4) + (S > 1 ? 2 : 0), with
 * 64-row tiles, waves = ceil(T x S x ceil(H / 64) / num_sms) (one CTA per token, split and
 * group of 64 heads, one CTA per SM) and 4 and 2 the fixed cost of a work item and of the
 * combine in tiles; every split keeps >= 1 tile (vLLM PR #52212 report, "实现拆解" item 2:
 * an occupancy target, low-batch long context up to 32 splits; that selector's cap of 4
 * for short work is not kept: here a work item's fixed cost outweighs the combine, so
 * short steps gain from more splits).  num_sms <= 0 means "the current device's SM
 * count".
 */
SMD_API int smd_select_num_splits(const smd_dims *dims, int num_splits, int num_sms);

/*
 * Device workspace bytes smd_sparse_mla_decode(_ex) needs for the given split request
 * (same num_splits/num_sms meaning as smd_select_num_splits): a 256-byte status word,
 * the converted indices [T, K+W] int32, the per-token counts [T, 2] int32 and, when
 * S > 1, the split partials o_part f32 [T, S, H, 512] and lse_part f32 [T, S, H], each
 * 256-byte aligned.  Returns 0 on bad dims.
 */
SMD_API size_t smd_workspace_size(const smd_dims *dims, int num_splits, int num_sms);

/*
 * The whole decode step (conversion, fused gather + dequant + tcgen05 attention, and
 * the LSE combine when S > 1).
 *   q           bf16 [T, H, 512], row-major, the latent order [NoPE 448 | RoPE 64]
 *   kv_cache    u8   [num_pages, block_size * row bytes] (format above)
 *   block_table i32  [R, bt_stride]: page of block b of request r, -1 = unused
 *   req_id      i32  [T]: request of token t
 *   topk_idx    i32  [T, topk_stride] request-local positions, -1 = none (NULL iff K=0)
 *   swa_idx     i32  [T, swa_stride]  request-local positions, -1 = none (NULL iff W=0)
 *   sink        f32  [H] per-head sink logits in the scaled-score domain, or NULL
 *   scale       softmax scale applied to q . k (e.g. 1/sqrt(512))
 *   out         bf16 [T, H, 512] (written)
 *   lse         f32  [T, H] natural-log denominator including the sink, or NULL
 *   num_splits  split request, as for smd_select_num_splits
 *   workspace   >= smd_workspace_size(dims, num_splits, device SMs) bytes, 16-B aligned;
 *               its first 4 bytes are a device status word (0 = ok) that the call
 *               resets and that a kernel sets if one of its bounded waits gives up
 */
SMD_API int smd_sparse_mla_decode(const smd_dims *dims, const void *q, const uint8_t *kv_cache,
                                  const int32_t *block_table, const int32_t *req_id,
                                  const int32_t *topk_idx, const int32_t *swa_idx,
                                  const float *sink, float scale, void *out, float *lse,
                                  int num_splits, void *workspace, size_t workspace_bytes,
                                  smd_stream_t stream);

/* smd_sparse_mla_decode with the optional parts of smd_decode_opts (NULL = none). */
SMD_API int smd_sparse_mla_decode_ex(const smd_dims *dims, const smd_decode_opts *opts, const void *q,
                                     const uint8_t *kv_cache, const int32_t *block_table,
                                     const int32_t *req_id, const int32_t *topk_idx,
                                     const int32_t *swa_idx, const float *sink, float scale, void *out,
                                     float *lse, int num_splits, void *workspace,
                                     size_t workspace_bytes, smd_stream_t stream);

/*
 * Steps 2-4 alone, for already-converted slots: the fused gather + dequant + tcgen05
 * attention kernel over gidx i32 [T, K+W] as written by smd_convert_req_index(_ex)
 * (entries < 0 or beyond their cache are masked).  counts (i32 [T, 2] or NULL) are that
 * conversion's per-token counts: token t then attends to its first counts[t, 1] entries,
 * the first counts[t, 0] of them in the main scope; without counts the first K entries
 * are the main scope and the rest the window scope.  Of opts only the window cache
 * (swa_kv_cache, swa_num_pages, swa_block_size) is read.  The split count S follows
 * num_splits as for smd_select_num_splits (current device's SM count).  S == 1: writes out bf16
 * [T, H, 512] and lse f32 [T, H] (lse may be NULL) with the sink in the denominator.
 * S > 1: writes each split's normalised output o_part f32 [T, S, H, 512] and its
 * sink-free lse_part f32 [T, S, H] (-inf for a split without valid entries), to be
 * merged by smd_lse_combine; out/lse are not touched.  status (optional, device int32)
 * gets bit 0 set if a bounded wait inside the kernel gives up.  dims->topk + dims->swa
 * is the row length of gidx; the index pointers of dims are not used.
 */
SMD_API int smd_sparse_mla_attention(const smd_dims *dims, const smd_decode_opts *opts, const void *q,
                                     const uint8_t *kv_cache, const int32_t *gidx, const int32_t *counts,
                                     const float *sink, float scale, int num_splits, void *out, float *lse,
                                     float *o_part, float *lse_part, int32_t *status, smd_stream_t stream);

/*
 * Step 1 alone: writes gidx i32 [T, K+W] (top-k entries first, window entries at
 * offset K) with the global slot of each valid entry and -1 for every invalid one
 * (index < 0, block outside [0, max_blocks), page outside [0, num_pages), request id
 * outside [0, R)).
 */
SMD_API int smd_convert_req_index(const smd_dims *dims, const int32_t *block_table,
                                  const int32_t *req_id, const int32_t *topk_idx,
                                  const int32_t *swa_idx, int32_t *gidx, smd_stream_t stream);

/*
 * smd_convert_req_index with the options: window entries through opts->swa_block_table
 * and the window paging fields when that table is non-NULL (-1 past swa_num_pages), top-k
 * columns cut at topk_length[t], and with opts->compact
 * each token's valid slots packed to the front of its gidx row in column order (the rest
 * of the row is left as it was) and counts i32 [T, 2] = (valid top-k entries, valid
 * entries) written; counts is required with compact and ignored without it.
 */
SMD_API int smd_convert_req_index_ex(const smd_dims *dims, const smd_decode_opts *opts,
                                     const int32_t *block_table, const int32_t *req_id,
                                     const int32_t *topk_idx, const int32_t *swa_idx, int32_t *gidx,
                                     int32_t *counts, smd_stream_t stream);

/*
 * The pages' ragged conversion (vLLM PR #41217 report, "关键源码片段",
 * _convert_req_index_to_global_index_kernel): token t writes out[cu_seqlens[t] + j] for
 * j in [0, cu_seqlens[t+1] - cu_seqlens[t]) from column j of token_indices
 * i32 [T, ti_stride]: block_table[req_id[t], i / P] * P + i % P, or 0 (the pages' fill)
 * when i < 0 or i / P >= max_blocks_per_req.  Like the pages' kernel it does not check
 * the physical page; a request id outside [0, num_requests) and a position j >= num_cols
 * (past the index array's columns) also give 0.  cu_seqlens i32 [T + 1] is
 * non-decreasing from 0 and out holds cu_seqlens[T] entries.  Only num_tokens,
 * num_requests, max_blocks_per_req, block_size and bt_stride of dims are read.
 */
SMD_API int smd_convert_req_index_ragged(const smd_dims *dims, const int32_t *block_table,
                                         const int32_t *req_id, const int32_t *token_indices,
                                         int32_t num_cols, int64_t ti_stride, const int32_t *cu_seqlens,
                                         int32_t *out, smd_stream_t stream);

/*
 * Step 2 alone (a test and debugging export): for each of num_rows global slots
 * gidx[i] writes the dequantised bf16 latent row kv_out[i, 0:512]; a slot that is
 * negative or >= num_pages * block_size gives a zero row.  Only dims->num_pages,
 * dims->block_size and dims->cache_format are read.
 */
SMD_API int smd_gather_dequant(const smd_dims *dims, const uint8_t *kv_cache, const int32_t *gidx,
                               int64_t num_rows, void *kv_out, smd_stream_t stream);

/*
 * Step 5 alone: merges S split partials per (token, head).  o_part f32 [T, S, H, 512]
 * holds each split's output normalised over its own entries, lse_part f32 [T, S, H]
 * its natural-log denominator without sink (-inf for an empty split; such a split adds
 * nothing, whatever its o_part row holds).  Writes out bf16 [T, H, 512] and, if
 * non-NULL, lse f32 [T, H]; sink may be NULL.  With no finite lse and no sink the output
 * row is 0 and lse is -inf.  Requires 1 <= S <= 32 and 1 <= H; o_part and out 16-byte
 * aligned.
 */
SMD_API int smd_lse_combine(int32_t num_tokens, int32_t num_splits, int32_t num_heads,
                            const float *o_part, const float *lse_part, const float *sink,
                            void *out, float *lse, smd_stream_t stream);

/*
 * Reads the device status word at the start of a decode workspace into *device_status
 * after synchronising `stream`.  Bit 0: a kernel's bounded wait gave up; bit 1: a range
 * check of a library built with SMD_DEBUG failed (that build re-checks the address of
 * every gathered row, index read and output write against the buffer sizes and skips an
 * access that fails).  Returns SMD_ERR_DEVICE_CHECK if bit 1 is set, else SMD_ERR_TIMEOUT
 * if bit 0 is set, SMD_OK otherwise (or SMD_ERR_CUDA if the copy fails).
 */
SMD_API int smd_read_status(const void *workspace, int32_t *device_status, smd_stream_t stream);

/*
 * Allocation-free variant of smd_sparse_mla_decode.  The pages have no counterpart: it
 * exists for callers that cannot allocate device memory -- a serving engine that gave
 * nearly all HBM to its paged KV cache at start-up and forbids further cudaMalloc, a
 * plugin living inside a process whose allocator owns the device, or a latency-critical
 * path that cannot take cudaMalloc's implicit device synchronisation.
 *
 * Same arguments and results as smd_sparse_mla_decode, minus the workspace: the scratch
 * (status word, converted slots, split partials) is a static device array of
 * SMD_STATIC_SCRATCH_BYTES inside the library, which every GPU that loads the library
 * holds until the process exits.  A step whose scratch need (smd_workspace_size) exceeds
 * that size is rejected with SMD_ERR_WORKSPACE and a message; nothing is launched.
 * The call allocates nothing.  Its first call on each device looks up the array's device
 * address (cudaGetSymbolAddress, with that device current); make that first call before
 * any stream capture.  All calls on a device share the one array and it keeps the last
 * call's contents (the call resets the status word itself and overwrites everything else
 * it reads), so calls whose kernels overlap on the GPU -- e.g. on two streams without an
 * ordering between them -- race on the scratch.  Serialise them.  The cached address
 * belongs to the device's primary context: after cudaDeviceReset it is stale, and this
 * call must not be used again in that process.
 */
#define SMD_STATIC_SCRATCH_BYTES (32u << 20)
SMD_API int smd_sparse_mla_decode_static_scratch(const smd_dims *dims, const void *q, const uint8_t *kv_cache,
                                                 const int32_t *block_table, const int32_t *req_id,
                                                 const int32_t *topk_idx, const int32_t *swa_idx,
                                                 const float *sink, float scale, void *out, float *lse,
                                                 int num_splits, smd_stream_t stream);

/*
 * smd_read_status for the static scratch of the current device: the status word of the
 * last smd_sparse_mla_decode_static_scratch call on it, after synchronising `stream`.
 * Returns SMD_ERR_TIMEOUT if a bounded wait gave up, SMD_ERR_INVALID_ARG if no such call
 * was made on this device yet.
 */
SMD_API int smd_read_static_scratch_status(int32_t *device_status, smd_stream_t stream);

/* ------------------------------------------------------------------------------------
 * The indexer step: the choice of each decode token's top-k positions (the topk_idx of
 * the decode calls above).
 *
 * Indexer key cache.  Position s of a request lives in page block_table[req, s / P] at
 * in-page position s % P.  A page of layout 0 holds the P positions' head_dim fp8 e4m3
 * key bytes (P * head_dim bytes), then their P little-endian float32 scales; layout 1
 * holds each position's head_dim bytes followed by its scale.  A key element is
 * e4m3(byte) * scale.  (vLLM PR #52212 report, "关键源码片段", the cp-gather kernel of
 * the indexer cache, which takes a layout switch and separate value and scale pointers;
 * the pages print neither layout, these are the plainest readings.)
 * ------------------------------------------------------------------------------------ */

/*
 * Key gather of a ragged batch (vLLM PR #52212 report, "关键源码片段",
 * _cp_gather_indexer_quant_cache_gfx950_kernel; "实现拆解" item 4: runtime batch count,
 * 64-bit block offsets).  For tid in [0, num_tokens): b = token_to_seq[tid]; the token is
 * skipped (nothing written) unless 0 <= b < num_batches and cu_seqlen[b] <= tid <
 * cu_seqlen[b + 1]; position pos = tid - cu_seqlen[b] reads block_table[b, pos / P]
 * (row stride bt_stride); a block at or past max_blocks or a page outside [0, num_pages)
 * writes scale_out[tid] = 0 and leaves k_out[tid] as it is; otherwise k_out[tid, :] =
 * the position's head_dim key bytes and scale_out[tid] = its scale.
 * cache u8 [num_pages, P * (head_dim + 4)], 16-byte aligned; block_table int32;
 * cu_seqlen int32 [num_batches + 1]; token_to_seq int32 [num_tokens]; k_out u8
 * [num_tokens, head_dim] and scale_out f32 [num_tokens], 4-byte aligned.
 * head_dim: a multiple of 4 in [4, 4096]; layout 0 or 1.
 */
SMD_API int smd_indexer_gather_k(const uint8_t *cache, int64_t num_pages, int32_t block_size, int32_t head_dim,
                                 int32_t layout, const int32_t *block_table, int32_t num_batches,
                                 int32_t max_blocks, int64_t bt_stride, const int32_t *cu_seqlen,
                                 const int32_t *token_to_seq, int32_t num_tokens, uint8_t *k_out, float *scale_out,
                                 smd_stream_t stream);

/* Shape of an indexer logits call. */
typedef struct smd_indexer_dims {
  int32_t num_tokens;          /* T query tokens (one per request, or several sharing one) */
  int32_t num_heads;           /* H indexer heads: 32, 64 or 128 */
  int32_t head_dim;            /* 128 */
  int32_t num_requests;        /* R rows of block_table */
  int32_t max_blocks_per_req;  /* W used columns of block_table */
  int32_t block_size;          /* P positions per page: 8, 16, 32, 64 or 128 */
  int64_t num_pages;
  int64_t bt_stride;           /* row stride of block_table, >= W */
  int32_t max_len;             /* L: logits row length (positions per token) */
  int32_t layout;              /* key cache layout: 0 */
} smd_indexer_dims;

/*
 * fp8 paged MQA logits (vLLM PR #41217 report, "实现拆解" item 6: per-head scores and
 * their weighted sum in one kernel; "关键源码片段", SparseAttnIndexer.forward: per-head
 * weights projected beside the key).  For token t of request r = req_id[t] and position
 * s < min(ctx_lens[t], L):
 *   logits[t, s] = sum_h weights[t, h] * max(0, sum_d e4m3(q[t, h, d]) * k_s[d])
 * (k_s = the position's key, its bytes times its scale; the rectifier is the reading of
 * the per-head stage: a score linear in q would let the heads fold into one vector).  A
 * position at or past the context, of a block at or past W, of a page outside
 * [0, num_pages) or of a request outside [0, R) gets -inf; every entry of the [T, L]
 * row-major logits array is written.
 * q u8 e4m3 [T, H, 128] and cache (layout 0) 16-byte aligned; weights f32 [T, H];
 * logits f32 [T, L] 16-byte aligned; device_status (optional) gets bit 0 if a bounded
 * wait gave up (it is not cleared; zero it before the call).  Tensor cores:
 * tcgen05.mma kind::f8f6f4, one CTA per token and 1 to 8 tiles of 128 positions.
 */
SMD_API int smd_indexer_mqa_logits(const smd_indexer_dims *dims, const uint8_t *q, const float *weights,
                                   const uint8_t *cache, const int32_t *block_table, const int32_t *req_id,
                                   const int32_t *ctx_lens, float *logits, int32_t *device_status,
                                   smd_stream_t stream);

/*
 * Top-k positions per token: topk[t, :] = the k positions s < min(ctx_lens[t], max_len)
 * of the largest finite logits[t, s] (row stride logits_stride >= max_len), those above
 * the k-th largest value first in ascending position, then the lowest positions equal
 * to it; -1 pads a token with fewer than k finite logits.  -inf and NaN are never
 * chosen.  topk int32 [num_tokens, k].  1 <= k <= 2^20.
 */
SMD_API int smd_indexer_topk(const float *logits, int32_t num_tokens, int32_t max_len, int64_t logits_stride,
                             const int32_t *ctx_lens, int32_t k, int32_t *topk, smd_stream_t stream);

/*
 * Test and fault-injection hook (not part of the decode semantics): sets the bound, in
 * nanoseconds of wall time, of every pipeline wait inside the attention kernel for launches
 * made after the call, process-wide; 0 restores the default of 2 s.  Returns the previous
 * bound.  A bound far below a tile's run time makes the waits give up on purpose: the
 * kernel then records bit 0 in its status word, drains the work it has in flight (those
 * waits keep a 2 s bound), frees its tensor memory and returns, so the context stays
 * usable and smd_read_status reports SMD_ERR_TIMEOUT.  Outputs of such a launch are
 * undefined.
 */
SMD_API uint64_t smd_set_wait_limit_ns(uint64_t limit_ns);

/* Message for the last non-OK status returned on this thread ("" if none). */
SMD_API const char *smd_last_error(void);

/* Library version, major * 10000 + minor * 100 + patch. */
SMD_API int smd_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SMD_H_ */
