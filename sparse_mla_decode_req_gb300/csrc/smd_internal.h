// Internal launch interface between the C-ABI layer (smd_api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace smd {

constexpr int kTileRows = 64;     // rows per split unit (one attention tile)
constexpr int kMaxSplits = 32;

// One paged cache of the decode: base, page size and page count (the second one, for the
// window scope, is optional).
struct CacheDesc {
  const uint8_t* base;
  int64_t num_pages;
  int32_t P;
  int32_t log2P;  // log2(P) when P is a power of two, else -1
};
// log2(P) for a power of two, else -1.
inline int32_t log2_if_pow2_host(int32_t P) {
  if (P <= 0 || (P & (P - 1)) != 0) return -1;
  int32_t l = 0;
  while ((1 << l) < P) ++l;
  return l;
}
inline CacheDesc make_cache_desc(const uint8_t* base, int64_t num_pages, int32_t P) {
  return CacheDesc{base, num_pages, P, log2_if_pow2_host(P)};
}

struct ConvertParams {
  const int32_t* block_table;
  const int32_t* req_id;
  const int32_t* topk;
  const int32_t* swa;
  const int32_t* topk_length;  // [T] or null: top-k column k of token t masked when k >= topk_length[t]
  const int32_t* swa_block_table;  // window scope's own block table, or null (the main one)
  int32_t* gidx;          // [T, K+W]
  int32_t* counts;        // [T, 2] (valid main entries, valid entries) or null
  uint32_t* status;       // reset to 0 by the launch when non-null
  int32_t T, R, max_blocks, P, K, W;
  int32_t swa_max_blocks, swa_P;
  int32_t compact;        // pack each token's valid entries to the front (counts required)
  int64_t num_pages, bt_stride, topk_stride, swa_stride, swa_num_pages, swa_bt_stride;
};
cudaError_t launch_convert(const ConvertParams& p, cudaStream_t s);

// The pages' ragged form: token t fills out[cu[t] .. cu[t+1]) from its first cu[t+1] - cu[t]
// request-local indices; invalid (negative index or block outside [0, max_blocks)) -> 0.
struct RaggedParams {
  const int32_t* req_id;
  const int32_t* block_table;
  const int32_t* token_indices;  // [T, ti_stride]
  const int32_t* cu_seqlens;     // [T + 1]
  int32_t* out;
  int32_t T, R, max_blocks, P;
  int32_t num_cols;              // columns of token_indices; a longer token writes 0 past them
  int64_t bt_stride, ti_stride;
};
cudaError_t launch_convert_ragged(const RaggedParams& p, cudaStream_t s);

struct GatherParams {
  const uint8_t* cache;
  const int32_t* gidx;
  void* kv_out;           // bf16 [rows, 512]
  int64_t rows, num_pages;
  int32_t P;
  int32_t fmt;            // 0: fp8_ds_mla rows, 1: bf16 rows
};
cudaError_t launch_gather_dequant(const GatherParams& p, cudaStream_t s);

struct CombineParams {
  const float* o_part;    // [T, S, H, 512]
  const float* lse_part;  // [T, S, H]
  const float* sink;      // [H] or null
  void* out;              // bf16 [T, H, 512]
  float* lse;             // [T, H] or null
  int32_t T, S, H;
  int32_t sms;            // SMs of the device (sizes the grid to one wave)
};
cudaError_t launch_combine(const CombineParams& p, cudaStream_t s);

struct AttnParams {
  const void* q;          // bf16 [T, H, 512]
  CacheDesc cache;        // the main (top-k) scope's cache
  CacheDesc cache2;       // the window scope's cache (== cache when there is one cache)
  const int32_t* gidx;    // [T, N] converted slots, -1 = masked
  const int32_t* counts;  // [T, 2] (entries of the main scope, all entries) or null: K and N
  const float* sink;      // [H] or null
  void* out;              // bf16 [T, H, 512]          (S == 1)
  float* lse;             // [T, H] or null            (S == 1)
  float* o_part;          // [T, S, H, 512]            (S > 1)
  float* lse_part;        // [T, S, H]                 (S > 1)
  uint32_t* status;       // device status word
  float scale;
  int32_t T, H, N, K, S;  // N = row length of gidx; K = entries of the main scope (no counts)
  int32_t fmt;            // 0: fp8_ds_mla rows, 1: bf16 rows
  int32_t tiles_per_split;
  int32_t HG;             // head groups of 64 (CTAs per token and split)
  int32_t G;              // CTAs launched; CTA c takes work items c, c + G, ...
  uint64_t wait_limit_ns; // bound of every pipeline wait inside the kernel
};
cudaError_t launch_attn(const AttnParams& p, cudaStream_t s);
// CTAs that share one (token, split): one per group of 64 heads.
int attn_ctas_per_split(int H);
// CTAs the attention kernel launches for `items` work items on a device with `sms` SMs.
int attn_ctas(int64_t items, int sms);
// Bound of the kernels' pipeline waits (a test hook can shorten it), default 2 s.
uint64_t wait_limit_ns();

// ---- indexer step (the step that picks each decode token's top-k positions)
struct IndexerGatherParams {
  const uint8_t* cache;          // [num_pages, P * (D + 4)]
  const int32_t* block_table;    // [B, W], row stride bt_stride
  const int32_t* cu_seqlen;      // [B + 1]
  const int32_t* token_to_seq;   // [n]
  uint8_t* k_out;                // [n, D]
  float* scale_out;              // [n]
  int64_t bt_stride;
  int32_t n, B, W, P, D, layout, num_pages;
};
cudaError_t launch_indexer_gather(const IndexerGatherParams& p, cudaStream_t s);

struct IndexerLogitsParams {
  const uint8_t* q;              // e4m3 [T, H, 128]
  const float* weights;          // [T, H]
  const uint8_t* cache;          // [num_pages, P * 132], layout 0
  const int32_t* block_table;    // [R, W], row stride bt_stride
  const int32_t* req_id;         // [T]
  const int32_t* ctx_lens;       // [T]
  float* logits;                 // [T, L], row stride L
  uint32_t* status;              // optional device status word (bit 0: a wait gave up)
  int64_t bt_stride;
  int32_t T, H, P, R, W, L, num_pages;
  uint64_t wait_limit_ns;
};
cudaError_t launch_indexer_logits(const IndexerLogitsParams& p, cudaStream_t s);

struct IndexerTopkParams {
  const float* logits;           // [T, L], row stride stride
  const int32_t* ctx_lens;       // [T]
  int32_t* topk;                 // [T, K]
  int64_t stride;
  int32_t T, L, K;
  int32_t slice_cap;             // keys per CTA of the clustered kernel (set by the launch)
};
cudaError_t launch_indexer_topk(const IndexerTopkParams& p, cudaStream_t s);

// Sets the thread-local message returned by smd_last_error() and returns `code`.
int set_error(int code, const char* fmt, ...);

}  // namespace smd
