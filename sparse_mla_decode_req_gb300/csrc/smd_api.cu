// C-ABI entry points of libsmd (declared in include/smd.h): argument validation, the
// workload-aware split selector, workspace layout and kernel launches.  Host code only.
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <atomic>

#include "smd.h"
#include "smd_internal.h"

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(SMD_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr int64_t kMaxEntries = 1 << 20;   // K + W per token
constexpr int32_t kMaxTokens = 65535;      // grid.y limit of the per-token launches
// Split-selector cost model, in units of one 64-row tile of one CTA: fixed work per work
// item (Q load, pipeline fill, epilogue) and the extra combine launch.
constexpr int kCtaOverheadTiles = 4;
constexpr int kCombineTiles = 2;
constexpr uint64_t kDefaultWaitLimitNs = 2000000000ull;  // 2 s: far beyond any legitimate wait
std::atomic<uint64_t> g_wait_limit_ns{kDefaultWaitLimitNs};

int check_dims(const smd_dims* d) {
  if (d == nullptr) return fail(SMD_ERR_INVALID_ARG, "dims is NULL");
  if (d->num_tokens < 0 || d->num_tokens > kMaxTokens)
    return fail(SMD_ERR_INVALID_ARG, "num_tokens %d outside [0, %d]", d->num_tokens, kMaxTokens);
  if (d->num_heads < 1 || d->num_heads > SMD_MAX_HEADS)
    return fail(SMD_ERR_INVALID_ARG, "num_heads %d outside [1, %d]", d->num_heads, SMD_MAX_HEADS);
  if (d->num_requests < 1) return fail(SMD_ERR_INVALID_ARG, "num_requests %d < 1", d->num_requests);
  if (d->max_blocks_per_req < 1)
    return fail(SMD_ERR_INVALID_ARG, "max_blocks_per_req %d < 1", d->max_blocks_per_req);
  if (d->block_size < 1) return fail(SMD_ERR_INVALID_ARG, "block_size %d < 1", d->block_size);
  if (d->num_pages < 1) return fail(SMD_ERR_INVALID_ARG, "num_pages %lld < 1", (long long)d->num_pages);
  if (d->num_pages > (int64_t)INT32_MAX / d->block_size)
    return fail(SMD_ERR_INVALID_ARG, "num_pages * block_size must stay below 2^31");
  if (d->topk < 0 || d->swa < 0) return fail(SMD_ERR_INVALID_ARG, "topk/swa must be >= 0");
  if ((int64_t)d->topk + d->swa > kMaxEntries)
    return fail(SMD_ERR_INVALID_ARG, "topk + swa = %lld exceeds %lld", (long long)d->topk + d->swa,
                (long long)kMaxEntries);
  if (d->bt_stride < d->max_blocks_per_req)
    return fail(SMD_ERR_INVALID_ARG, "bt_stride %lld < max_blocks_per_req", (long long)d->bt_stride);
  if (d->topk > 0 && d->topk_stride < d->topk)
    return fail(SMD_ERR_INVALID_ARG, "topk_stride %lld < topk", (long long)d->topk_stride);
  if (d->swa > 0 && d->swa_stride < d->swa)
    return fail(SMD_ERR_INVALID_ARG, "swa_stride %lld < swa", (long long)d->swa_stride);
  if (d->cache_format != SMD_CACHE_FP8_DS_MLA && d->cache_format != SMD_CACHE_BF16)
    return fail(SMD_ERR_INVALID_ARG, "cache_format %d is neither 0 (fp8_ds_mla) nor 1 (bf16)", d->cache_format);
  return SMD_OK;
}

bool has_swa_cache(const smd_decode_opts* o) { return o != nullptr && o->swa_kv_cache != nullptr; }

// What each entry point reads of the window scope's options: the decode both the cache and
// its block table, the conversion only the block table, the attention only the cache.
enum class OptsUse { kDecode, kConvert, kAttention };

int check_opts(const smd_decode_opts* o, OptsUse use) {
  if (o == nullptr) return SMD_OK;
  const bool cache = o->swa_kv_cache != nullptr, table = o->swa_block_table != nullptr;
  if (use == OptsUse::kDecode && cache != table)
    return fail(SMD_ERR_INVALID_ARG, "swa_kv_cache and swa_block_table must be given together");
  const bool paged = (cache && use != OptsUse::kConvert) || (table && use != OptsUse::kAttention);
  if (!paged) return SMD_OK;
  if (o->swa_block_size < 1) return fail(SMD_ERR_INVALID_ARG, "swa_block_size %d < 1", o->swa_block_size);
  if (o->swa_num_pages < 1) return fail(SMD_ERR_INVALID_ARG, "swa_num_pages %lld < 1", (long long)o->swa_num_pages);
  if (o->swa_num_pages > (int64_t)INT32_MAX / o->swa_block_size)
    return fail(SMD_ERR_INVALID_ARG, "swa_num_pages * swa_block_size must stay below 2^31");
  if (cache && use != OptsUse::kConvert && !aligned16(o->swa_kv_cache))
    return fail(SMD_ERR_INVALID_ARG, "swa_kv_cache not 16-byte aligned");
  if (table && use != OptsUse::kAttention) {
    if (o->swa_max_blocks_per_req < 1)
      return fail(SMD_ERR_INVALID_ARG, "swa_max_blocks_per_req %d < 1", o->swa_max_blocks_per_req);
    if (o->swa_bt_stride < o->swa_max_blocks_per_req)
      return fail(SMD_ERR_INVALID_ARG, "swa_bt_stride %lld < swa_max_blocks_per_req", (long long)o->swa_bt_stride);
  }
  return SMD_OK;
}

bool compacting(const smd_decode_opts* o) { return o != nullptr && o->compact != 0; }

int device_sms(int num_sms) {
  if (num_sms > 0) return num_sms;
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  return n;
}

int select_splits(const smd_dims* d, int request, int sms) {
  const int64_t N = (int64_t)d->topk + d->swa;
  const int64_t tiles = (N + smd::kTileRows - 1) / smd::kTileRows;
  if (request < 0) {
    const int s = -request;
    return s > smd::kMaxSplits ? smd::kMaxSplits : s;
  }
  // (no separate cap for short work: on GB300 a CTA's fixed cost -- Q load, pipeline fill,
  // epilogue -- outweighs the combine, so short work gains from every split the cost model
  // below asks for; one request of 640 entries: 27.8 us at 4 splits, 25.7 at 5, 20.6 at 10)
  int cap = request == 0 ? smd::kMaxSplits : (request > smd::kMaxSplits ? smd::kMaxSplits : request);
  if (tiles < cap) cap = (int)(tiles > 0 ? tiles : 1);
  if (d->num_tokens == 0 || tiles == 0) return 1;
  const int64_t cps = smd::attn_ctas_per_split(d->num_heads);
  int best = 1;
  int64_t best_cost = INT64_MAX;
  for (int s = 1; s <= cap; ++s) {
    const int64_t tps = (tiles + s - 1) / s;
    if ((int64_t)(s - 1) * tps >= tiles) continue;  // would leave a split without a tile
    const int64_t ctas = (int64_t)d->num_tokens * s * cps;  // one CTA per SM
    const int64_t waves = (ctas + sms - 1) / sms;
    const int64_t cost = waves * (tps + kCtaOverheadTiles) + (s > 1 ? kCombineTiles : 0);
    if (cost < best_cost) {
      best_cost = cost;
      best = s;
    }
  }
  return best;
}

struct Layout {
  size_t status = 0, gidx = 0, counts = 0, o_part = 0, lse_part = 0, total = 0;
};

size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

Layout workspace_layout(const smd_dims* d, int S) {
  Layout L;
  const size_t T = (size_t)d->num_tokens, N = (size_t)d->topk + (size_t)d->swa, H = (size_t)d->num_heads;
  size_t off = 0;
  L.status = off;
  off += 256;
  L.gidx = off;
  off += up256(T * N * sizeof(int32_t));
  L.counts = off;
  off += up256(T * 2 * sizeof(int32_t));
  if (S > 1) {
    L.o_part = off;
    off += up256(T * (size_t)S * H * SMD_LATENT_DIM * sizeof(float));
    L.lse_part = off;
    off += up256(T * (size_t)S * H * sizeof(float));
  }
  L.total = off;
  return L;
}

// Attention launch parameters shared by the whole-step and the stage entry points.
smd::AttnParams attn_params(const smd_dims* d, const smd_decode_opts* o, int S, int sms, const void* q,
                            const uint8_t* cache, const int32_t* gidx, const int32_t* counts, const float* sink,
                            float scale, void* out, float* lse, float* o_part, float* lse_part, uint32_t* status) {
  const int64_t N = (int64_t)d->topk + d->swa;
  const int64_t tiles = (N + smd::kTileRows - 1) / smd::kTileRows;
  smd::AttnParams a{};
  a.q = q;
  a.cache = smd::make_cache_desc(cache, d->num_pages, d->block_size);
  a.cache2 = has_swa_cache(o) ? smd::make_cache_desc(o->swa_kv_cache, o->swa_num_pages, o->swa_block_size) : a.cache;
  a.gidx = gidx;
  a.counts = counts;
  a.sink = sink;
  a.out = out;
  a.lse = lse;
  a.o_part = S > 1 ? o_part : nullptr;
  a.lse_part = S > 1 ? lse_part : nullptr;
  a.status = status;
  a.scale = scale;
  a.T = d->num_tokens;
  a.H = d->num_heads;
  a.N = (int32_t)N;
  a.K = d->topk;
  a.S = S;
  a.fmt = d->cache_format;
  a.tiles_per_split = (int32_t)((tiles + S - 1) / S);
  if (a.tiles_per_split < 1) a.tiles_per_split = 1;
  a.HG = smd::attn_ctas_per_split(d->num_heads);
  a.G = smd::attn_ctas((int64_t)a.T * S * a.HG, sms);
  a.wait_limit_ns = smd::wait_limit_ns();
  return a;
}

smd::ConvertParams convert_params(const smd_dims* d, const smd_decode_opts* o, const int32_t* bt,
                                  const int32_t* req, const int32_t* topk, const int32_t* swa, int32_t* gidx,
                                  int32_t* counts, uint32_t* status) {
  smd::ConvertParams p{};
  p.block_table = bt;
  p.req_id = req;
  p.topk = topk;
  p.swa = swa;
  p.gidx = gidx;
  p.status = status;
  if (o != nullptr) {
    p.topk_length = o->topk_length;
    if (o->swa_block_table != nullptr) {
      p.swa_block_table = o->swa_block_table;
      p.swa_max_blocks = o->swa_max_blocks_per_req;
      p.swa_P = o->swa_block_size;
      p.swa_num_pages = o->swa_num_pages;
      p.swa_bt_stride = o->swa_bt_stride;
    }
    p.compact = o->compact != 0;
  }
  p.counts = p.compact ? counts : nullptr;
  p.T = d->num_tokens;
  p.R = d->num_requests;
  p.max_blocks = d->max_blocks_per_req;
  p.P = d->block_size;
  p.K = d->topk;
  p.W = d->swa;
  p.num_pages = d->num_pages;
  p.bt_stride = d->bt_stride;
  p.topk_stride = d->topk_stride;
  p.swa_stride = d->swa_stride;
  return p;
}

int check_index_ptrs(const smd_dims* d, const int32_t* bt, const int32_t* req, const int32_t* topk,
                     const int32_t* swa) {
  if (d->num_tokens == 0) return SMD_OK;
  if (bt == nullptr || req == nullptr) return fail(SMD_ERR_INVALID_ARG, "block_table and req_id are required");
  if (d->topk > 0 && topk == nullptr) return fail(SMD_ERR_INVALID_ARG, "topk_idx is NULL with topk > 0");
  if (d->swa > 0 && swa == nullptr) return fail(SMD_ERR_INVALID_ARG, "swa_idx is NULL with swa > 0");
  return SMD_OK;
}

}  // namespace

namespace smd {
uint64_t wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }

int set_error(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return code;
}
}  // namespace smd

extern "C" {

SMD_API const char* smd_last_error(void) { return g_err; }

SMD_API int smd_version(void) { return 200; }

SMD_API int smd_select_num_splits(const smd_dims* dims, int num_splits, int num_sms) {
  g_err[0] = '\0';
  const int rc = check_dims(dims);
  if (rc != SMD_OK) return rc;
  if (num_splits < -SMD_MAX_SPLITS) return fail(SMD_ERR_INVALID_ARG, "num_splits %d < -%d", num_splits, SMD_MAX_SPLITS);
  const int sms = device_sms(num_sms);
  if (sms <= 0) return fail(SMD_ERR_CUDA, "cannot query the device SM count");
  return select_splits(dims, num_splits, sms);
}

SMD_API size_t smd_workspace_size(const smd_dims* dims, int num_splits, int num_sms) {
  const int S = smd_select_num_splits(dims, num_splits, num_sms);
  if (S < 1) return 0;
  return workspace_layout(dims, S).total;
}

SMD_API uint64_t smd_set_wait_limit_ns(uint64_t limit_ns) {
  return g_wait_limit_ns.exchange(limit_ns == 0 ? kDefaultWaitLimitNs : limit_ns);
}

SMD_API int smd_convert_req_index(const smd_dims* dims, const int32_t* block_table, const int32_t* req_id,
                                  const int32_t* topk_idx, const int32_t* swa_idx, int32_t* gidx,
                                  smd_stream_t stream) {
  g_err[0] = '\0';
  int rc = check_dims(dims);
  if (rc != SMD_OK) return rc;
  rc = check_index_ptrs(dims, block_table, req_id, topk_idx, swa_idx);
  if (rc != SMD_OK) return rc;
  if (dims->num_tokens > 0 && dims->topk + dims->swa > 0 && gidx == nullptr)
    return fail(SMD_ERR_INVALID_ARG, "gidx is NULL");
  const cudaError_t e = smd::launch_convert(
      convert_params(dims, nullptr, block_table, req_id, topk_idx, swa_idx, gidx, nullptr, nullptr), stream);
  return e == cudaSuccess ? SMD_OK : cuda_fail(e, "convert launch");
}

SMD_API int smd_convert_req_index_ex(const smd_dims* dims, const smd_decode_opts* opts, const int32_t* block_table,
                                     const int32_t* req_id, const int32_t* topk_idx, const int32_t* swa_idx,
                                     int32_t* gidx, int32_t* counts, smd_stream_t stream) {
  g_err[0] = '\0';
  int rc = check_dims(dims);
  if (rc != SMD_OK) return rc;
  rc = check_opts(opts, OptsUse::kConvert);
  if (rc != SMD_OK) return rc;
  rc = check_index_ptrs(dims, block_table, req_id, topk_idx, swa_idx);
  if (rc != SMD_OK) return rc;
  if (dims->num_tokens > 0 && dims->topk + dims->swa > 0 && gidx == nullptr)
    return fail(SMD_ERR_INVALID_ARG, "gidx is NULL");
  if (dims->num_tokens > 0 && compacting(opts) && counts == nullptr)
    return fail(SMD_ERR_INVALID_ARG, "counts is required with compact");
  const cudaError_t e = smd::launch_convert(
      convert_params(dims, opts, block_table, req_id, topk_idx, swa_idx, gidx, counts, nullptr), stream);
  return e == cudaSuccess ? SMD_OK : cuda_fail(e, "convert launch");
}

SMD_API int smd_convert_req_index_ragged(const smd_dims* dims, const int32_t* block_table, const int32_t* req_id,
                                         const int32_t* token_indices, int32_t num_cols, int64_t ti_stride,
                                         const int32_t* cu_seqlens, int32_t* out, smd_stream_t stream) {
  g_err[0] = '\0';
  if (dims == nullptr) return fail(SMD_ERR_INVALID_ARG, "dims is NULL");
  if (dims->num_tokens < 0 || dims->num_tokens > kMaxTokens)
    return fail(SMD_ERR_INVALID_ARG, "num_tokens %d outside [0, %d]", dims->num_tokens, kMaxTokens);
  if (dims->num_requests < 1 || dims->max_blocks_per_req < 1 || dims->block_size < 1 ||
      dims->bt_stride < dims->max_blocks_per_req)
    return fail(SMD_ERR_INVALID_ARG, "bad num_requests/max_blocks_per_req/block_size/bt_stride");
  if (num_cols < 0 || ti_stride < num_cols)
    return fail(SMD_ERR_INVALID_ARG, "num_cols %d < 0 or ti_stride %lld < num_cols", num_cols, (long long)ti_stride);
  if (dims->num_tokens == 0) return SMD_OK;
  if (block_table == nullptr || req_id == nullptr || cu_seqlens == nullptr || out == nullptr ||
      (num_cols > 0 && token_indices == nullptr))
    return fail(SMD_ERR_INVALID_ARG, "block_table, req_id, token_indices, cu_seqlens and out are required");
  smd::RaggedParams p{};
  p.req_id = req_id;
  p.block_table = block_table;
  p.token_indices = token_indices;
  p.cu_seqlens = cu_seqlens;
  p.out = out;
  p.T = dims->num_tokens;
  p.R = dims->num_requests;
  p.max_blocks = dims->max_blocks_per_req;
  p.P = dims->block_size;
  p.num_cols = num_cols;
  p.bt_stride = dims->bt_stride;
  p.ti_stride = ti_stride;
  const cudaError_t e = smd::launch_convert_ragged(p, stream);
  return e == cudaSuccess ? SMD_OK : cuda_fail(e, "ragged convert launch");
}

SMD_API int smd_gather_dequant(const smd_dims* dims, const uint8_t* kv_cache, const int32_t* gidx,
                               int64_t num_rows, void* kv_out, smd_stream_t stream) {
  g_err[0] = '\0';
  if (dims == nullptr) return fail(SMD_ERR_INVALID_ARG, "dims is NULL");
  if (dims->block_size < 1 || dims->num_pages < 1 || dims->num_pages > (int64_t)INT32_MAX / dims->block_size)
    return fail(SMD_ERR_INVALID_ARG, "bad block_size/num_pages");
  if (num_rows < 0) return fail(SMD_ERR_INVALID_ARG, "num_rows < 0");
  if (num_rows == 0) return SMD_OK;
  if (kv_cache == nullptr || gidx == nullptr || kv_out == nullptr)
    return fail(SMD_ERR_INVALID_ARG, "NULL pointer");
  if (!aligned16(kv_cache) || !aligned16(kv_out)) return fail(SMD_ERR_INVALID_ARG, "kv_cache/kv_out not 16-byte aligned");
  if (dims->cache_format != SMD_CACHE_FP8_DS_MLA && dims->cache_format != SMD_CACHE_BF16)
    return fail(SMD_ERR_INVALID_ARG, "cache_format %d is neither 0 nor 1", dims->cache_format);
  smd::GatherParams p{kv_cache, gidx, kv_out, num_rows, dims->num_pages, dims->block_size, dims->cache_format};
  const cudaError_t e = smd::launch_gather_dequant(p, stream);
  return e == cudaSuccess ? SMD_OK : cuda_fail(e, "gather launch");
}

SMD_API int smd_lse_combine(int32_t num_tokens, int32_t num_splits, int32_t num_heads, const float* o_part,
                            const float* lse_part, const float* sink, void* out, float* lse, smd_stream_t stream) {
  g_err[0] = '\0';
  if (num_tokens < 0 || num_heads < 1 || num_splits < 1 || num_splits > SMD_MAX_SPLITS)
    return fail(SMD_ERR_INVALID_ARG, "bad combine shape T=%d S=%d H=%d", num_tokens, num_splits, num_heads);
  if (num_tokens == 0) return SMD_OK;
  if (o_part == nullptr || lse_part == nullptr || out == nullptr) return fail(SMD_ERR_INVALID_ARG, "NULL pointer");
  if (!aligned16(o_part) || !aligned16(out)) return fail(SMD_ERR_INVALID_ARG, "o_part/out not 16-byte aligned");
  const int sms = device_sms(0);
  if (sms <= 0) return fail(SMD_ERR_CUDA, "cannot query the device SM count");
  smd::CombineParams p{o_part, lse_part, sink, out, lse, num_tokens, num_splits, num_heads, sms};
  const cudaError_t e = smd::launch_combine(p, stream);
  return e == cudaSuccess ? SMD_OK : cuda_fail(e, "combine launch");
}

SMD_API int smd_sparse_mla_decode_ex(const smd_dims* dims, const smd_decode_opts* opts, const void* q,
                                     const uint8_t* kv_cache, const int32_t* block_table, const int32_t* req_id,
                                     const int32_t* topk_idx, const int32_t* swa_idx, const float* sink, float scale,
                                     void* out, float* lse, int num_splits, void* workspace, size_t workspace_bytes,
                                     smd_stream_t stream) {
  g_err[0] = '\0';
  int rc = check_dims(dims);
  if (rc != SMD_OK) return rc;
  rc = check_opts(opts, OptsUse::kDecode);
  if (rc != SMD_OK) return rc;
  rc = check_index_ptrs(dims, block_table, req_id, topk_idx, swa_idx);
  if (rc != SMD_OK) return rc;
  if (num_splits < -SMD_MAX_SPLITS) return fail(SMD_ERR_INVALID_ARG, "num_splits %d < -%d", num_splits, SMD_MAX_SPLITS);
  if (dims->num_tokens > 0) {
    if (q == nullptr || kv_cache == nullptr || out == nullptr)
      return fail(SMD_ERR_INVALID_ARG, "q, kv_cache and out are required");
    if (!aligned16(q) || !aligned16(out) || !aligned16(kv_cache))
      return fail(SMD_ERR_INVALID_ARG, "q/out/kv_cache not 16-byte aligned");
  }
  if (workspace == nullptr || !aligned16(workspace))
    return fail(SMD_ERR_INVALID_ARG, "workspace is NULL or not 16-byte aligned");
  const int sms = device_sms(0);
  if (sms <= 0) return fail(SMD_ERR_CUDA, "cannot query the device SM count");
  const int S = select_splits(dims, num_splits, sms);
  const Layout L = workspace_layout(dims, S);
  if (workspace_bytes < L.total)
    return fail(SMD_ERR_WORKSPACE, "workspace %zu bytes < required %zu", workspace_bytes, L.total);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint32_t* status = reinterpret_cast<uint32_t*>(ws + L.status);
  int32_t* gidx = reinterpret_cast<int32_t*>(ws + L.gidx);
  int32_t* counts = compacting(opts) ? reinterpret_cast<int32_t*>(ws + L.counts) : nullptr;

  cudaError_t e = smd::launch_convert(
      convert_params(dims, opts, block_table, req_id, topk_idx, swa_idx, gidx, counts, status), stream);
  if (e != cudaSuccess) return cuda_fail(e, "convert launch");
  if (dims->num_tokens == 0) return SMD_OK;

  const smd::AttnParams a =
      attn_params(dims, opts, S, sms, q, kv_cache, gidx, counts, sink, scale, out, lse,
                  reinterpret_cast<float*>(ws + L.o_part), reinterpret_cast<float*>(ws + L.lse_part), status);
  e = smd::launch_attn(a, stream);
  if (e != cudaSuccess) return cuda_fail(e, "attention launch");
  if (S > 1) {
    smd::CombineParams c{a.o_part, a.lse_part, sink, out, lse, dims->num_tokens, S, dims->num_heads, sms};
    e = smd::launch_combine(c, stream);
    if (e != cudaSuccess) return cuda_fail(e, "combine launch");
  }
  return SMD_OK;
}

SMD_API int smd_sparse_mla_decode(const smd_dims* dims, const void* q, const uint8_t* kv_cache,
                                  const int32_t* block_table, const int32_t* req_id, const int32_t* topk_idx,
                                  const int32_t* swa_idx, const float* sink, float scale, void* out, float* lse,
                                  int num_splits, void* workspace, size_t workspace_bytes, smd_stream_t stream) {
  return smd_sparse_mla_decode_ex(dims, nullptr, q, kv_cache, block_table, req_id, topk_idx, swa_idx, sink, scale,
                                  out, lse, num_splits, workspace, workspace_bytes, stream);
}

SMD_API int smd_sparse_mla_attention(const smd_dims* dims, const smd_decode_opts* opts, const void* q,
                                     const uint8_t* kv_cache, const int32_t* gidx, const int32_t* counts,
                                     const float* sink, float scale, int num_splits, void* out, float* lse,
                                     float* o_part, float* lse_part, int32_t* status, smd_stream_t stream) {
  g_err[0] = '\0';
  int rc = check_dims(dims);
  if (rc != SMD_OK) return rc;
  rc = check_opts(opts, OptsUse::kAttention);
  if (rc != SMD_OK) return rc;
  if (num_splits < -SMD_MAX_SPLITS) return fail(SMD_ERR_INVALID_ARG, "num_splits %d < -%d", num_splits, SMD_MAX_SPLITS);
  if (dims->num_tokens == 0) return SMD_OK;
  const int sms = device_sms(0);
  if (sms <= 0) return fail(SMD_ERR_CUDA, "cannot query the device SM count");
  const int S = select_splits(dims, num_splits, sms);
  const int64_t N = (int64_t)dims->topk + dims->swa;
  if (q == nullptr || kv_cache == nullptr || (N > 0 && gidx == nullptr))
    return fail(SMD_ERR_INVALID_ARG, "q, kv_cache and gidx are required");
  if (S == 1 && out == nullptr) return fail(SMD_ERR_INVALID_ARG, "out is required with one split");
  if (S > 1 && (o_part == nullptr || lse_part == nullptr))
    return fail(SMD_ERR_INVALID_ARG, "o_part and lse_part are required with %d splits", S);
  if (!aligned16(q) || !aligned16(kv_cache) || (out != nullptr && !aligned16(out)) ||
      (o_part != nullptr && !aligned16(o_part)))
    return fail(SMD_ERR_INVALID_ARG, "q/kv_cache/out/o_part not 16-byte aligned");
  const smd::AttnParams a = attn_params(dims, opts, S, sms, q, kv_cache, gidx, counts, sink, scale, out, lse, o_part,
                                        lse_part, reinterpret_cast<uint32_t*>(status));
  const cudaError_t e = smd::launch_attn(a, stream);
  return e == cudaSuccess ? SMD_OK : cuda_fail(e, "attention launch");
}

SMD_API int smd_indexer_gather_k(const uint8_t* cache, int64_t num_pages, int32_t block_size, int32_t head_dim,
                                 int32_t layout, const int32_t* block_table, int32_t num_batches,
                                 int32_t max_blocks, int64_t bt_stride, const int32_t* cu_seqlen,
                                 const int32_t* token_to_seq, int32_t num_tokens, uint8_t* k_out, float* scale_out,
                                 smd_stream_t stream) {
  g_err[0] = '\0';
  if (num_tokens < 0) return fail(SMD_ERR_INVALID_ARG, "num_tokens %d < 0", num_tokens);
  if (num_tokens == 0) return SMD_OK;
  if (head_dim < 4 || head_dim > 4096 || head_dim % 4 != 0)
    return fail(SMD_ERR_INVALID_ARG, "head_dim %d: a multiple of 4 in [4, 4096]", head_dim);
  if (layout != 0 && layout != 1) return fail(SMD_ERR_INVALID_ARG, "layout %d is not 0 or 1", layout);
  if (block_size < 1 || num_pages < 1 || num_batches < 0 || max_blocks < 1 || bt_stride < max_blocks)
    return fail(SMD_ERR_INVALID_ARG, "bad block_size/num_pages/num_batches/max_blocks/bt_stride");
  if (num_pages > INT32_MAX) return fail(SMD_ERR_INVALID_ARG, "num_pages above 2^31 - 1");
  if (cache == nullptr || block_table == nullptr || cu_seqlen == nullptr || token_to_seq == nullptr ||
      k_out == nullptr || scale_out == nullptr)
    return fail(SMD_ERR_INVALID_ARG, "NULL pointer");
  if (!aligned16(cache)) return fail(SMD_ERR_INVALID_ARG, "cache not 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(k_out) & 3u) || (reinterpret_cast<uintptr_t>(scale_out) & 3u))
    return fail(SMD_ERR_INVALID_ARG, "k_out/scale_out not 4-byte aligned");
  smd::IndexerGatherParams p{cache, block_table, cu_seqlen, token_to_seq, k_out, scale_out, bt_stride,
                             num_tokens, num_batches, max_blocks, block_size, head_dim, layout, (int32_t)num_pages};
  const cudaError_t e = smd::launch_indexer_gather(p, stream);
  return e == cudaSuccess ? SMD_OK : cuda_fail(e, "indexer gather launch");
}

SMD_API int smd_indexer_mqa_logits(const smd_indexer_dims* d, const uint8_t* q, const float* weights,
                                   const uint8_t* cache, const int32_t* block_table, const int32_t* req_id,
                                   const int32_t* ctx_lens, float* logits, int32_t* device_status,
                                   smd_stream_t stream) {
  g_err[0] = '\0';
  if (d == nullptr) return fail(SMD_ERR_INVALID_ARG, "dims is NULL");
  if (d->num_tokens < 0 || d->num_tokens > kMaxTokens)
    return fail(SMD_ERR_INVALID_ARG, "num_tokens %d outside [0, %d]", d->num_tokens, kMaxTokens);
  if (d->head_dim != 128) return fail(SMD_ERR_UNSUPPORTED, "head_dim %d: the logits kernel takes 128", d->head_dim);
  if (d->num_heads != 32 && d->num_heads != 64 && d->num_heads != 128)
    return fail(SMD_ERR_UNSUPPORTED, "num_heads %d: the logits kernel takes 32, 64 or 128", d->num_heads);
  const int32_t P = d->block_size;
  if (P < 8 || P > 128 || (P & (P - 1)) != 0)
    return fail(SMD_ERR_UNSUPPORTED, "block_size %d: the logits kernel takes 8, 16, 32, 64 or 128", P);
  if (d->layout != 0) return fail(SMD_ERR_UNSUPPORTED, "layout %d: the logits kernel reads layout 0", d->layout);
  if (d->num_requests < 1 || d->max_blocks_per_req < 1 || d->bt_stride < d->max_blocks_per_req || d->num_pages < 1)
    return fail(SMD_ERR_INVALID_ARG, "bad num_requests/max_blocks_per_req/bt_stride/num_pages");
  if (d->num_pages > INT32_MAX) return fail(SMD_ERR_INVALID_ARG, "num_pages above 2^31 - 1");
  if (d->max_len < 0) return fail(SMD_ERR_INVALID_ARG, "max_len %d < 0", d->max_len);
  if (d->num_tokens == 0 || d->max_len == 0) return SMD_OK;
  if (q == nullptr || weights == nullptr || cache == nullptr || block_table == nullptr || req_id == nullptr ||
      ctx_lens == nullptr || logits == nullptr)
    return fail(SMD_ERR_INVALID_ARG, "NULL pointer");
  if (!aligned16(q) || !aligned16(cache) || !aligned16(logits))
    return fail(SMD_ERR_INVALID_ARG, "q/cache/logits not 16-byte aligned");
  smd::IndexerLogitsParams p{q, weights, cache, block_table, req_id, ctx_lens, logits,
                             reinterpret_cast<uint32_t*>(device_status), d->bt_stride, d->num_tokens, d->num_heads,
                             P, d->num_requests, d->max_blocks_per_req, d->max_len, (int32_t)d->num_pages,
                             smd::wait_limit_ns()};
  const cudaError_t e = smd::launch_indexer_logits(p, stream);
  return e == cudaSuccess ? SMD_OK : cuda_fail(e, "indexer logits launch");
}

SMD_API int smd_indexer_topk(const float* logits, int32_t num_tokens, int32_t max_len, int64_t logits_stride,
                             const int32_t* ctx_lens, int32_t k, int32_t* topk, smd_stream_t stream) {
  g_err[0] = '\0';
  if (num_tokens < 0 || max_len < 0 || logits_stride < max_len)
    return fail(SMD_ERR_INVALID_ARG, "bad num_tokens/max_len/logits_stride");
  if (k < 1 || k > (1 << 20)) return fail(SMD_ERR_INVALID_ARG, "k %d outside [1, 2^20]", k);
  if (num_tokens == 0) return SMD_OK;
  if (logits == nullptr || ctx_lens == nullptr || topk == nullptr) return fail(SMD_ERR_INVALID_ARG, "NULL pointer");
  smd::IndexerTopkParams p{logits, ctx_lens, topk, logits_stride, num_tokens, max_len, k, 0};
  const cudaError_t e = smd::launch_indexer_topk(p, stream);
  return e == cudaSuccess ? SMD_OK : cuda_fail(e, "indexer top-k launch");
}

SMD_API int smd_read_status(const void* workspace, int32_t* device_status, smd_stream_t stream) {
  g_err[0] = '\0';
  if (workspace == nullptr || device_status == nullptr) return fail(SMD_ERR_INVALID_ARG, "NULL pointer");
  int32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  *device_status = v;
  if (v & 2) return fail(SMD_ERR_DEVICE_CHECK, "a device range check failed (status 0x%x)", v);
  return v != 0 ? fail(SMD_ERR_TIMEOUT, "a kernel's bounded wait gave up (status 0x%x)", v) : SMD_OK;
}

}  // extern "C"
