// The index conversion rule of the conversion kernels (dense, compacting).
//
// vLLM PR #41217 report, "关键源码片段", _convert_req_index_to_global_index_kernel: for
// column j of token t the block is index // P and the in-page offset index % P; the block
// must lie in [0, max_num_blocks_per_req) and the slot is block_table[req, block] * P +
// offset.  The physical page is also range-checked against the cache, as the cp-gather
// kernel of vLLM PR #52212 report ("关键源码片段") does.  Window entries follow the top-k
// entries at column offset K (SGLang PR #26208 report, _gather_dequant_dsv4_kernel's
// k_offset); when the window scope has its own cache, its entries go through that cache's
// block table and page size (vLLM PR #52212 report, "实现拆解" items 1 and 3).  A top-k
// column k of token t is masked when k >= TopkLength[t] (SGLang PR #26208 report,
// "关键源码片段", HAS_TOPK_LENGTH).
//
// The rule runs in two halves around its one dependent load (the block-table entry):
// index_block() checks the request-local index and finds the block-table entry to read,
// index_slot() checks the page read from it.
#pragma once

#include "smd_device.cuh"
#include "smd_internal.h"

namespace smd {

// The request-local index of column j of token t.
__device__ __forceinline__ const int32_t* index_addr(const ConvertParams& p, int32_t t, int32_t j) {
  return j >= p.K ? p.swa + (int64_t)t * p.swa_stride + (j - p.K) : p.topk + (int64_t)t * p.topk_stride + j;
}

// Where an entry stands after its block-table lookup was located.
struct IndexStep {
  const int32_t* bt_entry;  // the block-table entry to read
  int32_t off;              // in-page offset
  int32_t scope;            // 0: main scope, 1: window scope (its own cache when it has one)
};

// First half: false if column j of token t (request-local index idx, request req) is
// already invalid; else the block-table entry to read.
__device__ __forceinline__ bool index_block(const ConvertParams& p, int32_t t, int32_t j, int32_t idx, int32_t req,
                                            IndexStep& s) {
  const bool window = j >= p.K;
  if (idx < 0) return false;
  if (!window && p.topk_length != nullptr && j >= __ldg(p.topk_length + t)) return false;
  if (req < 0 || req >= p.R) return false;
  const bool own = window && p.swa_block_table != nullptr;  // the window scope's own cache
  const int32_t P = own ? p.swa_P : p.P;
  const int32_t b = idx / P;
  if (b >= (own ? p.swa_max_blocks : p.max_blocks)) return false;
  s.off = idx - b * P;
  s.bt_entry = own ? p.swa_block_table + (int64_t)req * p.swa_bt_stride + b : p.block_table + (int64_t)req * p.bt_stride + b;
  s.scope = own ? 1 : 0;
  return true;
}

// Second half: the global slot for the page read from the entry, or -1 if the page is
// outside the scope's cache.
__device__ __forceinline__ int32_t index_slot(const ConvertParams& p, const IndexStep& s, int32_t page) {
  const int32_t P = s.scope ? p.swa_P : p.P;
  if (page < 0 || (int64_t)page >= (s.scope ? p.swa_num_pages : p.num_pages)) return -1;
  return page * P + s.off;
}

}  // namespace smd
