// Internal launch interface between the C-ABI layer (smd_api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace smd {

constexpr int kTileRows = 64;     // rows per split unit (one attention tile)
constexpr int kMaxSplits = 32;

struct ConvertParams {
  const int32_t* block_table;
  const int32_t* req_id;
  const int32_t* topk;
  const int32_t* swa;
  int32_t* gidx;          // [T, K+W]
  uint32_t* status;       // reset to 0 by the launch when non-null
  int32_t T, R, max_blocks, P, K, W;
  int64_t num_pages, bt_stride, topk_stride, swa_stride;
};
cudaError_t launch_convert(const ConvertParams& p, cudaStream_t s);

struct GatherParams {
  const uint8_t* cache;
  const int32_t* gidx;
  void* kv_out;           // bf16 [rows, 512]
  int64_t rows, num_pages;
  int32_t P;
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
  const uint8_t* cache;
  const int32_t* gidx;    // [T, N] converted slots, -1 = masked
  const float* sink;      // [H] or null
  void* out;              // bf16 [T, H, 512]          (S == 1)
  float* lse;             // [T, H] or null            (S == 1)
  float* o_part;          // [T, S, H, 512]            (S > 1)
  float* lse_part;        // [T, S, H]                 (S > 1)
  uint32_t* status;       // device status word
  float scale;
  int64_t num_pages;
  int32_t T, H, N, P, S;
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

// Sets the thread-local message returned by smd_last_error() and returns `code`.
int set_error(int code, const char* fmt, ...);

}  // namespace smd
