// Index conversion: request-local top-k / window positions -> global cache slots, by the
// rule of smd_index.cuh.
//
// Three kernels:
//   convert_kernel: dense [T, K+W] output, -1 for invalid entries; one thread per entry,
//     consecutive threads on consecutive columns of one token (coalesced).
//   convert_compact_kernel: the same rule, then each token's valid slots packed to the
//     front in column order with the counts (valid main-scope entries, valid entries), so
//     the attention gathers no masked row (vLLM PR #41217 report, "实现拆解" item 2: the
//     sparse lengths built before the decode).  One CTA per token: a block-wide scan of
//     each 512-column chunk gives every valid entry its packed position.
//   convert_ragged_kernel: the pages' own ragged form, token t filling positions
//     [cu_seqlens[t], cu_seqlens[t+1]) from its first columns, 0 for an invalid entry (a
//     negative index or a block outside [0, max_blocks)); like that kernel it checks
//     neither the physical page nor the request id (a request id outside [0, R) and a
//     position past the index array's columns, which that kernel would read out of
//     bounds, are written as 0 here).
//
// In an SMD_DEBUG build a failed range check here sets bit 1 of the status word; one made
// by another CTA before CTA 0 resets the word in the same launch can be lost.
#include "smd_device.cuh"
#include "smd_index.cuh"
#include "smd_internal.h"

namespace smd {
namespace {

// Slot of column j of token t under the dense rule, -1 if invalid.
__device__ __forceinline__ int32_t convert_one(const ConvertParams& p, int32_t t, int32_t j) {
  IndexStep s;
  if (!index_block(p, t, j, __ldg(index_addr(p, t, j)), __ldg(p.req_id + t), s)) return -1;
  return index_slot(p, s, __ldg(s.bt_entry));
}

__global__ void __launch_bounds__(256) convert_kernel(ConvertParams p) {
  grid_dep_wait();  // launched as a programmatic dependent of the previous kernel
  const int32_t t = blockIdx.y;
  const int32_t N = p.K + p.W;
  if (p.status != nullptr && t == 0 && blockIdx.x == 0 && threadIdx.x == 0) *p.status = 0u;
  const int32_t j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= N || !in_range(t < p.T, p.status)) return;
  p.gidx[(int64_t)t * N + j] = convert_one(p, t, j);
}

constexpr int kCompactThreads = 512;

__global__ void __launch_bounds__(kCompactThreads) convert_compact_kernel(ConvertParams p) {
  grid_dep_wait();
  __shared__ int32_t warp_total[kCompactThreads / 32][2];
  __shared__ int32_t running[2];  // (main entries, all entries) packed so far
  const int32_t t = blockIdx.x;
  const int32_t N = p.K + p.W;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (p.status != nullptr && t == 0 && threadIdx.x == 0) *p.status = 0u;
  if (threadIdx.x == 0) running[0] = running[1] = 0;
  __syncthreads();
  for (int32_t c0 = 0; c0 < N; c0 += kCompactThreads) {
    const int32_t j = c0 + threadIdx.x;
    const int32_t g = j < N ? convert_one(p, t, j) : -1;
    const bool valid = g >= 0;
    const uint32_t vb = __ballot_sync(0xffffffffu, valid);
    const uint32_t mb = __ballot_sync(0xffffffffu, valid && j < p.K);
    if (lane == 0) {
      warp_total[warp][0] = __popc(vb);
      warp_total[warp][1] = __popc(mb);
    }
    __syncthreads();
    int32_t before = 0, chunk_total = 0, chunk_main = 0;
    for (int w = 0; w < kCompactThreads / 32; ++w) {
      const int32_t n = warp_total[w][0];
      before += w < warp ? n : 0;
      chunk_total += n;
      chunk_main += warp_total[w][1];
    }
    const int32_t pos = running[1] + before + __popc(vb & ((1u << lane) - 1u));
    if (valid && in_range(pos < N, p.status)) p.gidx[(int64_t)t * N + pos] = g;
    __syncthreads();  // every thread has read running[] and warp_total[]
    if (threadIdx.x == 0) {
      running[0] += chunk_main;
      running[1] += chunk_total;
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    p.counts[2 * t] = running[0];
    p.counts[2 * t + 1] = running[1];
  }
}

__global__ void __launch_bounds__(256) convert_ragged_kernel(RaggedParams p) {
  const int32_t t = blockIdx.y;
  const int32_t start = __ldg(p.cu_seqlens + t);
  const int32_t len = __ldg(p.cu_seqlens + t + 1) - start;
  for (int32_t j = blockIdx.x * blockDim.x + threadIdx.x; j < len; j += gridDim.x * blockDim.x) {
    int32_t out = 0;
    const int32_t req = __ldg(p.req_id + t);
    if (j < p.num_cols && req >= 0 && req < p.R) {
      const int32_t idx = __ldg(p.token_indices + (int64_t)t * p.ti_stride + j);
      if (idx >= 0) {
        const int32_t b = idx / p.P;
        if (b < p.max_blocks) out = __ldg(p.block_table + (int64_t)req * p.bt_stride + b) * p.P + (idx - b * p.P);
      }
    }
    p.out[start + j] = out;
  }
}

cudaError_t launch_pdl(const void* fn, dim3 grid, dim3 block, void** args, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace

cudaError_t launch_convert(const ConvertParams& p, cudaStream_t s) {
  const int32_t N = p.K + p.W;
  if (p.T == 0) {
    if (p.status != nullptr) return cudaMemsetAsync(p.status, 0, sizeof(uint32_t), s);
    return cudaSuccess;
  }
  ConvertParams q = p;
  void* args[] = {&q};
  if (p.compact) return launch_pdl((const void*)convert_compact_kernel, dim3(p.T), dim3(kCompactThreads), args, s);
  if (N == 0) {
    if (p.status != nullptr) return cudaMemsetAsync(p.status, 0, sizeof(uint32_t), s);
    return cudaSuccess;
  }
  return launch_pdl((const void*)convert_kernel, dim3((N + 255) / 256, p.T), dim3(256), args, s);
}

cudaError_t launch_convert_ragged(const RaggedParams& p, cudaStream_t s) {
  if (p.T == 0) return cudaSuccess;
  const unsigned gx = (unsigned)((p.num_cols + 255) / 256 > 0 ? (p.num_cols + 255) / 256 : 1);
  convert_ragged_kernel<<<dim3(gx, p.T), 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace smd
