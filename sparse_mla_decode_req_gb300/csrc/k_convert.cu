// Index conversion: request-local top-k / window positions -> global cache slots.
//
// vLLM PR #41217 report, "关键源码片段", _convert_req_index_to_global_index_kernel: for
// each (token, column) the block is index // P and the in-page offset index % P; the block
// must lie in [0, max_num_blocks_per_req) and the slot is block_table[req, block] * P +
// offset.  The physical page is also range-checked against the cache, as the cp-gather
// kernel of vLLM PR #52212 report ("关键源码片段") does.  Unlike the ragged 0-filled
// output of that kernel, the output here is dense [T, K+W] with -1 for invalid entries;
// window entries follow the top-k entries at column offset K (SGLang PR #26208 report,
// _gather_dequant_dsv4_kernel's k_offset).
//
// One thread per output entry; consecutive threads take consecutive columns of one
// token, so index reads and slot writes are coalesced.  The block table is tiny and
// stays in L1/L2.
#include "smd_device.cuh"
#include "smd_internal.h"

namespace smd {

__global__ void __launch_bounds__(256) convert_kernel(ConvertParams p) {
  grid_dep_wait();  // launched as a programmatic dependent of the previous kernel
  const int32_t t = blockIdx.y;
  const int32_t N = p.K + p.W;
  if (p.status != nullptr && t == 0 && blockIdx.x == 0 && threadIdx.x == 0) *p.status = 0u;
  const int32_t j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= N) return;
  const int32_t idx = j < p.K ? __ldg(p.topk + (int64_t)t * p.topk_stride + j)
                              : __ldg(p.swa + (int64_t)t * p.swa_stride + (j - p.K));
  const int32_t req = __ldg(p.req_id + t);
  int32_t g = -1;
  if (idx >= 0 && req >= 0 && req < p.R) {
    const int32_t b = idx / p.P;
    const int32_t off = idx - b * p.P;
    if (b < p.max_blocks) {
      const int32_t page = __ldg(p.block_table + (int64_t)req * p.bt_stride + b);
      if (page >= 0 && (int64_t)page < p.num_pages) g = page * p.P + off;
    }
  }
  p.gidx[(int64_t)t * N + j] = g;
}

cudaError_t launch_convert(const ConvertParams& p, cudaStream_t s) {
  const int32_t N = p.K + p.W;
  if (p.T == 0 || N == 0) {
    if (p.status != nullptr) return cudaMemsetAsync(p.status, 0, sizeof(uint32_t), s);
    return cudaSuccess;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((N + 255) / 256, p.T, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, convert_kernel, p);
}

}  // namespace smd
