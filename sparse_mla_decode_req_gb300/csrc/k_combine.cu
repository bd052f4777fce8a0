// Warp-shuffle log-sum-exp combine of split-K partials, with the attention sink.
//
// vLLM PR #52212 report, "实现拆解" item 2 (split-K with a separate reduce launch,
// test symbol _launch_sparse_decode_reduce).  Per (token, head):
//   M   = max(max_s lse_s, sink)        w_s = exp(lse_s - M)
//   den = sum_s w_s + exp(sink - M)     out = sum_s w_s o_s / den     lse = M + ln den
// with the -inf guard of SGLang PR #26208 report, "评论区精华" (an empty split has
// lse_s = -inf and weight 0; no terms at all gives out = 0, lse = -inf).
//
// One warp per (token, head).  Lane s < S holds lse_s, so the max and the weight sum
// are two butterfly reductions; each lane then owns 16 of the 512 output dims and
// streams the S partial rows with 16-byte loads (a warp reads 2 KB contiguous per
// split) and writes 32 contiguous bytes of bf16.
#include "smd_device.cuh"
#include "smd_internal.h"

namespace smd {

__global__ void __launch_bounds__(256) lse_combine_kernel(CombineParams p) {
  grid_dep_wait();  // launched as a programmatic dependent of the attention kernel
  const int64_t pair = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);  // t * H + h
  const int lane = threadIdx.x & 31;
  if (pair >= (int64_t)p.T * p.H) return;
  const int32_t t = (int32_t)(pair / p.H);
  const int32_t h = (int32_t)(pair - (int64_t)t * p.H);
  constexpr float kLog2e = 1.4426950408889634f;
  constexpr float kLn2 = 0.6931471805599453f;

  const float ninf = -INFINITY;
  const float l_mine = lane < p.S ? __ldg(p.lse_part + ((int64_t)t * p.S + lane) * p.H + h) : ninf;
  const float sink = p.sink != nullptr ? __ldg(p.sink + h) : ninf;
  float M = l_mine;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  M = fmaxf(M, sink);

  uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.out) + pair * (kLatent * 2)) + lane * 2;
  if (M == ninf) {  // no entries and no sink
    dst[0] = make_uint4(0, 0, 0, 0);
    dst[1] = make_uint4(0, 0, 0, 0);
    if (p.lse != nullptr && lane == 0) p.lse[pair] = ninf;
    return;
  }
  const float w_mine = l_mine == ninf ? 0.f : exp2f((l_mine - M) * kLog2e);
  float den = w_mine;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
  den += sink == ninf ? 0.f : exp2f((sink - M) * kLog2e);
  const float inv = 1.f / den;

  float acc[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.f;
  for (int s = 0; s < p.S; ++s) {
    const float w = __shfl_sync(0xffffffffu, w_mine, s);
    if (w == 0.f) continue;  // warp-uniform
    const float4* src = reinterpret_cast<const float4*>(p.o_part + (((int64_t)t * p.S + s) * p.H + h) * kLatent) +
                        lane * 4;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 v = __ldg(src + i);
      acc[4 * i + 0] = fmaf(w, v.x, acc[4 * i + 0]);
      acc[4 * i + 1] = fmaf(w, v.y, acc[4 * i + 1]);
      acc[4 * i + 2] = fmaf(w, v.z, acc[4 * i + 2]);
      acc[4 * i + 3] = fmaf(w, v.w, acc[4 * i + 3]);
    }
  }
  uint32_t packed[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    packed[i] = bf16x2_bits(__floats2bfloat162_rn(acc[2 * i] * inv, acc[2 * i + 1] * inv));
  dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
  dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
  if (p.lse != nullptr && lane == 0) p.lse[pair] = M + log2f(den) * kLn2;
}

cudaError_t launch_combine(const CombineParams& p, cudaStream_t s) {
  const int64_t pairs = (int64_t)p.T * p.H;
  if (pairs == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((pairs + 7) / 8), 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, lse_combine_kernel, p);
}

}  // namespace smd
