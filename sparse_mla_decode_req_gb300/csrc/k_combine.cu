// Warp-shuffle log-sum-exp combine of split-K partials, with the attention sink.
//
// vLLM PR #52212 report, "实现拆解" item 2 (split-K with a separate reduce launch,
// test symbol _launch_sparse_decode_reduce).  Per (token, head):
//   M   = max(max_s lse_s, sink)        w_s = exp(lse_s - M)
//   den = sum_s w_s + exp(sink - M)     out = sum_s w_s o_s / den     lse = M + ln den
// with the -inf guard of SGLang PR #26208 report, "评论区精华" (an empty split has
// lse_s = -inf and weight 0; no terms at all gives out = 0, lse = -inf).
//
// WPP warps per (token, head) (1, 2 or 4), each owning 512 / WPP output dims.  Lane
// s < S holds lse_s, so the max and the weight sum are two butterfly reductions (each
// warp does them); each lane then streams its 16 / WPP consecutive dims of the S
// partial rows with 16-byte loads (a warp reads 2048 / WPP contiguous bytes per split)
// and writes them as bf16.
// The host takes WPP = 4 when the step has few (token, head) pairs, so that enough
// loads are in flight, and fewer warps per pair once the grid would pass one wave.
#include "smd_device.cuh"
#include "smd_internal.h"

namespace smd {

template <int WPP>
__global__ void __launch_bounds__(256) lse_combine_kernel(CombineParams p) {
  constexpr int kNv = 4 / WPP;                 // float4 per lane and split
  constexpr int kDimsPerWarp = kLatent / WPP;  // 128 * kNv
  grid_dep_wait();  // launched as a programmatic dependent of the attention kernel
  const int64_t gw = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int64_t pair = gw / WPP;  // t * H + h
  const int part = (int)(gw - pair * WPP);
  const int lane = threadIdx.x & 31;
  if (pair >= (int64_t)p.T * p.H) return;
  const int32_t t = (int32_t)(pair / p.H);
  const int32_t h = (int32_t)(pair - (int64_t)t * p.H);
  constexpr float kLog2e = 1.4426950408889634f;
  constexpr float kLn2 = 0.6931471805599453f;

  const float ninf = -INFINITY;
  // This lane's dims: 4 kNv consecutive ones from d0.  The first kPre splits' rows are
  // loaded before the lse reduction, so that their round trip overlaps the lse one.
  const int d0 = part * kDimsPerWarp + lane * 4 * kNv;
  auto row_of = [&](int s) {
    return reinterpret_cast<const float4*>(p.o_part + (((int64_t)t * p.S + s) * p.H + h) * kLatent + d0);
  };
  constexpr int kPre = 8 / kNv;  // splits preloaded (8 float4 per lane)
  float4 pre[kPre][kNv];
#pragma unroll
  for (int s = 0; s < kPre; ++s)
#pragma unroll
    for (int i = 0; i < kNv; ++i) pre[s][i] = s < p.S ? __ldg(row_of(s) + i) : make_float4(0.f, 0.f, 0.f, 0.f);
  const float l_mine = lane < p.S ? __ldg(p.lse_part + ((int64_t)t * p.S + lane) * p.H + h) : ninf;
  const float sink = p.sink != nullptr ? __ldg(p.sink + h) : ninf;
  float M = l_mine;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  M = fmaxf(M, sink);

  uint2* dst = reinterpret_cast<uint2*>(static_cast<uint8_t*>(p.out) + (pair * kLatent + d0) * 2);
  const bool writes_lse = p.lse != nullptr && part == 0 && lane == 0;
  if (M == ninf) {  // no entries and no sink
#pragma unroll
    for (int i = 0; i < kNv; ++i) dst[i] = make_uint2(0, 0);
    if (writes_lse) p.lse[pair] = ninf;
    return;
  }
  const float w_mine = l_mine == ninf ? 0.f : exp2f((l_mine - M) * kLog2e);
  float den = w_mine;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
  den += sink == ninf ? 0.f : exp2f((sink - M) * kLog2e);
  const float inv = 1.f / den;

  float4 acc[kNv];
#pragma unroll
  for (int i = 0; i < kNv; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  // Loads are unconditional (a batch of them in flight per unrolled group); a split of
  // weight 0 (lse -inf: no valid entries) contributes an exact 0 whatever its row holds.
#pragma unroll
  for (int s = 0; s < kPre; ++s) {
    const float w = __shfl_sync(0xffffffffu, w_mine, s);  // 0 past S
#pragma unroll
    for (int i = 0; i < kNv; ++i) {
      float4 v = pre[s][i];
      if (w == 0.f) v = make_float4(0.f, 0.f, 0.f, 0.f);
      acc[i].x = fmaf(w, v.x, acc[i].x);
      acc[i].y = fmaf(w, v.y, acc[i].y);
      acc[i].z = fmaf(w, v.z, acc[i].z);
      acc[i].w = fmaf(w, v.w, acc[i].w);
    }
  }
#pragma unroll(kNv == 4 ? 2 : kNv == 2 ? 4 : 8)
  for (int s = kPre; s < p.S; ++s) {
    const float w = __shfl_sync(0xffffffffu, w_mine, s);
    const float4* src = row_of(s);
#pragma unroll
    for (int i = 0; i < kNv; ++i) {
      float4 v = __ldg(src + i);
      if (w == 0.f) v = make_float4(0.f, 0.f, 0.f, 0.f);
      acc[i].x = fmaf(w, v.x, acc[i].x);
      acc[i].y = fmaf(w, v.y, acc[i].y);
      acc[i].z = fmaf(w, v.z, acc[i].z);
      acc[i].w = fmaf(w, v.w, acc[i].w);
    }
  }
  uint32_t packed[2 * kNv];
#pragma unroll
  for (int i = 0; i < kNv; ++i) {
    packed[2 * i] = bf16x2_bits(__floats2bfloat162_rn(acc[i].x * inv, acc[i].y * inv));
    packed[2 * i + 1] = bf16x2_bits(__floats2bfloat162_rn(acc[i].z * inv, acc[i].w * inv));
  }
  if constexpr (kNv == 1) {
    *dst = make_uint2(packed[0], packed[1]);
  } else {  // 16-byte stores
#pragma unroll
    for (int i = 0; i < kNv / 2; ++i)
      reinterpret_cast<uint4*>(dst)[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
  }
  if (writes_lse) p.lse[pair] = M + log2f(den) * kLn2;
}

cudaError_t launch_combine(const CombineParams& p, cudaStream_t s) {
  const int64_t pairs = (int64_t)p.T * p.H;
  if (pairs == 0) return cudaSuccess;
  // Warps per pair: as many as keep the grid within one wave of 32 warps per SM.
  const int64_t kWaveWarps = (int64_t)(p.sms > 0 ? p.sms : 1) * 32;
  const int wpp = pairs * 4 <= kWaveWarps ? 4 : pairs * 2 <= kWaveWarps ? 2 : 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((pairs * wpp + 7) / 8), 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (wpp == 4) return cudaLaunchKernelEx(&cfg, lse_combine_kernel<4>, p);
  if (wpp == 2) return cudaLaunchKernelEx(&cfg, lse_combine_kernel<2>, p);
  return cudaLaunchKernelEx(&cfg, lse_combine_kernel<1>, p);
}

}  // namespace smd
