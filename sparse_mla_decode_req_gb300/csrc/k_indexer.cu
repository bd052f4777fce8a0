// The indexer step: the per-token choice of the top-k cached positions that the sparse
// decode then attends to.  Three kernels:
//
//   indexer_gather_kernel: the pages' key gather from the paged fp8 key cache (vLLM PR
//     #52212 report, "关键源码片段", _cp_gather_indexer_quant_cache_gfx950_kernel): token
//     tid of a ragged batch belongs to sequence token_to_seq[tid] (valid in [0, B)) and
//     must lie in [cu_seqlen[b], cu_seqlen[b + 1]); its position in the sequence selects a
//     block-table entry whose page must lie in [0, num_pages); the position's D key bytes
//     go to k_out[tid] and its float32 scale to scale_out[tid] (0, with the key bytes left
//     as they are, for an invalid page; nothing for an invalid token).  Block offsets are
//     64-bit.  One warp per token.
//
//   indexer_logits_kernel: the fp8 paged MQA logits (vLLM PR #41217 report, "实现拆解"
//     item 6: one kernel for the per-head scores and their weighted sum), as read in the
//     design notes: logit[t, s] = scale_s * sum_h w[t, h] * max(0, q[t, h, :] . k_s) with
//     e4m3 q and k.  One CTA per (token, 128 positions): TMA brings the tile's key rows
//     (one 3-D box per page of the 128B-swizzled [page][position][128 bytes] view of
//     layout 0) and the token's query heads; one elected lane issues four
//     tcgen05.mma.kind::f8f6f4 (M = 128 positions, N = H heads, K = 32 bytes each) into
//     TMEM; the four warps read their 32 positions' H head scores back, rectify, weight,
//     sum and scale them.  Positions at or past the token's context, and positions whose
//     block or page is invalid, get -inf.  The step is bound by reading the key cache
//     (132 bytes per position against 2 * 128 * H flops on the tensor cores).
//
//   indexer_topk_kernel: per token the K positions of the largest finite logits among its
//     first ctx_lens[t]: a radix select (four 8-bit passes over order-preserving keys)
//     finds the K-th largest logit, then one ordered pass writes the positions above it
//     (ascending) followed by the lowest positions equal to it; -1 pads a token with
//     fewer than K finite logits.  One CTA of 1024 threads per token; the logits are read
//     from L2, six passes.
#include <cuda.h>

#include "smd_device.cuh"
#include "smd_internal.h"

namespace smd {
namespace {

// ------------------------------------------------------------------ key gather
constexpr int kGatherThreads = 256;

__global__ void __launch_bounds__(kGatherThreads) indexer_gather_kernel(IndexerGatherParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (kGatherThreads / 32);
  const int64_t page_bytes = (int64_t)p.P * (p.D + 4);
  for (int64_t tid = (int64_t)blockIdx.x * (kGatherThreads / 32) + (threadIdx.x >> 5); tid < p.n; tid += warps) {
    const int32_t b = __ldg(p.token_to_seq + tid);
    if (b < 0 || b >= p.B) continue;
    const int32_t start = __ldg(p.cu_seqlen + b), end = __ldg(p.cu_seqlen + b + 1);
    if (tid < start || tid >= end) continue;
    const int64_t pos = tid - start;
    const int64_t blk = pos / p.P;
    const int32_t off = (int32_t)(pos - blk * p.P);
    const int32_t page = blk < p.W ? __ldg(p.block_table + (int64_t)b * p.bt_stride + blk) : -1;
    if (page < 0 || page >= p.num_pages) {
      if (lane == 0) p.scale_out[tid] = 0.f;
      continue;
    }
    const uint8_t* pg = p.cache + (int64_t)page * page_bytes;
    const int64_t vo = p.layout == 0 ? (int64_t)off * p.D : (int64_t)off * (p.D + 4);
    const int64_t so = p.layout == 0 ? (int64_t)p.P * p.D + 4 * off : vo + p.D;
    const uint32_t* src = reinterpret_cast<const uint32_t*>(pg + vo);
    uint32_t* dst = reinterpret_cast<uint32_t*>(p.k_out + tid * p.D);
    for (int w = lane; w < p.D / 4; w += 32) dst[w] = __ldg(src + w);
    if (lane == 0) p.scale_out[tid] = __ldg(reinterpret_cast<const float*>(pg + so));
  }
}

// ------------------------------------------------------------------ paged MQA logits
constexpr int kLgRows = 128;       // positions per CTA (UMMA M)
constexpr int kLgDim = 128;        // key / query bytes per row (one 128-byte swizzled row)
constexpr int kLgThreads = 128;
constexpr uint32_t kLgKBytes = kLgRows * kLgDim;           // 16 KB key tile
constexpr uint64_t kLgDrainLimitNs = 2000000000ull;

__host__ __device__ constexpr uint32_t lg_smem_used(int H) {
  return kLgKBytes + (uint32_t)H * kLgDim + (uint32_t)H * 4 + 64;
}

struct LogitsKernelParams {
  IndexerLogitsParams p;
  CUtensorMap kmap;   // key bytes of layout 0: [num_pages][P positions][128 bytes], 128B swizzle
  CUtensorMap qmap;   // q: [T * H rows][128 bytes], 128B swizzle
};

template <int H>
__global__ void __launch_bounds__(kLgThreads) indexer_logits_kernel(const __grid_constant__ LogitsKernelParams kp) {
  const IndexerLogitsParams& p = kp.p;
  const int t = blockIdx.y;
  const int pos0 = blockIdx.x * kLgRows;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int pos = pos0 + tid;
  float* const out = p.logits + (int64_t)t * p.L;
  const int ctx = min(__ldg(p.ctx_lens + t), p.L);
  if (pos0 >= ctx) {  // a tile wholly past the context: -inf only
    if (pos < p.L) out[pos] = -INFINITY;
    return;
  }
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* const sK = smem;                                  // [128 positions][128 B], swizzled
  uint8_t* const sQ = smem + kLgKBytes;                      // [H heads][128 B], swizzled
  float* const sW = reinterpret_cast<float*>(sQ + H * kLgDim);
  uint64_t* const bar = reinterpret_cast<uint64_t*>(sW + H);  // [0]: tile landed, [1]: MMAs done
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(bar + 2);

  const int32_t r = __ldg(p.req_id + t);
  const bool req_ok = r >= 0 && r < p.R;
  auto page_of = [&](int position) -> int32_t {  // -1 if the block or the page is invalid
    if (!req_ok) return -1;
    const int32_t blk = position / p.P;
    if (blk >= p.W) return -1;
    const int32_t pg = __ldg(p.block_table + (int64_t)r * p.bt_stride + blk);
    return pg >= 0 && pg < p.num_pages ? pg : -1;
  };
  // this thread's position: its page and float32 scale (layout 0: after the page's key bytes)
  const int32_t my_page = pos < ctx ? page_of(pos) : -1;
  float my_scale = 0.f;
  if (my_page >= 0)
    my_scale = __ldg(reinterpret_cast<const float*>(p.cache + (int64_t)my_page * p.P * (kLgDim + 4) +
                                                    (int64_t)p.P * kLgDim + 4 * (pos % p.P)));
  if (tid < H) sW[tid] = __ldg(p.weights + (int64_t)t * H + tid);
  if (tid == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, H);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (tid == 0) {
    mbar_arrive_expect_tx(&bar[0], kLgKBytes + H * kLgDim);
    // one box per page of the tile (P divides 128); an invalid page reads as zeros
    for (int j = 0; j < kLgRows / p.P; ++j)
      tma_load_3d(smem_u32(sK) + j * p.P * kLgDim, &kp.kmap, 0, 0, page_of(pos0 + j * p.P), &bar[0]);
    tma_load_2d(smem_u32(sQ), &kp.qmap, 0, t * H, &bar[0]);
  }
  bool ok = true;
  if (warp == 0) {
    ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bar[0], 0, p.wait_limit_ns));
    if (ok) {
      tc_fence_after();
      const uint64_t da = desc_sw128(smem_u32(sK), 16, 1024);  // A: keys, K-major
      const uint64_t db = desc_sw128(smem_u32(sQ), 16, 1024);  // B: query heads, K-major
      constexpr uint32_t kId = idesc_e4m3_f32(kLgRows, H);
#pragma unroll
      for (int kk = 0; kk < kLgDim / 32; ++kk)  // 32 bytes per step: +2 in the descriptors' 16-byte units
        umma_f8_elect(tmem, da + (uint64_t)(2 * kk), db + (uint64_t)(2 * kk), kId, kk > 0 ? 1u : 0u);
      umma_commit_elect(&bar[1]);
    } else if (lane == 0) {
      if (p.status != nullptr) atomicOr(p.status, kStatusTimeout);
      (void)mbar_wait_bounded(&bar[0], 0, kLgDrainLimitNs);  // no TMA write may outlive the CTA
    }
  }
  ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bar[1], 0, p.wait_limit_ns));
  if (ok) {
    tc_fence_after();
    float acc = 0.f;
#pragma unroll
    for (int c = 0; c < H / 32; ++c) {
      uint32_t v[32];
      tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + c * 32, v);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; ++i) acc = fmaf(sW[c * 32 + i], fmaxf(__uint_as_float(v[i]), 0.f), acc);
    }
    if (pos < p.L) out[pos] = my_page >= 0 ? acc * my_scale : -INFINITY;
  } else if (lane == 0 && p.status != nullptr) {
    atomicOr(p.status, kStatusTimeout);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, H);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return (EncodeTiledFn) nullptr;
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

template <int H>
cudaError_t launch_logits_h(const LogitsKernelParams& kp, cudaStream_t s) {
  // at most 512 / H resident CTAs per SM, so that every CTA's TMEM allocation succeeds at once
  const uint32_t per_sm = 512u / H;
  uint32_t smem = lg_smem_used(H) + 1024;
  const uint32_t share = 232448u / per_sm;
  if (smem < share) smem = share;
  static thread_local bool done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !done[dev]) {
    e = cudaFuncSetAttribute(indexer_logits_kernel<H>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) done[dev] = true;
  }
  const dim3 grid((unsigned)((kp.p.L + kLgRows - 1) / kLgRows), (unsigned)kp.p.T);
  indexer_logits_kernel<H><<<grid, kLgThreads, smem, s>>>(kp);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ top-k
constexpr int kTopkThreads = 1024;
constexpr int kTopkWarps = kTopkThreads / 32;

// Order-preserving key of a logit: larger logit, larger key; -inf and NaN map to 0 and are
// never selected; -0 is read as +0.
__device__ __forceinline__ uint32_t order_key(float x) {
  if (!(x > -INFINITY)) return 0u;
  const uint32_t u = x == 0.f ? 0u : __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive block-wide ranks of two predicates (in thread order) and their totals.
__device__ __forceinline__ void block_rank2(bool a, bool b, int& ra, int& rb, int& ta, int& tb, int (*wsum)[2]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t ba = __ballot_sync(0xffffffffu, a), bb = __ballot_sync(0xffffffffu, b);
  const uint32_t below = (1u << lane) - 1u;
  if (lane == 0) {
    wsum[warp][0] = __popc(ba);
    wsum[warp][1] = __popc(bb);
  }
  __syncthreads();
  int pa = 0, pb = 0, sa = 0, sb = 0;
  for (int w = 0; w < kTopkWarps; ++w) {
    const int x = wsum[w][0], y = wsum[w][1];
    pa += w < warp ? x : 0;
    pb += w < warp ? y : 0;
    sa += x;
    sb += y;
  }
  ra = pa + __popc(ba & below);
  rb = pb + __popc(bb & below);
  ta = sa;
  tb = sb;
  __syncthreads();  // wsum is reused by the next call
}

__global__ void __launch_bounds__(kTopkThreads) indexer_topk_kernel(IndexerTopkParams p) {
  __shared__ uint32_t hist[256];
  __shared__ int wsum[kTopkWarps][2];
  __shared__ uint32_t s_bin, s_remaining;
  const int t = blockIdx.x;
  const int n = max(0, min(__ldg(p.ctx_lens + t), p.L));
  const float* row = p.logits + (int64_t)t * p.stride;
  int32_t* out = p.topk + (int64_t)t * p.K;
  const int tid = threadIdx.x;

  // finite logits
  int cnt = 0;
  for (int i = tid; i < n; i += kTopkThreads) cnt += order_key(row[i]) != 0u;
  for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
  if ((tid & 31) == 0) wsum[tid >> 5][0] = cnt;
  __syncthreads();
  int total = 0;
  for (int w = 0; w < kTopkWarps; ++w) total += wsum[w][0];
  __syncthreads();

  uint32_t tau = 0u;      // key of the K-th largest logit (0: take every finite one)
  int need_eq = 0;        // positions equal to tau to take
  if (total > p.K) {
    uint32_t prefix = 0u, mask = 0u;
    uint32_t remaining = (uint32_t)p.K;
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int i = tid; i < 256; i += kTopkThreads) hist[i] = 0u;
      __syncthreads();
      for (int i = tid; i < n; i += kTopkThreads) {
        const uint32_t k = order_key(row[i]);
        if (k != 0u && (k & mask) == prefix) atomicAdd(&hist[(k >> shift) & 255u], 1u);
      }
      __syncthreads();
      if (tid == 0) {
        uint32_t cum = 0u;
        int b = 255;
        for (; b > 0; --b) {
          if (cum + hist[b] >= remaining) break;
          cum += hist[b];
        }
        s_bin = (uint32_t)b;
        s_remaining = remaining - cum;
      }
      __syncthreads();
      prefix |= s_bin << shift;
      mask |= 255u << shift;
      remaining = s_remaining;
      __syncthreads();
    }
    tau = prefix;
    need_eq = (int)remaining;
  }
  const int n_gt = total > p.K ? p.K - need_eq : total;  // positions strictly above tau (all finite if none)
  // ordered pass: positions above tau ascending into [0, n_gt), then the lowest positions
  // equal to tau into [n_gt, K)
  int base_gt = 0, base_eq = 0;
  for (int c0 = 0; c0 < n; c0 += kTopkThreads) {
    const int i = c0 + tid;
    const uint32_t k = i < n ? order_key(row[i]) : 0u;
    const bool gt = k != 0u && k > tau;
    const bool eq = tau != 0u && k == tau;
    int rg, re, tg, te;
    block_rank2(gt, eq, rg, re, tg, te, wsum);
    if (gt) out[base_gt + rg] = i;
    if (eq && base_eq + re < need_eq) out[n_gt + base_eq + re] = i;
    base_gt += tg;
    base_eq += te;
  }
  const int written = n_gt + (need_eq < base_eq ? need_eq : base_eq);
  for (int i = written + tid; i < p.K; i += kTopkThreads) out[i] = -1;
}

}  // namespace

cudaError_t launch_indexer_gather(const IndexerGatherParams& p, cudaStream_t s) {
  if (p.n == 0) return cudaSuccess;
  const int64_t per = kGatherThreads / 32;
  int64_t blocks = (p.n + per - 1) / per;
  if (blocks > 65535 * 16) blocks = 65535 * 16;
  indexer_gather_kernel<<<(unsigned)blocks, kGatherThreads, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_indexer_logits(const IndexerLogitsParams& p, cudaStream_t s) {
  if (p.T == 0 || p.L == 0) return cudaSuccess;
  EncodeTiledFn enc = encode_tiled();
  if (enc == nullptr) return cudaErrorNotSupported;
  LogitsKernelParams kp;
  kp.p = p;
  {
    const cuuint64_t gdim[3] = {(cuuint64_t)kLgDim, (cuuint64_t)p.P, (cuuint64_t)p.num_pages};
    const cuuint64_t gstride[2] = {(cuuint64_t)kLgDim, (cuuint64_t)p.P * (kLgDim + 4)};
    const cuuint32_t box[3] = {(cuuint32_t)kLgDim, (cuuint32_t)p.P, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (enc(&kp.kmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(p.cache), gdim, gstride, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t gdim[2] = {(cuuint64_t)kLgDim, (cuuint64_t)p.T * (cuuint64_t)p.H};
    const cuuint64_t gstride[1] = {(cuuint64_t)kLgDim};
    const cuuint32_t box[2] = {(cuuint32_t)kLgDim, (cuuint32_t)p.H};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(&kp.qmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(p.q), gdim, gstride, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  switch (p.H) {
    case 32: return launch_logits_h<32>(kp, s);
    case 64: return launch_logits_h<64>(kp, s);
    case 128: return launch_logits_h<128>(kp, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_indexer_topk(const IndexerTopkParams& p, cudaStream_t s) {
  if (p.T == 0 || p.K == 0) return cudaSuccess;
  indexer_topk_kernel<<<(unsigned)p.T, kTopkThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace smd
