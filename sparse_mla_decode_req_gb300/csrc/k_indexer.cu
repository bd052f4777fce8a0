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
//     item 6: one kernel for the per-head scores and their weighted sum).  The pages print
//     no formula; the reading here is logit[t, s] = scale_s * sum_h w[t, h] * max(0,
//     q[t, h, :] . k_s) with e4m3 q and k (a per-head stage before the sum implies a
//     per-head non-linearity, taken as the rectifier).  One CTA per token and 1-8 tiles of
//     128 positions: a TMA warp streams the key rows (one 3-D box per page of the
//     128B-swizzled [page][position][128 bytes] view of layout 0) through a 4-stage ring
//     and loads the token's query heads; an MMA warp issues four tcgen05.mma.kind::f8f6f4
//     per tile (M = 128 positions, N = H heads, K = 32 bytes each) into one of two TMEM
//     buffers; four warps read their 32 positions' H head scores back, rectify, weight,
//     sum and scale them.  Positions at or past the token's context, and positions whose
//     request, block or page is invalid, get -inf.  The step is bound by reading the key
//     cache (132 bytes per position against 2 * 128 * H flops on the tensor cores).
//
//   indexer_topk_kernel: per token the K positions of the largest finite logits among its
//     first ctx_lens[t]: a radix select over order-preserving keys (a 12-bit pass fused
//     with the one read of the row, then two 10-bit passes over the keys under the chosen
//     digit) finds the K-th largest logit, then one ordered pass writes the positions
//     above it (ascending) followed by the lowest positions equal to it; -1 pads a token
//     with fewer than K finite logits.  One CTA of 512 threads per token, the row's keys
//     in shared memory when it holds up to 40 K positions.
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
constexpr int kLgRows = 128;        // positions per tile (UMMA M)
constexpr int kLgDim = 128;         // key / query bytes per row (one 128-byte swizzled row)
constexpr int kLgMaxTilesPerCta = 8;  // tiles of one token per CTA, at most (the launch picks 1..8)
constexpr int kLgStages = 4;        // key tiles in flight per CTA
constexpr int kLgThreads = 192;     // warps 0-3 epilogue (one TMEM lane quarter each), 4 TMA, 5 MMA
constexpr int kLgTmaWarp = 4, kLgMmaWarp = 5;
constexpr uint32_t kLgKBytes = kLgRows * kLgDim;  // 16 KB key tile

__host__ __device__ constexpr uint32_t lg_smem_used(int H) {
  return kLgStages * kLgKBytes + (uint32_t)H * kLgDim + (uint32_t)H * 4 + 256;
}

struct LogitsKernelParams {
  IndexerLogitsParams p;
  int tiles_per_cta;
  CUtensorMap kmap;   // key bytes of layout 0: [num_pages][P positions][128 bytes], 128B swizzle
  CUtensorMap qmap;   // q: [T * H rows][128 bytes], 128B swizzle
};

struct LgBars {
  uint64_t full[kLgStages];   // TMA -> MMA: key tile landed
  uint64_t empty[kLgStages];  // MMA commit -> TMA: key tile read
  uint64_t tfull[2];          // MMA commit -> epilogue: scores in TMEM buffer
  uint64_t tempty[2];         // epilogue (4 warps) -> MMA: TMEM buffer read
  uint64_t qfull;             // the token's query heads landed
  uint64_t drain;             // MMA warp's own UMMAs, before TMEM is freed
  uint32_t tmem;
  uint32_t abort;
};

// One CTA per (token, 8 tiles of 128 positions): a TMA warp streams the key tiles through
// a 4-stage ring, an MMA warp scores each tile against the token's H query heads into one
// of two TMEM buffers (four kind::f8f6f4 UMMAs of K = 32 bytes), and four epilogue warps
// turn each buffer into 128 logits while the next tile is scored.
template <int H>
__global__ void __launch_bounds__(kLgThreads) indexer_logits_kernel(const __grid_constant__ LogitsKernelParams kp) {
  const IndexerLogitsParams& p = kp.p;
  const int t = blockIdx.y;
  const int tpc = kp.tiles_per_cta;
  const int tile0 = blockIdx.x * tpc;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  float* const out = p.logits + (int64_t)t * p.L;
  const int ctx = min(__ldg(p.ctx_lens + t), p.L);
  const int ntiles = min(tpc, (ctx + kLgRows - 1) / kLgRows - tile0);  // tiles with positions < ctx
  if (ntiles <= 0) {  // every position of the CTA is past the context: -inf only
    for (int i = tid; i < tpc * kLgRows; i += kLgThreads) {
      const int pos = tile0 * kLgRows + i;
      if (pos < p.L) out[pos] = -INFINITY;
    }
    return;
  }
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* const sK = smem;                                   // kLgStages x [128 positions][128 B]
  uint8_t* const sQ = smem + kLgStages * kLgKBytes;           // [H heads][128 B] (1 KB aligned)
  float* const sW = reinterpret_cast<float*>(sQ + H * kLgDim);
  LgBars* const bars = reinterpret_cast<LgBars*>(sW + H);
  const uint64_t limit = p.wait_limit_ns;

  const int32_t r = __ldg(p.req_id + t);
  const bool req_ok = r >= 0 && r < p.R;
  auto page_of = [&](int position) -> int32_t {  // -1 if the block or the page is invalid
    if (!req_ok) return -1;
    const int32_t blk = position / p.P;
    if (blk >= p.W) return -1;
    const int32_t pg = __ldg(p.block_table + (int64_t)r * p.bt_stride + blk);
    return pg >= 0 && pg < p.num_pages ? pg : -1;
  };
  if (tid < H) sW[tid] = __ldg(p.weights + (int64_t)t * H + tid);
  if (tid == 0) {
    for (int i = 0; i < kLgStages; ++i) {
      mbar_init(&bars->full[i], 1);
      mbar_init(&bars->empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->tfull[i], 1);
      mbar_init(&bars->tempty[i], 4);
    }
    mbar_init(&bars->qfull, 1);
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&bars->tmem, 2 * H);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem;
  auto give_up = [&]() {
    atomicExch(&bars->abort, 1u);
    if (p.status != nullptr) atomicOr(p.status, kStatusTimeout);
  };
  auto aborted_ = [&]() { return *reinterpret_cast<volatile uint32_t*>(&bars->abort) != 0u; };
  auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {  // bounded, warp-uniform
    bool ok = true;
    if (!mbar_test(bar, parity)) {
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(bar, parity)) {
        if (aborted_() || globaltimer_ns() - t0 > limit) {
          ok = false;
          break;
        }
      }
    }
    return __all_sync(0xffffffffu, ok);
  };

  if (warp == kLgTmaWarp) {
    int issued = 0;
    if (lane == 0) {
      mbar_arrive_expect_tx(&bars->qfull, H * kLgDim);
      tma_load_2d(smem_u32(sQ), &kp.qmap, 0, t * H, &bars->qfull);
    }
    for (int i = 0; i < ntiles; ++i) {
      const int s = i % kLgStages;
      if (i >= kLgStages && !wait(&bars->empty[s], ((i / kLgStages) - 1) & 1)) {
        if (lane == 0) give_up();
        break;
      }
      if (lane == 0) {
        const int pos0 = (tile0 + i) * kLgRows;
        mbar_arrive_expect_tx(&bars->full[s], kLgKBytes);
        // one box per page of the tile (P divides 128); an invalid page reads as zeros
        for (int j = 0; j < kLgRows / p.P; ++j)
          tma_load_3d(smem_u32(sK + s * kLgKBytes) + j * p.P * kLgDim, &kp.kmap, 0, 0, page_of(pos0 + j * p.P),
                      &bars->full[s]);
      }
      __syncwarp();
      ++issued;
    }
    // every key tile issued has landed before the CTA may leave
    if (lane == 0)
      for (int i = issued - kLgStages < 0 ? 0 : issued - kLgStages; i < issued; ++i)
        (void)mbar_wait_bounded(&bars->full[i % kLgStages], (i / kLgStages) & 1, 2000000000ull);
    if (lane == 0) (void)mbar_wait_bounded(&bars->qfull, 0, 2000000000ull);
    __syncwarp();
  } else if (warp == kLgMmaWarp) {
    const uint64_t db = desc_sw128(smem_u32(sQ), 16, 1024);  // B: query heads, K-major
    constexpr uint32_t kId = idesc_e4m3_f32(kLgRows, H);
    bool ok = wait(&bars->qfull, 0);
    for (int i = 0; i < ntiles && ok; ++i) {
      const int s = i % kLgStages, b = i & 1;
      ok = wait(&bars->full[s], (i / kLgStages) & 1);
      ok = ok && (i < 2 || wait(&bars->tempty[b], ((i >> 1) - 1) & 1));
      if (!ok) break;
      tc_fence_after();
      const uint64_t da = desc_sw128(smem_u32(sK + s * kLgKBytes), 16, 1024);  // A: keys, K-major
#pragma unroll
      for (int kk = 0; kk < kLgDim / 32; ++kk)  // 32 bytes per step: +2 in the descriptors' 16-byte units
        umma_f8_elect(tmem + b * H, da + (uint64_t)(2 * kk), db + (uint64_t)(2 * kk), kId, kk > 0 ? 1u : 0u);
      umma_commit_elect(&bars->empty[s]);
      umma_commit_elect(&bars->tfull[b]);
    }
    if (!ok && lane == 0) give_up();
    // every UMMA issued has completed before TMEM is freed
    umma_commit_elect(&bars->drain);
    if (lane == 0) (void)mbar_wait_bounded(&bars->drain, 0, 2000000000ull);
    __syncwarp();
  } else {  // epilogue warps 0-3: warp w owns TMEM lanes (positions) 32w .. 32w+31
    for (int i = 0; i < ntiles; ++i) {
      const int b = i & 1;
      const int pos = (tile0 + i) * kLgRows + tid;
      // this position's page and scale (layout 0: the page's float32 scales follow its keys)
      const int32_t pg = pos < ctx ? page_of(pos) : -1;
      const bool valid = pg >= 0;
      float sc = 0.f;
      if (valid)
        sc = __ldg(reinterpret_cast<const float*>(p.cache + (int64_t)pg * p.P * (kLgDim + 4) + (int64_t)p.P * kLgDim +
                                                  4 * (pos % p.P)));
      if (!wait(&bars->tfull[b], (i >> 1) & 1)) {
        if (lane == 0) give_up();
        break;
      }
      tc_fence_after();
      float acc = 0.f;
#pragma unroll
      for (int c = 0; c < H / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + b * H + c * 32, v);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 32; ++k) acc = fmaf(sW[c * 32 + k], fmaxf(__uint_as_float(v[k]), 0.f), acc);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->tempty[b]);
      if (pos < p.L) out[pos] = valid ? acc * sc : -INFINITY;
    }
    // positions of this CTA past its last scored tile
    for (int i = ntiles * kLgRows + tid; i < tpc * kLgRows; i += 128) {
      const int pos = tile0 * kLgRows + i;
      if (pos < p.L) out[pos] = -INFINITY;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 2 * H);
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
  // at most 512 / (2H) resident CTAs per SM, so that every CTA's TMEM allocation succeeds at once
  const uint32_t per_sm = 512u / (2u * H);
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
  // tiles per CTA: about four waves of resident CTAs over the launch's tiles (counted at the
  // row length L, since the contexts are device data), 1 .. 8
  const int tiles_row = (kp.p.L + kLgRows - 1) / kLgRows;
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) sms = 1;
  const int resident = sms * (int)(232448u / (smem + 1024));
  int64_t tpc = ((int64_t)tiles_row * kp.p.T) / ((int64_t)(resident > 0 ? resident : 1) * 4);
  tpc = tpc < 1 ? 1 : (tpc > kLgMaxTilesPerCta ? kLgMaxTilesPerCta : tpc);
  LogitsKernelParams k2 = kp;
  k2.tiles_per_cta = (int)tpc;
  const dim3 grid((unsigned)((tiles_row + tpc - 1) / tpc), (unsigned)kp.p.T);
  indexer_logits_kernel<H><<<grid, kLgThreads, smem, s>>>(k2);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ top-k
constexpr int kTopkThreads = 512;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kTopkVec = 8;                          // consecutive positions per thread in the ordered pass
constexpr int kTopkChunk = kTopkThreads * kTopkVec;  // positions per ordered-pass step
constexpr int kTopkSmemKeys = 40 * 1024;             // rows up to this length keep their keys in shared memory
constexpr int kTopkCand = 8192;                      // candidates kept after the first radix pass
constexpr int kTopkBins1 = 4096;                     // first pass: the keys' top 12 bits

// Order-preserving key of a logit: larger logit, larger key; -inf and NaN map to 0 and are
// never selected; -0 is read as +0.
__device__ __forceinline__ uint32_t order_key(float x) {
  if (!(x > -INFINITY)) return 0u;
  const uint32_t u = x == 0.f ? 0u : __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Block-wide exclusive prefix sums of two per-thread counts (thread order) and their totals.
__device__ __forceinline__ void block_scan2(int a, int b, int& pa, int& pb, int& ta, int& tb, int (*wsum)[2]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int ia = a, ib = b;
  for (int o = 1; o < 32; o <<= 1) {
    const int va = __shfl_up_sync(0xffffffffu, ia, o), vb = __shfl_up_sync(0xffffffffu, ib, o);
    if (lane >= o) {
      ia += va;
      ib += vb;
    }
  }
  if (lane == 31) {
    wsum[warp][0] = ia;
    wsum[warp][1] = ib;
  }
  __syncthreads();
  int wa = 0, wb = 0, sa = 0, sb = 0;
  for (int w = 0; w < kTopkWarps; ++w) {
    const int x = wsum[w][0], y = wsum[w][1];
    wa += w < warp ? x : 0;
    wb += w < warp ? y : 0;
    sa += x;
    sb += y;
  }
  pa = wa + ia - a;
  pb = wb + ib - b;
  ta = sa;
  tb = sb;
  __syncthreads();  // wsum is reused by the next call
}

// Counts keys into `hist` by the digit (k >> shift) & (bins - 1) among those with
// (k & mask) == prefix; lanes of a warp with the same digit add once, together.
__device__ __forceinline__ void count_digit(uint32_t k, bool in, uint32_t mask, uint32_t prefix, int shift,
                                            uint32_t bins, uint32_t* hist) {
  const bool take = in && k != 0u && (k & mask) == prefix;
  if (__ballot_sync(0xffffffffu, take) == 0u) return;
  const uint32_t digit = take ? (k >> shift) & (bins - 1u) : bins;
  const uint32_t peers = __match_any_sync(0xffffffffu, digit);
  if (take && (threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&hist[digit], (uint32_t)__popc(peers));
}

// The digit holding the remaining-th largest counted key, scanning `bins` bins from the top,
// and the rank left inside it.  Every thread of the block calls it.
__device__ __forceinline__ void pick_digit(const uint32_t* hist, uint32_t bins, uint32_t remaining, int (*wsum)[2],
                                           uint32_t* s_digit, uint32_t* s_left) {
  // thread i holds bins (from the top) per*i .. per*i + per - 1
  const int per = (int)bins / kTopkThreads;  // 8 for 4096 bins, 2 for 1024
  const int tid = threadIdx.x;
  int sum = 0;
  for (int k = 0; k < per; ++k) sum += (int)hist[bins - 1 - (tid * per + k)];
  int above, pb, total, tb;
  block_scan2(sum, 0, above, pb, total, tb, wsum);
  if ((uint32_t)above < remaining && (uint32_t)(above + sum) >= remaining) {  // exactly one thread
    uint32_t cum = (uint32_t)above;
    int k = 0;
    for (; k < per - 1; ++k) {
      const uint32_t c = hist[bins - 1 - (tid * per + k)];
      if (cum + c >= remaining) break;
      cum += c;
    }
    *s_digit = bins - 1 - (uint32_t)(tid * per + k);
    *s_left = remaining - cum;
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kTopkThreads) indexer_topk_kernel(IndexerTopkParams p) {
  extern __shared__ uint32_t dyn[];  // [candidates][the row's keys when it fits]
  __shared__ uint32_t hist[kTopkBins1];
  __shared__ int wsum[kTopkWarps][2];
  __shared__ uint32_t s_digit, s_left, s_ncand;
  uint32_t* const cand = dyn;
  uint32_t* const skey = dyn + kTopkCand;
  const int t = blockIdx.x;
  const int n = max(0, min(__ldg(p.ctx_lens + t), p.L));
  const float* row = p.logits + (int64_t)t * p.stride;
  int32_t* out = p.topk + (int64_t)t * p.K;
  const int tid = threadIdx.x, lane = tid & 31;
  const bool in_smem = p.L <= kTopkSmemKeys;  // the launch gives L keys of shared memory then
  auto key_at = [&](int i) -> uint32_t { return in_smem ? skey[i] : order_key(__ldg(row + i)); };
  const int n_round = (n + kTopkThreads - 1) / kTopkThreads * kTopkThreads;  // warp-uniform loop bound

  for (int i = tid; i < kTopkBins1; i += kTopkThreads) hist[i] = 0u;
  if (tid == 0) s_ncand = 0u;
  __syncthreads();
  // one read of the row (four vector loads in flight per thread where aligned): keys into
  // shared memory, the count of finite logits, and the first pass's histogram (top 12 bits)
  int cnt = 0;
  const bool vec = (reinterpret_cast<uintptr_t>(row) & 15u) == 0;
  constexpr int kU = 4;
  for (int b0 = 0; b0 < n; b0 += kTopkThreads * 4 * kU) {
    float v[kU][4];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int i0 = b0 + (u * kTopkThreads + tid) * 4;
      if (vec && i0 + 4 <= n) {
        const float4 f = __ldg(reinterpret_cast<const float4*>(row + i0));
        v[u][0] = f.x; v[u][1] = f.y; v[u][2] = f.z; v[u][3] = f.w;
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) v[u][k] = i0 + k < n ? __ldg(row + i0 + k) : -INFINITY;
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int i0 = b0 + (u * kTopkThreads + tid) * 4;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t key = order_key(v[u][k]);
        if (in_smem && i0 + k < n) skey[i0 + k] = key;
        cnt += key != 0u;
        count_digit(key, i0 + k < n, 0u, 0u, 20, kTopkBins1, hist);
      }
    }
  }
  int total;
  {
    int pa, pb, tb;
    block_scan2(cnt, 0, pa, pb, total, tb, wsum);
  }

  uint32_t tau = 0u;      // key of the K-th largest logit (0: take every finite one)
  int need_eq = 0;        // positions equal to tau to take
  if (total > p.K) {
    pick_digit(hist, kTopkBins1, (uint32_t)p.K, wsum, &s_digit, &s_left);
    uint32_t prefix = s_digit << 20, mask = 0xFFF00000u;
    uint32_t remaining = s_left;
    // the keys under the chosen 12-bit digit, compacted (unordered) if they fit
    for (int i = tid; i < n_round; i += kTopkThreads) {
      const uint32_t k = i < n ? key_at(i) : 0u;
      const bool c = k != 0u && (k & mask) == prefix;
      const uint32_t bal = __ballot_sync(0xffffffffu, c);
      if (bal == 0u) continue;
      uint32_t base = 0u;
      if (lane == 0) base = atomicAdd(&s_ncand, (uint32_t)__popc(bal));
      base = __shfl_sync(0xffffffffu, base, 0);
      const uint32_t at = base + __popc(bal & ((1u << lane) - 1u));
      if (c && at < (uint32_t)kTopkCand) cand[at] = k;
    }
    __syncthreads();
    const uint32_t ncand = s_ncand;
    const bool compact = ncand <= (uint32_t)kTopkCand;
    // two more passes of 10 bits, over the candidates (or the whole row if they did not fit)
    for (int shift = 10; shift >= 0; shift -= 10) {
      for (int i = tid; i < 1024; i += kTopkThreads) hist[i] = 0u;
      __syncthreads();
      const int m = compact ? (int)ncand : n;
      const int m_round = (m + kTopkThreads - 1) / kTopkThreads * kTopkThreads;
      for (int i = tid; i < m_round; i += kTopkThreads) {
        const uint32_t k = i < m ? (compact ? cand[i] : key_at(i)) : 0u;
        count_digit(k, i < m, mask, prefix, shift, 1024u, hist);
      }
      __syncthreads();
      pick_digit(hist, 1024u, remaining, wsum, &s_digit, &s_left);
      prefix |= s_digit << shift;
      mask |= 1023u << shift;
      remaining = s_left;
      __syncthreads();
    }
    tau = prefix;
    need_eq = (int)remaining;
  }
  const int n_gt = total > p.K ? p.K - need_eq : total;  // positions strictly above tau (all finite if none)
  // ordered pass: positions above tau ascending into [0, n_gt), then the lowest positions
  // equal to tau into [n_gt, K); each thread takes kTopkVec consecutive positions per step
  int base_gt = 0, base_eq = 0;
  for (int c0 = 0; c0 < n; c0 += kTopkChunk) {
    const int i0 = c0 + tid * kTopkVec;
    uint32_t keys[kTopkVec];
    int cg = 0, ce = 0;
#pragma unroll
    for (int k = 0; k < kTopkVec; ++k) {
      keys[k] = i0 + k < n ? key_at(i0 + k) : 0u;
      cg += keys[k] != 0u && keys[k] > tau;
      ce += tau != 0u && keys[k] == tau;
    }
    int og, oe, tg, te;
    block_scan2(cg, ce, og, oe, tg, te, wsum);
    og += base_gt;
    oe += base_eq;
#pragma unroll
    for (int k = 0; k < kTopkVec; ++k) {
      if (keys[k] != 0u && keys[k] > tau) out[og++] = i0 + k;
      else if (tau != 0u && keys[k] == tau) {
        if (oe < need_eq) out[n_gt + oe] = i0 + k;
        ++oe;
      }
    }
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
  // shared memory for the candidates and the keys of the longest row that fits (longer rows
  // are read from global memory on every pass)
  const int keys = p.L <= kTopkSmemKeys ? p.L : 0;
  const int smem = (kTopkCand + keys) * 4;
  static thread_local bool done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !done[dev]) {
    e = cudaFuncSetAttribute(indexer_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (kTopkCand + kTopkSmemKeys) * 4);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) done[dev] = true;
  }
  indexer_topk_kernel<<<(unsigned)p.T, kTopkThreads, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace smd
