// The indexer step's scoring kernel (the key gather and the top-k are in k_indexer.cu):
//
//   indexer_logits_kernel: the fp8 paged MQA logits (vLLM PR #41217 report, "实现拆解"
//     item 6: one kernel for the per-head scores and their weighted sum).  The pages print
//     no formula; the reading here is logit[t, s] = scale_s * sum_h w[t, h] * max(0,
//     q[t, h, :] . k_s) with e4m3 q and k (a per-head stage before the sum implies a
//     per-head non-linearity, taken as the rectifier).  One CTA per token and 1-8 tiles of
//     128 positions: a TMA warp reads the pages of all its tiles at once (its lanes, one
//     round trip) and streams the key rows (one 3-D box per page of the 128B-swizzled
//     [page][position][128 bytes] view of layout 0) through a 4-stage ring
//     and loads the token's query heads; an MMA warp issues four tcgen05.mma.kind::f8f6f4
//     per tile (M = 128 positions, N = H heads, K = 32 bytes each) into one of two TMEM
//     buffers; four warps read their 32 positions' H head scores back, rectify, weight,
//     sum and scale them.  Positions at or past the token's context, and positions whose
//     request, block or page is invalid, get -inf.  The step is bound by reading the key
//     cache (132 bytes per position against 2 * 128 * H flops on the tensor cores).
#include <cuda.h>

#include "smd_device.cuh"
#include "smd_internal.h"

namespace smd {
namespace {

// ------------------------------------------------------------------ paged MQA logits
constexpr int kLgRows = 128;        // positions per tile (UMMA M)
constexpr int kLgDim = 128;         // key / query bytes per row (one 128-byte swizzled row)
constexpr int kLgMaxTilesPerCta = 8;  // tiles of one token per CTA, at most (the launch picks 1..8)
constexpr int kLgStages = 4;        // key tiles in flight per CTA
constexpr int kLgThreads = 192;     // warps 0-3 epilogue (one TMEM lane quarter each), 4 TMA, 5 MMA
constexpr int kLgTmaWarp = 4, kLgMmaWarp = 5;
constexpr uint32_t kLgKBytes = kLgRows * kLgDim;  // 16 KB key tile

constexpr int kLgMaxPages = kLgMaxTilesPerCta * kLgRows / 8;  // pages a CTA's tiles span, at most (P >= 8)
__host__ __device__ constexpr uint32_t lg_smem_used(int H) {
  return kLgStages * kLgKBytes + (uint32_t)H * kLgDim + (uint32_t)H * 4 + 256 + kLgMaxPages * 4;
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
static_assert(sizeof(LgBars) <= 256, "the barriers fit the 256 bytes before the page list");

// One CTA per (token, 1-8 tiles of 128 positions): a TMA warp streams the key tiles through
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
  grid_dep_wait();  // launched as a programmatic dependent of the previous kernel
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
  int32_t* const sPage = reinterpret_cast<int32_t*>(reinterpret_cast<uint8_t*>(bars) + 256);  // the TMA warp's page list
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
    // the pages of all the CTA's tiles, read by the warp's lanes at once (one round trip)
    // rather than by the issuing lane box by box
    const int ppt = kLgRows / p.P;  // pages per tile (P divides 128)
    for (int g = lane; g < ntiles * ppt; g += 32) sPage[g] = page_of(tile0 * kLgRows + g * p.P);
    __syncwarp();
    for (int i = 0; i < ntiles; ++i) {
      const int s = i % kLgStages;
      if (i >= kLgStages && !wait(&bars->empty[s], ((i / kLgStages) - 1) & 1)) {
        if (lane == 0) give_up();
        break;
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars->full[s], kLgKBytes);
        // one box per page of the tile (P divides 128); an invalid page reads as zeros
        for (int j = 0; j < ppt; ++j)
          tma_load_3d(smem_u32(sK + s * kLgKBytes) + j * p.P * kLgDim, &kp.kmap, 0, 0, sPage[i * ppt + j],
                      &bars->full[s]);
      }
      __syncwarp();
      ++issued;
    }
    // every key tile issued has landed before the CTA may leave (2 s bound: work in flight)
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
    // this thread's position in each of the CTA's tiles: its page and scale (layout 0: the
    // page's float32 scales follow its keys), all read up front so that their two
    // dependent round trips are paid once per CTA rather than once per tile
    int32_t pgs[kLgMaxTilesPerCta];
    float scs[kLgMaxTilesPerCta];
#pragma unroll
    for (int i = 0; i < kLgMaxTilesPerCta; ++i) {
      const int pos = (tile0 + i) * kLgRows + tid;
      pgs[i] = i < ntiles && pos < ctx ? page_of(pos) : -1;
    }
#pragma unroll
    for (int i = 0; i < kLgMaxTilesPerCta; ++i) {
      const int pos = (tile0 + i) * kLgRows + tid;
      scs[i] = pgs[i] >= 0 ? __ldg(reinterpret_cast<const float*>(p.cache + (int64_t)pgs[i] * p.P * (kLgDim + 4) +
                                                                   (int64_t)p.P * kLgDim + 4 * (pos % p.P)))
                           : 0.f;
    }
#pragma unroll
    for (int i = 0; i < kLgMaxTilesPerCta; ++i) {
      if (i >= ntiles) break;
      const int b = i & 1;
      const int pos = (tile0 + i) * kLgRows + tid;
      const bool valid = pgs[i] >= 0;
      const float sc = scs[i];
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
  // tiles per CTA: about two waves of resident CTAs over the launch's tiles (counted at the
  // row length L, since the contexts are device data), 1 .. 8
  const int tiles_row = (kp.p.L + kLgRows - 1) / kLgRows;
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) sms = 1;
  const int resident = sms * (int)(232448u / (smem + 1024));
  int64_t tpc = ((int64_t)tiles_row * kp.p.T) / ((int64_t)(resident > 0 ? resident : 1) * 2);
  tpc = tpc < 1 ? 1 : (tpc > kLgMaxTilesPerCta ? kLgMaxTilesPerCta : tpc);
  LogitsKernelParams k2 = kp;
  k2.tiles_per_cta = (int)tpc;
  const dim3 grid((unsigned)((tiles_row + tpc - 1) / tpc), (unsigned)kp.p.T);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kLgThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];  // a programmatic dependent of the previous kernel (grid_dep_wait above)
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, indexer_logits_kernel<H>, k2);
}

}  // namespace

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

}  // namespace smd
