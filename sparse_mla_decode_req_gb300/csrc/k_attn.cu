// Fused row gather -> dequant -> tcgen05 partial attention for sparse MLA decode.
//
// What it computes (vLLM PR #52212 report, "实现拆解" item 1; SGLang PR #26208 report,
// _unified_sparse_decode_kernel interface Q, KV, Mask, AttnSink, Output, LSE, sm_scale):
// for token t and split s, over the split's gathered entries e (64-row tiles of the
// converted slot list), s[h,e] = scale * q[t,h,:] . k_e with one 512-wide dot for all
// heads, invalid entries masked, online softmax, o[h,:] = sum_e p[h,e] k_e over the same
// 512-wide latent (K = V).  One split: the sink logit joins the denominator here and
// bf16 out + lse are written directly.  Several splits: the split's normalised o and
// its lse (no sink) go to the workspace for the combine kernel.
//
// GB300 mapping.  Heads are the MMA M dimension (zero-padded to 128).  O = 128 x 512
// fp32 would fill all 512 TMEM columns, so each (token, split) is handled by two CTAs
// that own latent dims [0,256) and [256,512) of the output: each computes the full
// 512-wide QK tile into TMEM (S, 64 columns), runs the softmax in registers (thread h =
// TMEM lane h = head h), writes P (bf16) to shared memory and accumulates its half of O
// (256 TMEM columns) with a second UMMA that reads the same dequantised tile as an
// MN-major B operand.  The gather uses 16-byte vector loads; the dequantised tile is
// written straight into the 128-byte-swizzled UMMA layout.
#include "smd_device.cuh"
#include "smd_internal.h"

namespace smd {
namespace {

constexpr int kM = 128;          // MMA M: heads, zero-padded
constexpr int kThreads = 128;    // thread h <-> TMEM lane h
constexpr int kDHalf = 256;      // output dims per CTA
constexpr uint32_t kQSlab = kM * 128;          // [128 rows x 64 dims] bf16 = 16 KB
constexpr uint32_t kKSlab = kTileRows * 128;   // [64 rows x 64 dims] bf16 = 8 KB
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + 8 * kQSlab;           // 128 KB
constexpr uint32_t kOffP = kOffK + 8 * kKSlab;           // +64 KB
constexpr uint32_t kOffMisc = kOffP + kM * 128;          // +16 KB
constexpr uint32_t kSmemBytes = kOffMisc + 512 + 1024;   // misc + alignment slack
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;
constexpr uint32_t kColO = 256;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far beyond any legitimate wait
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct Misc {
  uint64_t mma_bar;
  uint32_t tmem_base;
  uint32_t pad;
  int32_t slot[kTileRows];
};

__device__ __forceinline__ float ex2(float x) { return exp2f(x); }

}  // namespace

template <bool ALIGN16>
__global__ void __launch_bounds__(kThreads, 1) attn_partial_kernel(AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + kOffQ;
  uint8_t* sK = smem + kOffK;
  uint8_t* sP = smem + kOffP;
  Misc* misc = reinterpret_cast<Misc*>(smem + kOffMisc);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int half = blockIdx.x & 1;
  const int split = blockIdx.x >> 1;
  const int t = blockIdx.y;
  const int N = p.N;
  const int n_tiles = (N + kTileRows - 1) / kTileRows;
  const int tile_begin = split * p.tiles_per_split;
  const int tile_end = min(n_tiles, tile_begin + p.tiles_per_split);

  if (warp == 0) {
    tmem_alloc(&misc->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&misc->mma_bar, 1);
    fence_mbar_init();
  }
  // Q[t] -> shared memory, 8 swizzled K-major slabs of [128 heads x 64 dims].
  const uint8_t* q_t = static_cast<const uint8_t*>(p.q) + (int64_t)t * p.H * (kLatent * 2);
  for (int i = tid; i < kM * 64; i += kThreads) {
    const int h = i >> 6, j = i & 63;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (h < p.H) v = __ldg(reinterpret_cast<const uint4*>(q_t + h * (kLatent * 2)) + j);
    *reinterpret_cast<uint4*>(sQ + (j >> 3) * kQSlab + sw128_off(h, j & 7)) = v;
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc->tmem_base;
  const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;

  const CacheView cv{p.cache, (int64_t)p.P * kRowBytes, (int64_t)p.P * kDataBytes, p.P};
  const int32_t* gidx_t = p.gidx + (int64_t)t * N;
  const int64_t n_slots = p.num_pages * p.P;
  const float sl2 = p.scale * kLog2e;
  constexpr uint32_t kIdescQK = idesc_bf16_f32(kM, kTileRows, false, false);
  constexpr uint32_t kIdescPV = idesc_bf16_f32(kM, kDHalf, false, true);
  const uint32_t aQ = smem_u32(sQ), aK = smem_u32(sK), aP = smem_u32(sP);

  float m_run = -INFINITY;  // running max, log2 domain
  float l_run = 0.f;        // running denominator (without sink)
  bool o_live = false;      // the O accumulator holds data
  bool aborted = false;
  uint32_t phase = 0;

  for (int tile = tile_begin; tile < tile_end; ++tile) {
    const int row0 = tile * kTileRows;
    if (tid < kTileRows) {
      const int r = row0 + tid;
      int32_t g = r < N ? __ldg(gidx_t + r) : -1;
      if ((int64_t)g >= n_slots) g = -1;
      misc->slot[tid] = g;
    }
    __syncthreads();

    // Gather + dequant: 64 rows x 36 sixteen-byte input chunks (28 NoPE, 8 RoPE).
#pragma unroll 6
    for (int i = tid; i < kTileRows * 36; i += kThreads) {
      const int r = i / 36, j = i - (i / 36) * 36;
      const int32_t g = misc->slot[r];
      uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
      if (j < 28) {
        if (g >= 0) {
          const uint4 raw = ldg16<ALIGN16>(row_data(cv, g) + j * 16);
          const float sc = ue8m0_to_float(__ldg(row_scales(cv, g) + (j >> 2)));
          dequant16(raw, sc, lo, hi);
        }
        uint8_t* slab = sK + (j >> 2) * kKSlab;
        *reinterpret_cast<uint4*>(slab + sw128_off(r, (j & 3) * 2)) = lo;
        *reinterpret_cast<uint4*>(slab + sw128_off(r, (j & 3) * 2 + 1)) = hi;
      } else {
        if (g >= 0) lo = scrub_bf16x8(ldg16<ALIGN16>(row_data(cv, g) + kNope + (j - 28) * 16));
        *reinterpret_cast<uint4*>(sK + 7 * kKSlab + sw128_off(r, j - 28)) = lo;
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();

    // S = Q K^T : M=128, N=64, K=512 (32 UMMAs of K=16).
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 32; ++kk) {
        const uint32_t slab = kk >> 2, koff = (kk & 3) * 32;
        umma_ss(tmem + kColS, desc_sw128(aQ + slab * kQSlab + koff, 16, 1024),
                desc_sw128(aK + slab * kKSlab + koff, 16, 1024), kIdescQK, kk > 0 ? 1u : 0u);
      }
      umma_commit(&misc->mma_bar);
    }
    bool ok = mbar_wait_bounded(&misc->mma_bar, phase, kWaitLimitNs);
    phase ^= 1u;
    if (__syncthreads_or(!ok)) {
      aborted = true;
      break;
    }
    tc_fence_after();

    // Online softmax for head row `tid` over the 64 columns of this tile.
    uint32_t sraw[2][32];
    tmem_ld32(tmem + lane_base + kColS, sraw[0]);
    tmem_ld32(tmem + lane_base + kColS + 32, sraw[1]);
    tmem_wait_ld();
    float tmax = -INFINITY;
#pragma unroll
    for (int j = 0; j < 64; ++j) {
      const float x = misc->slot[j] >= 0 ? __uint_as_float(sraw[j >> 5][j & 31]) * sl2 : -INFINITY;
      sraw[j >> 5][j & 31] = __float_as_uint(x);
      tmax = fmaxf(tmax, x);
    }
    const float m_new = fmaxf(m_run, tmax);
    float alpha = 1.f, psum = 0.f;
    uint32_t pk[32];
    if (m_new == -INFINITY) {
#pragma unroll
      for (int i = 0; i < 32; ++i) pk[i] = 0u;
    } else {
      alpha = ex2(m_run - m_new);
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float x0 = __uint_as_float(sraw[(2 * i) >> 5][(2 * i) & 31]);
        const float x1 = __uint_as_float(sraw[(2 * i + 1) >> 5][(2 * i + 1) & 31]);
        const float p0 = ex2(x0 - m_new), p1 = ex2(x1 - m_new);
        psum += p0 + p1;  // the denominator keeps the unrounded weights
        pk[i] = bf16x2_bits(__floats2bfloat162_rn(p0, p1));
      }
    }
    l_run = l_run * alpha + psum;
    m_run = m_new;
#pragma unroll
    for (int ch = 0; ch < 8; ++ch)
      *reinterpret_cast<uint4*>(sP + sw128_off(tid, ch)) =
          make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
    // Rescale the 256 accumulator columns when any lane of the warp needs it: tcgen05.ld/st
    // are warp-collective, so the branch must be warp-uniform (lanes with alpha == 1
    // rewrite their values unchanged).
    const bool rescale = __any_sync(0xffffffffu, alpha != 1.f);
    if (o_live && rescale) {
#pragma unroll 1
      for (int cc = 0; cc < kDHalf / 32; ++cc) {
        uint32_t o[32];
        tmem_ld32(tmem + lane_base + kColO + cc * 32, o);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
        tmem_st32(tmem + lane_base + kColO + cc * 32, o);
      }
      tmem_wait_st();
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();

    // O_half += P V_half : M=128, N=256, K=64 (4 UMMAs of K=16); V is the same tile,
    // read MN-major (dims contiguous): 64-dim slabs 8 KB apart, 8-row groups 1 KB apart.
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        umma_ss(tmem + kColO, desc_sw128(aP + kk * 32, 16, 1024),
                desc_sw128(aK + (4 * half) * kKSlab + kk * 2048, kKSlab, 1024), kIdescPV,
                (o_live || kk > 0) ? 1u : 0u);
      }
      umma_commit(&misc->mma_bar);
    }
    ok = mbar_wait_bounded(&misc->mma_bar, phase, kWaitLimitNs);
    phase ^= 1u;
    if (__syncthreads_or(!ok)) {
      aborted = true;
      break;
    }
    tc_fence_after();
    o_live = true;
  }

  if (aborted) {
    // A bounded wait gave up: record it, give in-flight MMAs one more bounded chance to
    // land, free TMEM and leave without writing outputs.
    if (tid == 0 && p.status != nullptr) atomicOr(p.status, 1u);
    mbar_wait_bounded(&misc->mma_bar, phase ^ 1u, kWaitLimitNs);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
      tc_fence_after();
      tmem_dealloc(tmem, kTmemCols);
    }
    return;
  }

  // Epilogue: thread h finalises head h for this CTA's 256 output dims.
  const int h = tid;
  const bool head_ok = h < p.H;
  if (p.S == 1) {
    const float sink_nat = (p.sink != nullptr && head_ok) ? __ldg(p.sink + h) : -INFINITY;
    const float ms = sink_nat * kLog2e;
    const float M = fmaxf(m_run, ms);
    float factor = 0.f, lse_v = -INFINITY;
    if (M != -INFINITY) {
      const float den = l_run * ex2(m_run - M) + (ms == -INFINITY ? 0.f : ex2(ms - M));
      factor = ex2(m_run - M) / den;
      // natural-log max taken from whichever term set it, so a sink-only row gives lse = sink exactly
      lse_v = (M == m_run ? m_run * kLn2 : sink_nat) + log2f(den) * kLn2;
    }
    uint8_t* orow = static_cast<uint8_t*>(p.out) + ((int64_t)t * p.H + h) * (kLatent * 2) + half * (kDHalf * 2);
#pragma unroll 1
    for (int cc = 0; cc < kDHalf / 32; ++cc) {
      uint32_t o[32];
      if (o_live) {
        tmem_ld32(tmem + lane_base + kColO + cc * 32, o);
        tmem_wait_ld();
      }
      uint32_t w[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float a = o_live ? __uint_as_float(o[2 * i]) * factor : 0.f;
        const float b = o_live ? __uint_as_float(o[2 * i + 1]) * factor : 0.f;
        w[i] = bf16x2_bits(__floats2bfloat162_rn(a, b));
      }
      if (head_ok) {
        uint4* dst = reinterpret_cast<uint4*>(orow + cc * 64);
        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
        dst[2] = make_uint4(w[8], w[9], w[10], w[11]);
        dst[3] = make_uint4(w[12], w[13], w[14], w[15]);
      }
    }
    if (head_ok && half == 0 && p.lse != nullptr) p.lse[(int64_t)t * p.H + h] = lse_v;
  } else {
    const float factor = l_run > 0.f ? 1.f / l_run : 0.f;
    const int64_t prow = ((int64_t)t * p.S + split) * p.H + h;
    float* orow = p.o_part + prow * kLatent + half * kDHalf;
#pragma unroll 1
    for (int cc = 0; cc < kDHalf / 32; ++cc) {
      uint32_t o[32];
      if (o_live) {
        tmem_ld32(tmem + lane_base + kColO + cc * 32, o);
        tmem_wait_ld();
      }
      if (head_ok) {
        float4* dst = reinterpret_cast<float4*>(orow + cc * 32);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          float4 v;
          v.x = o_live ? __uint_as_float(o[4 * i + 0]) * factor : 0.f;
          v.y = o_live ? __uint_as_float(o[4 * i + 1]) * factor : 0.f;
          v.z = o_live ? __uint_as_float(o[4 * i + 2]) * factor : 0.f;
          v.w = o_live ? __uint_as_float(o[4 * i + 3]) * factor : 0.f;
          dst[i] = v;
        }
      }
    }
    if (head_ok && half == 0) p.lse_part[prow] = l_run > 0.f ? (m_run + log2f(l_run)) * kLn2 : -INFINITY;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

int attn_ctas_per_split() { return 2; }

cudaError_t launch_attn(const AttnParams& p, cudaStream_t s) {
  if (p.T == 0) return cudaSuccess;
  const bool align16 = ((int64_t)p.P * kRowBytes) % 16 == 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static bool attr_done[2][64] = {};
  if (dev < 64 && !attr_done[align16][dev]) {
    e = align16 ? cudaFuncSetAttribute(attn_partial_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kSmemBytes)
                : cudaFuncSetAttribute(attn_partial_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_done[align16][dev] = true;
  }
  const dim3 grid(2 * p.S, p.T);
  if (align16)
    attn_partial_kernel<true><<<grid, kThreads, kSmemBytes, s>>>(p);
  else
    attn_partial_kernel<false><<<grid, kThreads, kSmemBytes, s>>>(p);
  return cudaGetLastError();
}

}  // namespace smd
