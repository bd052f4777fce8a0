// Fused row gather -> dequant -> tcgen05 partial attention for sparse MLA decode.
//
// What it computes (vLLM PR #52212 report, "实现拆解" item 1; SGLang PR #26208 report,
// _unified_sparse_decode_kernel interface Q, KV, Mask, AttnSink, Output, LSE, sm_scale):
// for token t and split s, over the split's gathered entries e (128-row tiles of the
// converted slot list), s[h,e] = scale * q[t,h,:] . k_e with one 512-wide dot for all
// heads, invalid entries masked, online softmax, o[h,:] = sum_e p[h,e] k_e over the same
// 512-wide latent (K = V).  One split: the sink logit joins the denominator and bf16 out
// + lse are written directly.  Several splits: the split's normalised o and its lse (no
// sink) go to the workspace for the combine kernel.
//
// GB300 mapping.  Heads are the UMMA M dimension (zero-padded to 128; M = 64 UMMAs run
// at half rate on this part, so nothing is lost by padding).  The O accumulator of 128
// heads x 512 dims in fp32 would fill all 512 TMEM columns, so a (token, split) is owned
// by a cluster of two CTAs, CTA c holding latent dims [256c, 256c+256) of K/V and of O:
//
//   TMEM (per CTA, 512 columns): Q half [0,128) as the A operand of QK (bf16 pairs), the
//   S partial [128,256), the O half [256,512).
//   SMEM: 2 stages x [128 rows x 256 dims] bf16 (128B-swizzled, 64 KB each), P as bf16
//   [128 heads x 128 rows] (32 KB, the A operand of PV), and a 33 KB buffer receiving the
//   peer's partial scores.
//
// Per 128-row tile j: producer warps gather the CTA's half of each 584-byte row with
// 16-byte loads (all in flight before the stage is needed) and dequantise it into the
// swizzled stage; S_c = Q_c K_c^T (M128 N128 K256, A from TMEM); the softmax threads load
// S_c into registers, which frees the S columns at once so QK of tile j+1 overlaps the rest
// of tile j; they send S_c to the peer over DSMEM and add the peer's partial, so both
// CTAs hold the 512-wide scores; online softmax; P to shared memory; O_c += P V_c
// (M128 N256 K128, the stage read MN-major).  Every QK flop is done once across the pair.
//
// The exchanged partials travel as int16 fixed point scaled by the largest magnitude of
// each (head, 64-column half): the absolute error of a received partial is at most
// max|partial| * 2^-16 (the scores keep fp32 accumulation on both sides; P itself is
// rounded to bf16 afterwards, a 2^-9 relative step).  This halves the DSMEM traffic that
// bounds the tile rate.  The running max only moves when it grows by more than 2^8, so the
// O accumulator is rarely rescaled.
//
// Roles: warps 0-7 softmax + epilogue (two threads per head, 64 score columns each;
// thread 0 also issues the UMMAs and warp 0 owns the TMEM allocation), warps 8-11
// gather/dequant.  Every wait is bounded; a wait that gives up records bit 0 in the
// status word and the CTA winds down (draining its UMMAs, freeing TMEM).
#include "smd_device.cuh"
#include "smd_internal.h"

namespace smd {
namespace {

constexpr int kTile = kTileRows;            // 128 gathered rows per tile
constexpr int kDHalf = 256;                 // latent dims per CTA
constexpr int kStages = 2;
constexpr int kSoftmaxThreads = 256;        // warps 0-7
constexpr int kThreads = kSoftmaxThreads + 128;  // + producer warps 8-11
constexpr uint32_t kSlab = kTile * 128;     // [128 rows x 64 dims] bf16 = 16 KB
constexpr uint32_t kStageBytes = 4 * kSlab; // 64 KB
constexpr uint32_t kOffP = kStages * kStageBytes;        // P: 2 slabs [128 heads x 64 rows]
constexpr uint32_t kOffXchg = kOffP + 2 * kSlab;         // peer partials: [128 heads][256 B]
constexpr uint32_t kXchgBytes = 128 * 256;
constexpr uint32_t kOffXscale = kOffXchg + kXchgBytes;   // peer partial scales [2][128] f32
constexpr uint32_t kOffMisc = kOffXscale + 2 * 128 * 4;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColQ = 0, kColS = 128, kColO = 256;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far beyond any legitimate wait
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: p <= 2^8 between rescales
constexpr float kQMax = 32767.f;           // int16 fixed-point range of the exchanged partials

struct Misc {
  uint64_t kfull[kStages];   // producers -> issuer: stage filled (128 arrivals)
  uint64_t kempty[kStages];  // PV commit -> producers: stage consumed
  uint64_t sfull;            // QK commit -> softmax: S partial ready
  uint64_t sfree;            // softmax -> issuer: S loaded into registers (256 arrivals)
  uint64_t pfull;            // softmax -> issuer: P in shared memory, O rescaled (256 arrivals)
  uint64_t pvdone;           // PV commit -> softmax: P buffer and O free again
  uint64_t xfull;            // peer softmax -> softmax: peer partial in xchg (256 remote arrivals)
  uint64_t xempty;           // peer softmax -> softmax: peer drained our writes (256 remote arrivals)
  uint64_t odone;            // last PV commit -> softmax: O final
  uint64_t drain;            // issuer self-drain before TMEM is freed after a failed wait
  uint64_t sgrp;             // softmax-group rendezvous (256 arrivals per use)
  uint64_t hpair[128];       // per-head rendezvous of the two threads of a head (2 arrivals)
  uint32_t tmem_base;
  uint32_t abort;
  uint32_t mask[kStages][4];        // valid-row bit masks of the staged tile
  float red[kStages][2][128];       // per-column-half tile maxima, then final denominators
};
constexpr uint32_t kSmemBytes = kOffMisc + sizeof(Misc) + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");

__device__ __forceinline__ float ex2(float x) { return fast_exp2(x); }

__device__ __forceinline__ bool aborted(const Misc* m) {
  return *reinterpret_cast<const volatile uint32_t*>(&m->abort) != 0u;
}

// Bounded wait that also gives up early once another role of this CTA has aborted.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, const Misc* m,
                                         bool cluster_acquire = false) {
  auto poll = [&]() { return cluster_acquire ? mbar_try_wait_acq_cluster(bar, parity) : mbar_try_wait(bar, parity); };
  if (poll()) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!poll()) {
    if (aborted(m) || globaltimer_ns() - t0 > kWaitLimitNs) return false;
  }
  return true;
}

__device__ __forceinline__ void record_abort(Misc* m, uint32_t* status) {
  atomicExch(&m->abort, 1u);
  if (status != nullptr) atomicOr(status, 1u);
}

// Byte offset of the 16-byte chunk holding local dims [d0, d0+8) of `row` in a stage
// made of four 128B-swizzled [128 rows x 64 dims] slabs.
__device__ __forceinline__ uint32_t stage_off(uint32_t row, uint32_t d0) {
  return (d0 >> 6) * kSlab + sw128_off(row, (d0 & 63) >> 3);
}

// int16 pair packing of two scaled partials (round to nearest; |v| <= 32767 by construction).
__device__ __forceinline__ uint32_t pack_q16(float a, float b) {
  const int32_t ia = __float2int_rn(a), ib = __float2int_rn(b);
  return (uint32_t)(ia & 0xFFFF) | ((uint32_t)ib << 16);
}
__device__ __forceinline__ float lo_q16(uint32_t w) { return (float)(int32_t)(int16_t)(w & 0xFFFFu); }
__device__ __forceinline__ float hi_q16(uint32_t w) { return (float)((int32_t)w >> 16); }

// Gather + dequantise this CTA's half of 128 rows.  Half 0: NoPE bytes [0,256) with scale
// codes 0..3 (16 chunks of 16 bytes per row).  Half 1: NoPE bytes [256,448) with codes
// 4..6 (12 chunks), then the 64 RoPE values (8 chunks).  Jobs are (row, chunk) pairs
// with consecutive threads on consecutive chunks of a row, so each warp load reads whole
// contiguous row segments and all lanes of a warp take the same path.  `issue` puts every
// load of the tile in flight (invalid rows read slot 0 and are zeroed later); `store`
// converts and writes the swizzled stage.
template <int HALF>
struct Gather {
  static constexpr int NN = HALF == 0 ? 16 : 12;  // NoPE chunks per row
  static constexpr int NR = HALF == 0 ? 0 : 8;    // RoPE chunks per row
  static constexpr int JN = NN;                   // NoPE jobs per thread (128 * NN / 128)
  static constexpr int JR = NR;                   // RoPE jobs per thread
  static constexpr int NOPE_BYTE0 = HALF == 0 ? 0 : 256;
  static constexpr int CODE0 = HALF == 0 ? 0 : 4;
  uint4 raw[JN + JR];
  uint32_t code[JN];
  int32_t slot[JN + JR];

  __device__ __forceinline__ static void job(int i, int ptid, int& row, int& ch) {
    if (i < JN) {
      const int k = i * 128 + ptid;
      row = k / NN;
      ch = k - row * NN;
    } else {
      const int k = (i - JN) * 128 + ptid;
      row = k >> 3;
      ch = k & 7;
    }
  }

  template <bool ALIGN16>
  __device__ __forceinline__ void issue(const int32_t* gidx_tile, int rows_left, int64_t n_slots,
                                        const CacheView& cv, int ptid) {
#pragma unroll
    for (int i = 0; i < JN + JR; ++i) {
      int row, ch;
      job(i, ptid, row, ch);
      const int32_t g = row < rows_left ? ldg_nc_s32(gidx_tile + row) : -1;
      slot[i] = ((int64_t)g >= n_slots) ? -1 : g;
    }
#pragma unroll
    for (int i = 0; i < JN + JR; ++i) {
      int row, ch;
      job(i, ptid, row, ch);
      const int32_t g = slot[i] >= 0 ? slot[i] : 0;
      int32_t page, off;
      slot_page_off(cv, g, page, off);
      const uint8_t* pg = cv.base + (int64_t)page * cv.page_bytes;
      const uint8_t* d = pg + (int64_t)off * kDataBytes;
      if (i < JN) {
        raw[i] = ldg16_early<ALIGN16>(d + NOPE_BYTE0 + ch * 16);
        code[i] = ldg_nc_u8(pg + cv.scale_start + (int64_t)off * kScaleBytes + CODE0 + (ch >> 2));
      } else {
        raw[i] = ldg16_early<ALIGN16>(d + kNope + ch * 16);
      }
    }
  }

  __device__ __forceinline__ void store(uint8_t* st, int ptid) const {
#pragma unroll
    for (int i = 0; i < JN + JR; ++i) {
      int row, ch;
      job(i, ptid, row, ch);
      const bool valid = slot[i] >= 0;
      if (i >= JN) {
        const uint4 v = valid ? scrub_bf16x8(raw[i]) : make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(st + stage_off(row, 192 + ch * 8)) = v;
      } else {
        uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
        if (valid) dequant16(raw[i], ue8m0_to_float(code[i]), lo, hi);
        *reinterpret_cast<uint4*>(st + stage_off(row, ch * 16)) = lo;
        *reinterpret_cast<uint4*>(st + stage_off(row, ch * 16 + 8)) = hi;
      }
    }
  }
};

// The producer role: for every tile, put the loads in flight, then wait for the stage to
// be free, publish the tile's valid-row mask, convert, and signal the UMMA issuer.
template <int HALF, bool ALIGN16>
__device__ __forceinline__ void produce(uint8_t* smem, Misc* m, const AttnParams& p, const int32_t* gidx_t,
                                        int tile_begin, int n, int ptid, int pwarp, int lane) {
  const CacheView cv = make_cache_view(p.cache, p.P);
  const int64_t n_slots = p.num_pages * p.P;
  Gather<HALF> gth;
  for (int j = 0; j < n; ++j) {
    const int s = j & 1;
    const int u = j >> 1;
    const int row0 = (tile_begin + j) * kTile;
    const int rows_left = p.N - row0;
    gth.template issue<ALIGN16>(gidx_t + row0, rows_left, n_slots, cv, ptid);
    int32_t g = ptid < rows_left ? ldg_nc_s32(gidx_t + row0 + ptid) : -1;
    if ((int64_t)g >= n_slots) g = -1;
    if (u > 0 && !wait_bar(&m->kempty[s], (u - 1) & 1, m)) {
      record_abort(m, p.status);
      return;
    }
    const uint32_t bits = __ballot_sync(0xffffffffu, g >= 0);
    if (lane == 0) m->mask[s][pwarp] = bits;
    gth.store(smem + s * kStageBytes, ptid);
    fence_async_smem();
    mbar_arrive(&m->kfull[s]);
  }
}

}  // namespace

template <bool ALIGN16>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1) attn_pair_kernel(AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sP = smem + kOffP;
  uint8_t* xchg = smem + kOffXchg;
  float* xscale = reinterpret_cast<float*>(smem + kOffXscale);
  Misc* m = reinterpret_cast<Misc*>(smem + kOffMisc);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const uint32_t half = cluster_rank();   // == blockIdx.x & 1
  const uint32_t peer = half ^ 1u;
  const int split = blockIdx.x >> 1;
  const int t = blockIdx.y;
  const int N = p.N;
  const int n_tiles_tok = (N + kTile - 1) / kTile;
  const int tile_begin = split * p.tiles_per_split;
  const int n = max(0, min(n_tiles_tok, tile_begin + p.tiles_per_split) - tile_begin);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&m->kfull[s], 128);
      mbar_init(&m->kempty[s], 1);
    }
    mbar_init(&m->sfull, 1);
    mbar_init(&m->sfree, kSoftmaxThreads);
    mbar_init(&m->pfull, kSoftmaxThreads);
    mbar_init(&m->pvdone, 1);
    mbar_init(&m->xfull, kSoftmaxThreads);
    mbar_init(&m->xempty, kSoftmaxThreads);
    mbar_init(&m->odone, 1);
    mbar_init(&m->drain, 1);
    mbar_init(&m->sgrp, kSoftmaxThreads);
    m->abort = 0;
    fence_mbar_init();
  }
  if (tid < 128) mbar_init(&m->hpair[tid], 2);
  if (warp == 0) {
    tmem_alloc(&m->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (tid < 128) fence_mbar_init();
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // the peer's barriers exist before anyone arrives on them remotely
  tc_fence_after();
  const uint32_t tmem = m->tmem_base;

  if (warp < 8) {
    // ------------------------------------------------------------ softmax + UMMA issue
    // Thread (h, hc): head h = TMEM lane h, column half hc of every 128-column tile.
    const int h = tid & 127;
    const int hc = warp >> 2;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const bool issuer = tid == 0;
    constexpr uint32_t kIdescQK = idesc_bf16_f32(128, kTile, false, false);
    constexpr uint32_t kIdescPV = idesc_bf16_f32(128, kDHalf, false, true);
    const uint32_t a_stage = smem_u32(smem);
    const uint32_t a_p = smem_u32(sP);
    bool ok = true;
    uint32_t sgrp_phase = 0;
    {  // this thread's half of head h's Q half -> TMEM columns [64 hc, 64 hc + 64) of lane h
      const uint8_t* qrow = static_cast<const uint8_t*>(p.q) + ((int64_t)t * p.H + h) * (kLatent * 2) +
                            half * (kDHalf * 2) + hc * 256;
      uint32_t r[2][32];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const uint4 v = h < p.H ? ldg_nc_v4(qrow + i * 16) : make_uint4(0, 0, 0, 0);
        r[i >> 3][(i & 7) * 4 + 0] = v.x;
        r[i >> 3][(i & 7) * 4 + 1] = v.y;
        r[i >> 3][(i & 7) * 4 + 2] = v.z;
        r[i >> 3][(i & 7) * 4 + 3] = v.w;
      }
      tmem_st32(tmem + lane_base + kColQ + hc * 64, r[0]);
      tmem_st32(tmem + lane_base + kColQ + hc * 64 + 32, r[1]);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&m->sgrp);
      ok = wait_bar(&m->sgrp, sgrp_phase, m);
      sgrp_phase ^= 1u;
      tc_fence_after();
    }
    auto issue_qk = [&](int j) {  // S = Q K^T for tile j
      const uint32_t base = a_stage + (j & 1) * kStageBytes;
#pragma unroll
      for (int kk = 0; kk < kDHalf / 16; ++kk)
        umma_ts(tmem + kColS, tmem + kColQ + kk * 8, desc_sw128(base + (kk >> 2) * kSlab + (kk & 3) * 32, 16, 1024),
                kIdescQK, kk > 0 ? 1u : 0u);
      umma_commit(&m->sfull);
    };
    auto issue_pv = [&](int j) {  // O += P V for tile j, then free its stage and P
      const uint32_t base = a_stage + (j & 1) * kStageBytes;
#pragma unroll
      for (int kk = 0; kk < kTile / 16; ++kk)
        umma_ss(tmem + kColO, desc_sw128(a_p + (kk >> 2) * kSlab + (kk & 3) * 32, 16, 1024),
                desc_sw128(base + kk * 2048, kSlab, 1024), kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
      umma_commit(&m->kempty[j & 1]);
      umma_commit(&m->pvdone);
    };
    if (ok && issuer && n > 0) {
      if ((ok = wait_bar(&m->kfull[0], 0, m))) {
        tc_fence_after();
        issue_qk(0);
      }
    }
    __syncwarp();

    const uint32_t peer_xchg_row = mapa(smem_u32(xchg + h * 256), peer);
    const uint32_t peer_xscale = mapa(smem_u32(xscale + hc * 128 + h), peer);
    const uint32_t peer_xfull = mapa(smem_u32(&m->xfull), peer);
    const uint32_t peer_xempty = mapa(smem_u32(&m->xempty), peer);
    const uint8_t* my_xchg_row = xchg + h * 256;
    const float sl2 = p.scale * kLog2e;
    float m_ref = -INFINITY;  // reference max (log2 domain) the weights are taken against
    float l_run = 0.f;        // this thread's share of the denominator relative to m_ref

    for (int j = 0; j < n && ok; ++j) {
      const int s = j & 1;
      if (!(ok = wait_bar(&m->sfull, j & 1, m))) break;
      tc_fence_after();
      float x[64];
#pragma unroll
      for (int c2 = 0; c2 < 2; ++c2) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_base + kColS + hc * 64 + c2 * 32, r);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) x[c2 * 32 + i] = __uint_as_float(r[i]);
      }
      // S is in registers: the issuer may start QK of the next tile right away.
      tc_fence_before();
      mbar_arrive(&m->sfree);
      if (issuer && j + 1 < n) {
        if ((ok = wait_bar(&m->sfree, j & 1, m)) && (ok = wait_bar(&m->kfull[(j + 1) & 1], ((j + 1) >> 1) & 1, m))) {
          tc_fence_after();
          issue_qk(j + 1);
        }
      }
      __syncwarp();
      if (!ok) break;

      // Send this half of the partial scores to the peer as int16 fixed point.
      float amax = 0.f;
#pragma unroll
      for (int c = 0; c < 64; ++c) amax = fmaxf(amax, fabsf(x[c]));
      const float enc = amax > 0.f ? kQMax / amax : 0.f;
      if (j > 0 && !(ok = wait_bar(&m->xempty, (j - 1) & 1, m, true))) break;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t ch = hc * 8 + i;
        uint32_t w[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) w[q] = pack_q16(x[i * 8 + 2 * q] * enc, x[i * 8 + 2 * q + 1] * enc);
        st_cluster_v4(peer_xchg_row + ((ch ^ (h & 7)) << 4), w[0], w[1], w[2], w[3]);
      }
      asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(peer_xscale), "f"(amax / kQMax) : "memory");
      mbar_arrive_cluster(peer_xfull);
      if (!(ok = wait_bar(&m->xfull, j & 1, m, true))) break;
      const float dec = xscale[hc * 128 + h];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t ch = hc * 8 + i;
        const uint4 v = *reinterpret_cast<const uint4*>(my_xchg_row + ((ch ^ (h & 7)) << 4));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          x[i * 8 + 2 * q] = fmaf(lo_q16(w[q]), dec, x[i * 8 + 2 * q]);
          x[i * 8 + 2 * q + 1] = fmaf(hi_q16(w[q]), dec, x[i * 8 + 2 * q + 1]);
        }
      }
      mbar_arrive_cluster(peer_xempty);

      // Online softmax over this thread's 64 columns; both threads of head h agree on m_ref.
      const uint32_t mk0 = m->mask[s][2 * hc], mk1 = m->mask[s][2 * hc + 1];
      float lmax = -INFINITY;
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        const uint32_t bits = c < 32 ? mk0 : mk1;
        const float v = ((bits >> (c & 31)) & 1u) ? x[c] * sl2 : -INFINITY;
        x[c] = v;
        lmax = fmaxf(lmax, v);
      }
      m->red[s][hc][h] = lmax;
      mbar_arrive(&m->hpair[h]);
      if (!(ok = wait_bar(&m->hpair[h], j & 1, m))) break;
      const float tmax = fmaxf(lmax, m->red[s][hc ^ 1][h]);
      float alpha = 1.f;
      const bool upd = tmax > m_ref + kRescaleThreshold;  // false while everything is masked
      if (upd) {
        alpha = ex2(m_ref - tmax);  // 0 when m_ref is -inf
        m_ref = tmax;
      }
      float psum = 0.f;
      uint32_t pk[32];
      if (m_ref == -INFINITY) {
#pragma unroll
        for (int i = 0; i < 32; ++i) pk[i] = 0u;
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float p0 = ex2(x[2 * i] - m_ref), p1 = ex2(x[2 * i + 1] - m_ref);
          psum += p0 + p1;  // the denominator keeps the unrounded weights
          pk[i] = bf16x2_bits(__floats2bfloat162_rn(p0, p1));
        }
      }
      l_run = l_run * alpha + psum;
      // P buffer and O are free once PV of the previous tile is done.
      if (j > 0 && !(ok = wait_bar(&m->pvdone, (j - 1) & 1, m))) break;
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4*>(sP + hc * kSlab + sw128_off(h, c)) =
            make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      if (j > 0 && __any_sync(0xffffffffu, upd)) {
#pragma unroll 1
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t o[32];
          const uint32_t col = kColO + hc * 128 + cc * 32;
          tmem_ld32(tmem + lane_base + col, o);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st32(tmem + lane_base + col, o);
        }
        tmem_wait_st();
      }
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(&m->pfull);
      if (issuer) {
        if ((ok = wait_bar(&m->pfull, j & 1, m))) {
          tc_fence_after();
          issue_pv(j);
          if (j + 1 == n) umma_commit(&m->odone);
        }
      }
      __syncwarp();
      ok = ok && !aborted(m);
    }
    if (issuer && n == 0) mbar_arrive(&m->odone);
    if (ok) ok = wait_bar(&m->odone, 0, m);
    if (!ok) {
      record_abort(m, p.status);
      if (issuer) {
        umma_commit(&m->drain);  // let issued UMMAs land before TMEM is freed
        mbar_wait_bounded(&m->drain, 0, kWaitLimitNs);
      }
    } else {
      // Epilogue: head h, local dims [128 hc, 128 hc + 128) of this CTA's 256.
      m->red[0][hc][h] = l_run;  // every use of red[][] by the loop is over (odone)
      mbar_arrive(&m->sgrp);
      ok = wait_bar(&m->sgrp, sgrp_phase, m);
      sgrp_phase ^= 1u;
    }
    if (!ok) {
      record_abort(m, p.status);
    } else {
      const float l_tot = l_run + m->red[0][hc ^ 1][h];
      tc_fence_after();
      const bool o_live = n > 0;
      const bool head_ok = h < p.H;
      const int d0 = half * kDHalf + hc * 128;  // first output dim of this thread
      if (p.S == 1) {
        const float sink_nat = (p.sink != nullptr && head_ok) ? __ldg(p.sink + h) : -INFINITY;
        const float ms = sink_nat * kLog2e;
        const float M = fmaxf(m_ref, ms);
        float factor = 0.f, lse_v = -INFINITY;
        if (M != -INFINITY) {
          const float den = l_tot * ex2(m_ref - M) + (ms == -INFINITY ? 0.f : ex2(ms - M));
          factor = ex2(m_ref - M) / den;
          // natural-log max from whichever term set it, so a sink-only row gives lse = sink exactly
          lse_v = (M == m_ref ? m_ref * kLn2 : sink_nat) + log2f(den) * kLn2;
        }
        uint8_t* orow = static_cast<uint8_t*>(p.out) + (((int64_t)t * p.H + h) * kLatent + d0) * 2;
#pragma unroll 1
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t o[32];
          if (o_live) {
            tmem_ld32(tmem + lane_base + kColO + hc * 128 + cc * 32, o);
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
        if (head_ok && half == 0 && hc == 0 && p.lse != nullptr) p.lse[(int64_t)t * p.H + h] = lse_v;
      } else {
        const float factor = l_tot > 0.f ? 1.f / l_tot : 0.f;
        const int64_t prow = ((int64_t)t * p.S + split) * p.H + h;
        float* orow = p.o_part + prow * kLatent + d0;
#pragma unroll 1
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t o[32];
          if (o_live) {
            tmem_ld32(tmem + lane_base + kColO + hc * 128 + cc * 32, o);
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
        if (head_ok && half == 0 && hc == 0)
          p.lse_part[prow] = l_tot > 0.f ? (m_ref + log2f(l_tot)) * kLn2 : -INFINITY;
      }
    }
  } else {
    // ------------------------------------------------------------ gather + dequant
    const int ptid = tid - kSoftmaxThreads;
    const int32_t* gidx_t = p.gidx + (int64_t)t * N;
    if (half == 0)
      produce<0, ALIGN16>(smem, m, p, gidx_t, tile_begin, n, ptid, warp - 8, lane);
    else
      produce<1, ALIGN16>(smem, m, p, gidx_t, tile_begin, n, ptid, warp - 8, lane);
  }

  // Wind down: nobody may leave while the peer can still write into this CTA's shared
  // memory, and TMEM is freed only after every tcgen05 access of this CTA is done.
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
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
    e = align16 ? cudaFuncSetAttribute(attn_pair_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kSmemBytes)
                : cudaFuncSetAttribute(attn_pair_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_done[align16][dev] = true;
  }
  const dim3 grid(2 * p.S, p.T);
  if (align16)
    attn_pair_kernel<true><<<grid, kThreads, kSmemBytes, s>>>(p);
  else
    attn_pair_kernel<false><<<grid, kThreads, kSmemBytes, s>>>(p);
  return cudaGetLastError();
}

}  // namespace smd
