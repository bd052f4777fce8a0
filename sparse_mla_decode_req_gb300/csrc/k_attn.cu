// Fused row gather -> dequant -> tcgen05 partial attention for sparse MLA decode.
//
// What it computes (vLLM PR #52212 report, "实现拆解" item 1; SGLang PR #26208 report,
// _unified_sparse_decode_kernel interface Q, KV, Mask, AttnSink, Output, LSE, sm_scale):
// for token t and split s, over the split's gathered entries e (64-row tiles of the
// converted slot list), s[h,e] = scale * q[t,h,:] . k_e with one 512-wide dot for all
// heads, invalid entries masked, online softmax, o[h,:] = sum_e p[h,e] k_e over the same
// 512-wide latent (K = V).  One split: the sink logit joins the denominator and bf16 out
// + lse are written directly.  Several splits: the split's normalised o and its lse (no
// sink) go to the workspace for the combine kernel.
//
// GB300 mapping.  Heads are the UMMA M dimension (zero-padded to 128; M = 64 UMMAs run
// at half rate on this part, so nothing is lost by padding).  The O accumulator of 128
// heads x 512 dims in fp32 would fill all 512 TMEM columns, so a (token, split) work
// item is owned by a cluster of two CTAs, CTA c holding latent dims [256c, 256c+256) of
// K/V and of O:
//
//   TMEM (per CTA, 512 columns): Q half [0,128) as the A operand of QK (bf16 pairs), two
//   S partial buffers [128,192) and [192,256), the O half [256,512).
//   SMEM: a ring of four stages [64 rows x 256 dims] bf16 (128B-swizzled, 32 KB each),
//   two P buffers [128 heads x 64 rows] bf16 (16 KB each, the A operand of PV) and a
//   3-slot ring of raw cache rows.
//
// The launch is persistent: G = min(items, SMs / 2) pairs, pair c taking the work items
// c, c + G, ...; the tile sequence (and every barrier phase) runs on across items, so the
// producers prefetch the next item's rows while the current one finishes.
//
// Roles (512 threads):
//   warps 8 and 9, the MMA warps: issue every UMMA from one lane each, after blocking
//     waits for their inputs: S_c(j) = Q_c K_c(j)^T (M128 N64 K256, A from TMEM) into S
//     buffer j&1 (warp 8), and O_c += P(j) V_c(j) (M128 N256 K64, the stage read
//     MN-major; warp 9, which also forwards the exchange events to the peer CTA).
//   warp 10, the loader: puts each tile's raw rows in flight with TMA row gathers (four
//     rows per gather, the CTA's half of every 576-byte data row) into the raw ring, with
//     each row's four scale codes of the half (read one tile ahead).
//   warps 11-15, the converters: dequantise each raw tile into its stage.
//   warps 0-7, softmax + epilogue: thread (h, hc) owns head h (TMEM lane h) and score
//     columns [32 hc, 32 hc + 32) of every tile.
//
// Partial scores.  Each CTA's S holds the dot over its 256 dims only; the softmax threads
// send theirs to the peer CTA through an fp32 exchange buffer in L2 and add the peer's,
// so both CTAs hold the exact 512-wide scores.  The softmax is skewed by one tile to hide
// that round trip: step j loads S(j) and sends it, then finishes tile j-1 (adds the
// peer's partials, which arrived meanwhile, masks, updates the running max, writes P(j-1)
// and hands it to PV).  The running max only moves when it grows by more than 2^8, so O
// is rarely rescaled.
//
// The kernel is launched as a programmatic dependent of the previous kernel in the
// stream and waits for it after its own set-up (shared memory and TMEM only), before any
// global access.  Every wait is bounded; a wait that gives up records
// bit 0 in the status word and the CTA winds down (draining its UMMAs and gathers,
// freeing TMEM).
#include <cuda.h>

#include "smd_device.cuh"
#include "smd_internal.h"

namespace smd {
namespace {

constexpr int kTile = 64;                   // gathered rows per tile (one raw chunk)
constexpr int kTilesPerSplitUnit = kTileRows / kTile;  // tiles per host split unit (kTileRows rows)
constexpr int kDHalf = 256;                 // latent dims per CTA
constexpr int kSoftmaxThreads = 256;        // warps 0-7
constexpr int kGroupThreads = 128;          // one producer warpgroup
constexpr int kThreads = kSoftmaxThreads + 2 * kGroupThreads;
constexpr uint32_t kSoftmaxRegs = 176, kProducerRegs = 80;
static_assert(kSoftmaxThreads * kSoftmaxRegs + 2 * kGroupThreads * kProducerRegs == 65536, "register split");
constexpr int kProducerThreads = 2 * kGroupThreads;  // warps 8-15
constexpr int kStages = 4;                  // bf16 tile stages
constexpr int kRingSlots = 3;               // raw tile slots
constexpr int kCols = 32;                   // score columns per softmax thread
constexpr uint32_t kSlab = kTile * 128;     // [64 rows x 64 dims] bf16 = 8 KB
constexpr uint32_t kStageBytes = 4 * kSlab; // 32 KB
constexpr uint32_t kPBytes = 128 * 128;     // [128 heads x 64 rows] bf16 = 16 KB
constexpr uint32_t kOffP = kStages * kStageBytes;
constexpr uint32_t kOffRing = kOffP + 2 * kPBytes;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColQ = 0, kColS = 128, kColO = 256;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far beyond any legitimate wait
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: p <= 2^8 between rescales

// A raw tile of one half: 64 rows of the half's data bytes (as the TMA gathers write
// them, back to back), then the 64 rows' 8-byte scale rows.
template <int HALF>
struct RawFmt {
  static constexpr int NN = HALF == 0 ? 16 : 12;     // NoPE 16-byte pieces per row
  static constexpr int NR = HALF == 0 ? 0 : 8;       // RoPE pieces per row
  static constexpr int NP = NN + NR;
  static constexpr int DATA = NP * 16;               // 256 / 320 bytes of a row
  static constexpr int SCALES = kTile * DATA;        // offset of the scale rows
  static constexpr int SLOT = SCALES + kTile * 8;
  static constexpr int BYTE0 = HALF == 0 ? 0 : 256;  // first row byte of the half
  static constexpr int CODE0 = HALF == 0 ? 0 : 4;    // first scale code of the half
};
constexpr uint32_t kRingBytes = kRingSlots * RawFmt<1>::SLOT;
constexpr uint32_t kOffMisc = kOffRing + kRingBytes;

// Exchange buffers of one CTA in the workspace (what its peer writes into): two buffers,
// each 8 pieces x 256 threads x 16 B of fp32 partial scores (piece-major, so every warp
// access is one contiguous 512-byte run).
constexpr uint32_t kXchgBuf = kCols * 4u * kSoftmaxThreads;  // 32 KB
constexpr uint32_t kXchgRegion = 2u * kXchgBuf;

struct Misc {
  uint64_t kfull[kStages];   // converters -> issuer, softmax: stage filled (one arrival per warp)
  uint64_t kempty[kStages];  // PV commit -> converters: stage consumed
  uint64_t sfull[2];         // QK commit -> softmax: S buffer filled
  uint64_t sfree[2];         // softmax -> issuer: S buffer loaded into registers (8 warps)
  uint64_t pfull[2];         // softmax -> issuer: P buffer written, O rescaled (8 warps)
  uint64_t pvdone[2];        // PV commit -> softmax: P buffer read, O updated
  uint64_t xsent[2];         // softmax -> PV warp: partials of a tile stored to L2 (8 warps)
  uint64_t xread[2];         // softmax -> PV warp: the peer's partials of a tile consumed (8 warps)
  uint64_t xfull[2];         // peer PV warp -> softmax: peer partials in my exchange buffer (1 remote)
  uint64_t xempty[2];        // peer PV warp -> softmax: peer has read my partials (1 remote)
  uint64_t odone;            // last PV commit of an item -> softmax: O final
  uint64_t drain[2];         // the MMA warps' self-drain before TMEM is freed
  uint64_t sgrp;             // softmax-group rendezvous (8 warps per use)
  uint64_t qready;           // softmax -> issuer: an item's Q is in TMEM (8 warps)
  uint64_t rawfull[kRingSlots];   // raw tile landed (loader expect-tx arrival + codes arrival + TMA bytes)
  uint64_t rawempty[kRingSlots];  // raw tile converted (one arrival per converter warp)
  uint64_t hpair[4];         // warps w and w+4 (the two threads of heads 32w..32w+31): 2
  uint32_t tmem_base;
  uint32_t abort;
  uint32_t mask[kStages][2];        // valid-row bit masks of each stage's 32-row halves
  uint32_t maskring[kRingSlots][2]; // valid-row masks of each raw tile
  float red[2][2][128];             // per-column-half tile maxima, then final denominators
};
// The stages need 1024-byte alignment; dynamic shared memory starts 1024-aligned here
// (checked at run time), so no slack is reserved.
constexpr uint32_t kSmemBytes = kOffMisc + sizeof(Misc);
static_assert(kSmemBytes <= 232448, "shared memory budget");

__device__ __forceinline__ float ex2(float x) { return fast_exp2(x); }

__device__ __forceinline__ bool aborted(const Misc* m) {
  return *reinterpret_cast<const volatile uint32_t*>(&m->abort) != 0u;
}

// Bounded wait that also gives up early once another role of this CTA has aborted.
__device__ __forceinline__ bool wait_bar_loop(uint64_t* bar, uint32_t parity, const Misc* m, bool cluster_acquire) {
  auto poll = [&]() { return cluster_acquire ? mbar_try_wait_acq_cluster(bar, parity) : mbar_try_wait(bar, parity); };
  const uint64_t t0 = globaltimer_ns();
  while (!poll()) {
    if (aborted(m) || globaltimer_ns() - t0 > kWaitLimitNs) return false;
  }
  return true;
}
// The producer warps' waits: first poll inline, the rest in one out-of-line copy, which
// keeps their many wait sites from filling the instruction cache.
__device__ __noinline__ bool wait_bar_slow(uint64_t* bar, uint32_t parity, const Misc* m, bool cluster_acquire) {
  return wait_bar_loop(bar, parity, m, cluster_acquire);
}
template <bool OUTLINE = false>
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, const Misc* m,
                                         bool cluster_acquire = false) {
  if (cluster_acquire ? mbar_try_wait_acq_cluster(bar, parity) : mbar_try_wait(bar, parity)) return true;
  if constexpr (OUTLINE)
    return wait_bar_slow(bar, parity, m, cluster_acquire);
  else
    return wait_bar_loop(bar, parity, m, cluster_acquire);
}

// The same wait done by a whole warp, with a warp-uniform result, so that a warp never
// splits into lanes that go on and lanes that leave (which would strand the first at the
// next warp-collective instruction).
template <bool OUTLINE = false>
__device__ __forceinline__ bool wait_bar_warp(uint64_t* bar, uint32_t parity, const Misc* m,
                                              bool cluster_acquire = false) {
  const bool r = wait_bar<OUTLINE>(bar, parity, m, cluster_acquire);
  return __all_sync(0xffffffffu, r);
}

// One arrival per warp: the warp's lanes converge (which orders their earlier memory
// accesses before lane 0's release), then lane 0 arrives.  Barriers that whole warps
// arrive on count warps, which keeps the per-tile shared-memory atomics (each arrival is
// one) from congesting the shared-memory pipe the converters and the softmax use.
__device__ __forceinline__ void warp_arrive(uint64_t* bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

__device__ __forceinline__ void record_abort(Misc* m, uint32_t* status) {
  atomicExch(&m->abort, 1u);
  if (status != nullptr) atomicOr(status, 1u);
}

// Byte offset of the 16-byte chunk holding local dims [d0, d0+8) of `row` in a stage
// made of four 128B-swizzled [64 rows x 64 dims] slabs.
__device__ __forceinline__ uint32_t stage_off(uint32_t row, uint32_t d0) {
  return (d0 >> 6) * kSlab + sw128_off(row, (d0 & 63) >> 3);
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void st_global_f4(float* p, float a, float b, float c, float d) {
  asm volatile("st.global.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}
// L2 load (the exchange buffers are written by the peer SM, so L1 must not serve them).
__device__ __forceinline__ float4 ld_cg_f4(const float* p) {
  float4 v;
  asm volatile("ld.global.cg.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p)
               : "memory");
  return v;
}

// One (token, split) work item: tiles [tile_begin, tile_begin + n) of the token's
// entries (64-row tiles; a split covers tiles_per_split units of kTileRows rows).
struct Item {
  int t, split, tile_begin, n;  // n = tiles of the item (0 for a split past the end)
};
__device__ __forceinline__ Item item_of(const AttnParams& p, int w) {
  Item it;
  it.t = w / p.S;
  it.split = w - it.t * p.S;
  const int tps = p.tiles_per_split * kTilesPerSplitUnit;
  it.tile_begin = it.split * tps;
  const int ntok = (p.N + kTile - 1) / kTile;
  it.n = max(0, min(ntok, it.tile_begin + tps) - it.tile_begin);
  return it;
}

// Walks the tiles of the items w0, w0 + G, ... in order, skipping items without tiles.
struct TileCursor {
  int w, k, n, G, items;
  int64_t row0;   // gidx offset of the tile's first row
  int rows;       // rows of the tile inside the token's entry list (1..64)
  __device__ void settle(const AttnParams& p) {
    while (w < items) {
      const Item it = item_of(p, w);
      if (k < it.n) {
        n = it.n;
        const int r0 = (it.tile_begin + k) * kTile;
        row0 = (int64_t)it.t * p.N + r0;
        rows = min(kTile, p.N - r0);
        return;
      }
      w += G;
      k = 0;
    }
  }
  __device__ void init(const AttnParams& p, int w0, int g, int items_) {
    w = w0; k = 0; n = 0; G = g; items = items_; row0 = 0; rows = 0;
    settle(p);
  }
  __device__ bool valid() const { return w < items; }
  __device__ void next(const AttnParams& p) {
    ++k;
    settle(p);
  }
};

// TMA gather of four rows of the cache viewed as a 2-D tensor of 16-byte-spaced rows
// (row y = bytes [16y, 16y + 576), u16 elements): rows y0..y3, elements [x, x + box),
// written back to back at `dst`.
__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap* map, int x, int y0, int y1, int y2,
                                            int y3, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
      "l"(map), "r"(x), "r"(y0), "r"(y1), "r"(y2), "r"(y3), "r"(smem_u32(bar))
      : "memory");
}

// Dequantises the 16-byte NoPE piece `k` of a raw row (scale code from its scale row)
// into the stage on the exact path (any bytes, any code), or zeros when the row is masked;
// elements in the (d0, d2, d1, d3) order of dequant16_perm_*.
__device__ __forceinline__ void convert_nope(uint8_t* stage, int srow, int k, uint4 raw, uint32_t code, bool valid) {
  uint4 lo, hi;
  if (!valid) {
    raw = make_uint4(0, 0, 0, 0);
    code = 0;
  }
  dequant16_perm_exact(raw, code, lo, hi);
  *reinterpret_cast<uint4*>(stage + stage_off(srow, k * 16)) = lo;
  *reinterpret_cast<uint4*>(stage + stage_off(srow, k * 16 + 8)) = hi;
}

constexpr int kConverters = kProducerThreads - 96;  // warps 11-15


// The MMA warps issue every UMMA of the CTA from one lane, each after a blocking wait for
// its inputs, in the order in which the skewed softmax frees them.
//   warp 8 (QK): QK of a tile once its stage is filled and its S buffer free, which runs
//     QK two tiles ahead of the softmax (an item's first two once its Q is in TMEM).
//   warp 9 (PV): in step k of an item's softmax, forwards the exchange events of that
//     step to the peer CTA (tile j's partials stored, tile j - 1's peer partials read;
//     cluster-scope release arrivals, whose memory barrier would otherwise stall the
//     softmax warps), then PV of tile j - 1 once its P is written; the item's last PV
//     also signals O final.
// Separate warps keep a PV (which waits for the softmax) from queueing behind a QK (which
// waits for the converters), since the converters in turn wait for PV to free a stage.
template <bool QK>
__device__ __forceinline__ void mma_warp(uint8_t* smem, Misc* m, const AttnParams& p, int cid, int items,
                                         uint32_t tmem, int lane, uint32_t peer) {
  constexpr uint32_t kIdescQK = idesc_bf16_f32(128, kTile, false, false);
  constexpr uint32_t kIdescPV = idesc_bf16_f32(128, kDHalf, false, true);
  // Shared-memory descriptors: a base descriptor per operand plus constant offsets in
  // its address field (address >> 4, 14 bits; every offset here stays inside the field).
  // The issue loops stay rolled: the tensor core, not the issuing lane, sets their pace,
  // and small loops keep these warps' code resident in the instruction cache.
  const uint64_t dstage = desc_sw128(smem_u32(smem), 16, 1024);         // K-major B of QK
  const uint64_t dvstage = desc_sw128(smem_u32(smem), kSlab, 1024);     // MN-major B of PV
  const uint64_t dp = desc_sw128(smem_u32(smem + kOffP), 16, 1024);     // A of PV
  auto qk = [&](int jj, bool wait_sfree) -> bool {  // S(jj) = Q K(jj)^T into S buffer jj & 1
    if (!wait_bar_warp<true>(&m->kfull[jj & (kStages - 1)], (jj / kStages) & 1, m)) return false;
    if (wait_sfree && !wait_bar_warp<true>(&m->sfree[jj & 1], ((jj >> 1) - 1) & 1, m)) return false;
    if (lane == 0) {
      tc_fence_after();
      const uint64_t b = dstage + (uint64_t)(((jj & (kStages - 1)) * kStageBytes) >> 4);
      const uint32_t d = tmem + kColS + (jj & 1) * kTile;
#pragma unroll 1
      for (int kk = 0; kk < kDHalf / 16; ++kk)
        umma_ts(d, tmem + kColQ + kk * 8, b + (uint64_t)((((kk >> 2) * kSlab) + (kk & 3) * 32) >> 4), kIdescQK,
                kk > 0 ? 1u : 0u);
      umma_commit(&m->sfull[jj & 1]);
    }
    __syncwarp();
    return true;
  };
  auto pv = [&](int jj, bool first, bool last) -> bool {  // O += P(jj) V(jj), then free the stage and P
    if (!wait_bar_warp<true>(&m->pfull[jj & 1], (jj >> 1) & 1, m)) return false;
    if (lane == 0) {
      tc_fence_after();
      const uint64_t a = dp + (uint64_t)(((jj & 1) * kPBytes) >> 4);
      const uint64_t b = dvstage + (uint64_t)(((jj & (kStages - 1)) * kStageBytes) >> 4);
#pragma unroll 1
      for (int kk = 0; kk < kTile / 16; ++kk)
        umma_ss(tmem + kColO, a + (uint64_t)((kk * 32) >> 4), b + (uint64_t)((kk * 2048) >> 4), kIdescPV,
                (!first || kk > 0) ? 1u : 0u);
      umma_commit(&m->kempty[jj & (kStages - 1)]);
      umma_commit(&m->pvdone[jj & 1]);
      if (last) umma_commit(&m->odone);
    }
    __syncwarp();
    return true;
  };
  auto forward = [&](uint64_t* local, uint32_t parity, uint64_t* remote) -> bool {
    if (!wait_bar_warp<true>(local, parity, m)) return false;
    if (lane == 0) mbar_arrive_cluster(mapa(smem_u32(remote), peer));
    __syncwarp();
    return true;
  };
  bool ok = true;
  int j0 = 0;   // sequence number of the item's first tile
  int neq = 0;  // items with tiles so far
  for (int w = cid; w < items && ok; w += p.G) {
    const int n = item_of(p, w).n;
    if (n == 0) continue;
    if constexpr (QK) {
      ok = wait_bar_warp<true>(&m->qready, neq & 1, m);  // the S buffers were freed before Q
      if (ok) ok = qk(j0, false);
      if (ok && n > 1) ok = qk(j0 + 1, false);
      for (int k = 2; k < n && ok; ++k) ok = qk(j0 + k, true);
    } else {
      for (int k = 0; k < n && ok; ++k) {
        const int jj = j0 + k;
        ok = forward(&m->xsent[jj & 1], (jj >> 1) & 1, &m->xfull[jj & 1]);
        if (ok && k > 0) ok = forward(&m->xread[(jj - 1) & 1], ((jj - 1) >> 1) & 1, &m->xempty[(jj - 1) & 1]);
        if (ok && k > 0) ok = pv(jj - 1, k == 1, false);
      }
      if (ok) ok = forward(&m->xread[(j0 + n - 1) & 1], ((j0 + n - 1) >> 1) & 1, &m->xempty[(j0 + n - 1) & 1]);
      if (ok) ok = pv(j0 + n - 1, n == 1, true);
    }
    j0 += n;
    ++neq;
  }
  if (!ok && lane == 0) record_abort(m, p.status);
  if (lane == 0) {
    umma_commit(&m->drain[QK ? 0 : 1]);  // every UMMA this warp issued lands before TMEM is freed
    mbar_wait_bounded(&m->drain[QK ? 0 : 1], 0, kWaitLimitNs);
  }
  __syncwarp();
}

// The loader warp (warp 10, TMA mode): puts the raw tiles in flight in order, four rows
// per TMA gather (the CTA's half of every 576-byte data row; masked rows read row 0 and
// are zeroed by the converters), as far ahead as the 3-slot ring allows.  The four scale
// codes of the half (one 32-bit word of each row's 8-byte scale row) are read with plain
// loads one tile ahead and stored into the slot with the tile; the slots of the next two
// tiles are prefetched into registers.
template <int HALF>
__device__ __forceinline__ void loader_warp(uint8_t* smem, Misc* m, const AttnParams& p, const CUtensorMap* map,
                                            int cid, int items, int lane) {
  using F = RawFmt<HALF>;
  const CacheView cv = make_cache_view(p.cache, p.P);
  const int64_t n_slots = p.num_pages * p.P;
  uint8_t* ring = smem + kOffRing;
  auto load_gidx = [&](const TileCursor& c, int r) -> int32_t {
    if (!c.valid() || r >= c.rows) return -1;
    const int32_t v = ldg_nc_s32(p.gidx + c.row0 + r);
    return ((int64_t)v >= n_slots) ? -1 : v;
  };
  const int32_t rows_per_page16 = p.P * (kRowBytes / 8) / 2;  // P * 584 / 16 (TMA mode: P even)
  auto row16 = [&](int32_t sl) -> int32_t {  // 16-byte row index of slot sl's data row
    int32_t page, off;
    slot_page_off(cv, sl, page, off);
    return page * rows_per_page16 + off * (kDataBytes / 16);
  };
  auto codes = [&](int32_t sl) -> uint32_t {  // the half's four scale codes of slot sl (0 if masked)
    if (sl < 0) return 0u;
    int32_t page, off;
    slot_page_off(cv, sl, page, off);
    return ldg_nc_u32(cv.base + (int64_t)page * cv.page_bytes + cv.scale_start + (int64_t)off * kScaleBytes +
                      F::CODE0);
  };
  TileCursor iss, pre;
  iss.init(p, cid, p.G, items);
  pre = iss;
  int32_t ga0 = load_gidx(pre, lane), gb0 = load_gidx(pre, lane + 32);
  uint32_t ca0 = codes(ga0), cb0 = codes(gb0);
  pre.next(p);
  int32_t ga1 = load_gidx(pre, lane), gb1 = load_gidx(pre, lane + 32);
  int issued = 0;
  for (int q = 0; iss.valid(); ++q) {
    const int slot = q % kRingSlots;
    if (q >= kRingSlots && !wait_bar_warp<true>(&m->rawempty[slot], (q / kRingSlots - 1) & 1, m)) {
      if (lane == 0) record_abort(m, p.status);
      break;
    }
    uint8_t* sbase = ring + slot * F::SLOT;
    const uint32_t base = smem_u32(sbase);
    const bool va = ga0 >= 0, vb = gb0 >= 0;
    const uint32_t ba = __ballot_sync(0xffffffffu, va), bb = __ballot_sync(0xffffffffu, vb);
    if (lane == 0) {
      m->maskring[slot][0] = ba;
      m->maskring[slot][1] = bb;
      mbar_arrive_expect_tx(&m->rawfull[slot], kTile * F::DATA);
    }
    __syncwarp();
    const int32_t ya = va ? row16(ga0) : 0, yb = vb ? row16(gb0) : 0;  // masked rows read row 0
    int32_t y[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int src = (4 * lane + i) & 31;
      const int32_t a = __shfl_sync(0xffffffffu, ya, src), b = __shfl_sync(0xffffffffu, yb, src);
      y[i] = lane < 8 ? a : b;
    }
    if (lane < 16)
      tma_gather4(base + 4 * lane * F::DATA, map, F::BYTE0 / 2, y[0], y[1], y[2], y[3], &m->rawfull[slot]);
    const uint32_t ca1 = codes(ga1), cb1 = codes(gb1);  // next tile's codes, in flight meanwhile
    *reinterpret_cast<uint32_t*>(sbase + F::SCALES + lane * 8 + F::CODE0) = ca0;
    *reinterpret_cast<uint32_t*>(sbase + F::SCALES + (lane + 32) * 8 + F::CODE0) = cb0;
    warp_arrive(&m->rawfull[slot]);  // releases maskring and the codes
    iss.next(p);
    ga0 = ga1;
    gb0 = gb1;
    ca0 = ca1;
    cb0 = cb1;
    pre.next(p);
    ga1 = load_gidx(pre, lane);
    gb1 = load_gidx(pre, lane + 32);
    ++issued;
  }
  // No gather may land after the CTA is gone (the converters skip their waits once the
  // CTA has aborted): wait, bounded, for the last tiles put in flight.
  if (lane == 0)
    for (int t = issued > kRingSlots ? issued - kRingSlots : 0; t < issued; ++t)
      (void)mbar_wait_bounded(&m->rawfull[t % kRingSlots], (t / kRingSlots) & 1, kWaitLimitNs);
  __syncwarp();
}

// The converter warps (11-15, ct = 0..159) of the TMA mode: each raw tile the loader
// warp put in flight is dequantised into its stage.
template <int HALF>
__device__ __forceinline__ void produce_tma(uint8_t* smem, Misc* m, const AttnParams& p, int cid, int items, int ct) {
  using F = RawFmt<HALF>;
  uint8_t* ring = smem + kOffRing;
  TileCursor conv;
  conv.init(p, cid, p.G, items);
  for (int j = 0; conv.valid(); ++j) {
    const int slot = j % kRingSlots;
    const int s = j & (kStages - 1);
    uint8_t* stage = smem + s * kStageBytes;
    // A wait that gives up flags the CTA; the converters still run their remaining tile
    // sequence without converting, and every later wait returns at once.
    bool live = j < kStages || wait_bar<true>(&m->kempty[s], ((j / kStages) - 1) & 1, m);
    live = live && wait_bar<true>(&m->rawfull[slot], (j / kRingSlots) & 1, m);
    if (!live) record_abort(m, p.status);
    live = __all_sync(0xffffffffu, live && !aborted(m));  // warp-uniform: the loop has warp collectives
    if (live) {
      const uint8_t* raw = ring + slot * F::SLOT;
      const uint32_t mk0 = m->maskring[slot][0], mk1 = m->maskring[slot][1];
      auto valid_row = [&](int r) { return (((r < 32 ? mk0 : mk1) >> (r & 31)) & 1u) != 0u; };
      // NoPE: 64 rows x NN pieces; consecutive threads take consecutive pieces of a row.
      // Pieces are loaded four at a time and converted on the fast path (exact for any
      // bytes when the scale code is at most 134); a thread redoes its pieces with larger
      // codes (rare) on the exact path afterwards, overwriting the fast result.
      constexpr int NI = (kTile * F::NN + kConverters - 1) / kConverters;
      constexpr int NB = 4;
#pragma unroll 1
      for (int i0 = 0; i0 < NI; i0 += NB) {
        uint4 v[NB];
        uint32_t code[NB];
        uint32_t redo = 0;
#pragma unroll
        for (int i = 0; i < NB; ++i) {
          const int pc = ct + kConverters * (i0 + i);
          const int r = pc / F::NN, k = pc - r * F::NN;
          v[i] = make_uint4(0, 0, 0, 0);
          code[i] = 0;
          if (i0 + i < NI && pc < kTile * F::NN) {
            v[i] = *reinterpret_cast<const uint4*>(raw + r * F::DATA + k * 16);
            code[i] = raw[F::SCALES + r * 8 + F::CODE0 + (k >> 2)];
          }
        }
#pragma unroll
        for (int i = 0; i < NB; ++i) {
          const int pc = ct + kConverters * (i0 + i);
          const int r = pc / F::NN, k = pc - r * F::NN;
          if (i0 + i < NI && pc < kTile * F::NN) {
            const bool valid = valid_row(r);
            uint4 lo, hi;
            dequant16_perm_nz(v[i], code[i], valid, lo, hi);
            *reinterpret_cast<uint4*>(stage + stage_off(r, k * 16)) = lo;
            *reinterpret_cast<uint4*>(stage + stage_off(r, k * 16 + 8)) = hi;
            redo |= (valid && code[i] > 134u) ? (1u << i) : 0u;
          }
        }
        if (redo != 0u) {
#pragma unroll 1
          for (int i = 0; i < NB; ++i) {
            if ((redo >> i) & 1u) {
              const int pc = ct + kConverters * (i0 + i);
              const int r = pc / F::NN, k = pc - r * F::NN;
              convert_nope(stage, r, k, *reinterpret_cast<const uint4*>(raw + r * F::DATA + k * 16),
                                  raw[F::SCALES + r * 8 + F::CODE0 + (k >> 2)], true);
            }
          }
        }
      }
      if constexpr (F::NR > 0) {
#pragma unroll 1
        for (int i = 0; i < (kTile * F::NR + kConverters - 1) / kConverters; ++i) {
          const int pc = ct + kConverters * i;
          if (pc < kTile * F::NR) {
            const int r = pc / F::NR, k = pc - r * F::NR;
            uint4 v = *reinterpret_cast<const uint4*>(raw + r * F::DATA + (F::NN + k) * 16);
            if (!valid_row(r)) v = make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(stage + stage_off(r, 192 + k * 8)) = scrub_bf16x8(v);
          }
        }
      }
      if (ct == 0) {
        m->mask[s][0] = mk0;
        m->mask[s][1] = mk1;
      }
    }
    warp_arrive(&m->rawempty[slot]);
    fence_async_smem();
    warp_arrive(&m->kfull[s]);
    conv.next(p);
  }
}

// Fallback producer for caches whose rows are only 8-byte aligned (pages of an odd slot
// count) or too large for 32-bit TMA row coordinates: every thread loads its pieces
// straight from global memory (no ring), one 64-row tile at a time.
template <int HALF>
__device__ __forceinline__ void produce_direct(uint8_t* smem, Misc* m, const AttnParams& p, int cid, int items,
                                               int ct) {
  using F = RawFmt<HALF>;
  const CacheView cv = make_cache_view(p.cache, p.P);
  const int64_t n_slots = p.num_pages * p.P;
  TileCursor conv;
  conv.init(p, cid, p.G, items);
  for (int j = 0; conv.valid(); ++j) {
    const int s = j & (kStages - 1);
    uint8_t* stage = smem + s * kStageBytes;
    bool live = j < kStages || wait_bar<true>(&m->kempty[s], ((j / kStages) - 1) & 1, m);
    if (!live) record_abort(m, p.status);
    live = __all_sync(0xffffffffu, live && !aborted(m));
    auto slot_of = [&](int r) -> int32_t {
      if (r >= conv.rows) return -1;
      const int32_t v = ldg_nc_s32(p.gidx + conv.row0 + r);
      return ((int64_t)v >= n_slots) ? -1 : v;
    };
    if (live) {
      for (int pc = ct; pc < kTile * F::NP; pc += kConverters) {
        const int r = pc / F::NP, k = pc - r * F::NP;
        const int32_t g = slot_of(r);
        uint4 v = make_uint4(0, 0, 0, 0);
        uint32_t code = 0;
        if (g >= 0) {
          const uint8_t* d = row_data(cv, g) + F::BYTE0 + k * 16;
          const uint2 a = ldg_nc_v2(d), b = ldg_nc_v2(d + 8);
          v = make_uint4(a.x, a.y, b.x, b.y);
          if (k < F::NN) code = ldg_nc_u8(row_scales(cv, g) + F::CODE0 + (k >> 2));
        }
        if (k < F::NN)
          convert_nope(stage, r, k, v, code, g >= 0);
        else
          *reinterpret_cast<uint4*>(stage + stage_off(r, 192 + (k - F::NN) * 8)) = scrub_bf16x8(v);
      }
      if (ct < 64) {  // valid-row masks of the tile's two 32-row halves
        const uint32_t bits = __ballot_sync(0xffffffffu, slot_of(ct) >= 0);
        if ((ct & 31) == 0) m->mask[s][ct >> 5] = bits;
      }
    }
    fence_async_smem();
    warp_arrive(&m->kfull[s]);
    conv.next(p);
  }
}

}  // namespace

// Kernel parameters: the call's parameters and, for the TMA producer, the cache's two
// gather tensor maps (one per latent half).
struct KernelParams {
  AttnParams p;
  CUtensorMap map[2];  // the type carries the 128-byte alignment of a tensor map
};

template <bool TMA>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    attn_pair_kernel(const __grid_constant__ KernelParams kp) {
  const AttnParams& p = kp.p;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  uint8_t* sP = smem + kOffP;
  Misc* m = reinterpret_cast<Misc*>(smem + kOffMisc);

  // Launched as a programmatic dependent of the previous kernel in the stream (the index
  // conversion): the setup below touches nothing that kernel writes, so it overlaps that
  // kernel's tail, and every thread waits for its completion before its role starts.
  // (No early trigger for the next kernel: a split combine launched early would pack its
  // blocks onto the few SMs this grid leaves free; launched at this grid's exit it
  // spreads over the whole GPU.)
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const uint32_t half = cluster_rank();   // == blockIdx.x & 1
  const uint32_t peer = half ^ 1u;
  const int cid = blockIdx.x >> 1;
  const int items = p.T * p.S;

  // The stage layout needs a 1024-byte aligned base (true for this kernel's dynamic
  // shared memory, which follows the 1 KB system reservation).  Both CTAs of the pair
  // see the same alignment, so both leave together before any cluster barrier.
  if ((smem_u32(smem_raw) & 1023u) != 0u) {
    grid_dep_wait();  // the conversion kernel clears the status word first
    if (tid == 0 && p.status != nullptr) atomicOr(p.status, 2u);
    return;
  }

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&m->kfull[s], kConverters / 32);
      mbar_init(&m->kempty[s], 1);
    }
    for (int r = 0; r < kRingSlots; ++r) {
      mbar_init(&m->rawfull[r], 2);  // the loader's expect-tx arrival, then its arrival after the codes
      mbar_init(&m->rawempty[r], kConverters / 32);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&m->sfull[b], 1);
      mbar_init(&m->sfree[b], kSoftmaxThreads / 32);
      mbar_init(&m->pfull[b], kSoftmaxThreads / 32);
      mbar_init(&m->pvdone[b], 1);
      mbar_init(&m->xsent[b], kSoftmaxThreads / 32);
      mbar_init(&m->xread[b], kSoftmaxThreads / 32);
      mbar_init(&m->xfull[b], 1);
      mbar_init(&m->xempty[b], 1);
    }
    mbar_init(&m->odone, 1);
    mbar_init(&m->drain[0], 1);
    mbar_init(&m->drain[1], 1);
    mbar_init(&m->sgrp, kSoftmaxThreads / 32);
    mbar_init(&m->qready, kSoftmaxThreads / 32);
    for (int i = 0; i < 4; ++i) mbar_init(&m->hpair[i], 2);
    m->abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&m->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // the peer's barriers exist before anyone arrives on them remotely
  tc_fence_after();
  const uint32_t tmem = m->tmem_base;
  grid_dep_wait();

  // Register budget: the launch gives 128 per thread (512 x 128 = the whole file); the
  // softmax warpgroups take 176 and the producer warpgroups keep 80 (2 x 128 x (176 + 80)
  // = 65536).
  if (warp < 8) {
    regs_inc<kSoftmaxRegs>();
    // ------------------------------------------------------------ softmax + epilogue
    // Thread (h, hc): head h = TMEM lane h, score columns [32 hc, 32 hc + 32) of every tile.
    const int h = tid & 127;
    const int hc = warp >> 2;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float sl2 = p.scale * kLog2e;
    const bool pad_warp = (warp & 3) * 32 >= p.H;  // all 32 heads of this warp are padding
    // head h's sink logit (natural log), read once here rather than at each item's end
    const float sink_h = (p.S == 1 && p.sink != nullptr && h < p.H) ? __ldg(p.sink + h) : -INFINITY;
    // Exchange buffers (CTA `rank`'s incoming partials) are recomputed at each use (kernel
    // parameters live in the constant bank), which keeps them out of the register budget.
    auto xbuf = [&](uint32_t rank, int b) {
      return reinterpret_cast<float*>(p.xchg + ((size_t)cid * 2 + rank) * kXchgRegion + (size_t)b * kXchgBuf) +
             tid * 4;
    };
    bool ok = true;
    uint32_t sgrp_phase = 0;
    int j = 0;       // sequence number of the next tile to load (runs on across items)
    int ne_no = 0;   // items with tiles taken by this pair so far

    for (int w = cid; w < items && ok; w += p.G) {
      const Item item = item_of(p, w);
      const int n = item.n;
      {  // this thread's half of head h's Q half -> TMEM columns [64 hc, 64 hc + 64) of lane h
        const uint8_t* qrow = static_cast<const uint8_t*>(p.q) + ((int64_t)item.t * p.H + h) * (kLatent * 2) +
                              half * (kDHalf * 2) + hc * 256;
        uint32_t r[2][32];
        // local dims [64 hc, 64 hc + 64)... of this CTA's 256: NoPE below local dim 448 - 256 half
        const int nope_chunks = half == 0 ? 16 : (hc == 0 ? 16 : 8);  // 16-byte chunks of NoPE dims
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          uint4 v = h < p.H ? ldg_nc_v4(qrow + i * 16) : make_uint4(0, 0, 0, 0);
          if (i < nope_chunks) {  // the stage's (d0, d2, d1, d3) order of NoPE dims
            v = make_uint4(__byte_perm(v.x, v.y, 0x5410u), __byte_perm(v.x, v.y, 0x7632u),
                           __byte_perm(v.z, v.w, 0x5410u), __byte_perm(v.z, v.w, 0x7632u));
          }
          r[i >> 3][(i & 7) * 4 + 0] = v.x;
          r[i >> 3][(i & 7) * 4 + 1] = v.y;
          r[i >> 3][(i & 7) * 4 + 2] = v.z;
          r[i >> 3][(i & 7) * 4 + 3] = v.w;
        }
        tmem_st32(tmem + lane_base + kColQ + hc * 64, r[0]);
        tmem_st32(tmem + lane_base + kColQ + hc * 64 + 32, r[1]);
        tmem_wait_st();
        tc_fence_before();
        if (n > 0) warp_arrive(&m->qready);  // the issuer may start QK of the item's first tile
      }

      float m_ref = -INFINITY;  // reference max (log2 domain) the weights are taken against
      float l_run = 0.f;        // this thread's share of the denominator relative to m_ref
      float xp[kCols];          // this CTA's partial scores of the previous tile (unscaled)
      // Step k loads and sends tile j (k < n), then finishes tile j - 1 (k > 0).
      for (int k = 0; k <= n; ++k) {
        const int jl = j - 1;
        if (pad_warp) {
          // Heads past H are zero padding whose rows nobody reads: keep only the barrier
          // protocol, each arrival after a wait that orders it behind the same barrier's
          // previous phase (sfull(j) follows sfree of tile j - 2; xempty(j) follows xsent
          // of tile j - 2; pvdone of tile jl - 2 follows every xread and pfull of it).
          if (k < n) {
            if (!(ok = wait_bar_warp(&m->sfull[j & 1], (j >> 1) & 1, m))) break;
            warp_arrive(&m->sfree[j & 1]);
            if (j >= 2 && !(ok = wait_bar_warp(&m->xempty[j & 1], ((j >> 1) - 1) & 1, m, true))) break;
            warp_arrive(&m->xsent[j & 1]);
          }
          if (k > 0) {
            if (jl >= 2 && !(ok = wait_bar_warp(&m->pvdone[jl & 1], ((jl >> 1) - 1) & 1, m))) break;
            warp_arrive(&m->xread[jl & 1]);
            warp_arrive(&m->pfull[jl & 1]);
            if (!(ok = __all_sync(0xffffffffu, !aborted(m)))) break;
          }
          if (k < n) ++j;
          continue;
        }
        float rv[kCols];  // the peer's partials of tile jl
        float xc[kCols];  // this CTA's partials of tile j
        if (k > 0) {  // start reading the peer's partials of tile jl; they are used below
          if (!(ok = wait_bar_warp(&m->xfull[jl & 1], (jl >> 1) & 1, m, true))) break;
          const float* src = xbuf(half, jl & 1);
#pragma unroll
          for (int i = 0; i < kCols / 4; ++i) {
            const float4 v = ld_cg_f4(src + i * (kSoftmaxThreads * 4));
            rv[4 * i] = v.x;
            rv[4 * i + 1] = v.y;
            rv[4 * i + 2] = v.z;
            rv[4 * i + 3] = v.w;
          }
        }
        if (k < n) {
          if (!(ok = wait_bar_warp(&m->sfull[j & 1], (j >> 1) & 1, m))) break;
          tc_fence_after();
          {
            uint32_t r[32];
            tmem_ld32(tmem + lane_base + kColS + (j & 1) * kTile + hc * kCols, r);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < kCols; ++i) xc[i] = __uint_as_float(r[i]);
          }
          // S is in registers: QK of tile j + 2 may reuse the buffer.
          tc_fence_before();
          warp_arrive(&m->sfree[j & 1]);
          // Send: the peer's buffer j & 1 is free once the peer has read tile j - 2.
          if (j >= 2 && !(ok = wait_bar_warp(&m->xempty[j & 1], ((j >> 1) - 1) & 1, m, true))) break;
          float* dst = xbuf(peer, j & 1);
#pragma unroll
          for (int i = 0; i < kCols / 4; ++i)
            st_global_f4(dst + i * (kSoftmaxThreads * 4), xc[4 * i], xc[4 * i + 1], xc[4 * i + 2], xc[4 * i + 3]);
          warp_arrive(&m->xsent[j & 1]);  // the PV warp publishes them to the peer
        }
        if (k > 0) {
          // Finish tile jl: the 512-wide scores in log2 units.
#pragma unroll
          for (int i = 0; i < kCols; ++i) rv[i] = (xp[i] + rv[i]) * sl2;
          warp_arrive(&m->xread[jl & 1]);  // the peer's partials of tile jl are consumed
          // The stage's valid-row mask (published by the converters before kfull).
          const int s = jl & (kStages - 1);
          if (!(ok = wait_bar_warp(&m->kfull[s], (jl / kStages) & 1, m))) break;
          const uint32_t mk = m->mask[s][hc];
          float lmax = -INFINITY;
          if (mk == 0xffffffffu) {
#pragma unroll
            for (int i = 0; i < kCols; ++i) lmax = fmaxf(lmax, rv[i]);
          } else {
#pragma unroll
            for (int i = 0; i < kCols; ++i) {
              const float v = ((mk >> i) & 1u) ? rv[i] : -INFINITY;
              rv[i] = v;
              lmax = fmaxf(lmax, v);
            }
          }
          // Both threads of head h agree on the tile max and so on m_ref.
          m->red[jl & 1][hc][h] = lmax;
          warp_arrive(&m->hpair[warp & 3]);
          if (!(ok = wait_bar_warp(&m->hpair[warp & 3], jl & 1, m))) break;
          const float tmax = fmaxf(lmax, m->red[jl & 1][hc ^ 1][h]);
          float alpha = 1.f;
          const bool upd = tmax > m_ref + kRescaleThreshold;  // false while everything is masked
          if (upd) {
            alpha = ex2(m_ref - tmax);  // 0 when m_ref is -inf
            m_ref = tmax;
          }
          float psum = 0.f;
          uint32_t pk[kCols / 2];
          if (m_ref == -INFINITY) {
#pragma unroll
            for (int i = 0; i < kCols / 2; ++i) pk[i] = 0u;
          } else {
#pragma unroll
            for (int i = 0; i < kCols / 2; ++i) {
              const float p0 = ex2(rv[2 * i] - m_ref), p1 = ex2(rv[2 * i + 1] - m_ref);
              psum += p0 + p1;  // the denominator keeps the unrounded weights
              pk[i] = bf16x2_bits(__floats2bfloat162_rn(p0, p1));
            }
          }
          l_run = l_run * alpha + psum;
          // P buffer jl & 1 was last read by PV of tile jl - 2.
          if (jl >= 2 && !(ok = wait_bar_warp(&m->pvdone[jl & 1], ((jl >> 1) - 1) & 1, m))) break;
          uint8_t* pbuf = sP + (jl & 1) * kPBytes;
#pragma unroll
          for (int c = 0; c < kCols / 8; ++c)
            *reinterpret_cast<uint4*>(pbuf + sw128_off(h, hc * (kCols / 8) + c)) =
                make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
          // O holds the item's PV up to tile jl - 1: rescale it once that PV has landed.
          if (k > 1 && __any_sync(0xffffffffu, upd)) {
            if (!(ok = wait_bar_warp(&m->pvdone[(jl - 1) & 1], ((jl - 1) >> 1) & 1, m))) break;
            tc_fence_after();
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
          warp_arrive(&m->pfull[jl & 1]);
          ok = !aborted(m);
          if (!(ok = __all_sync(0xffffffffu, ok))) break;
        }
        if (k < n) {
#pragma unroll
          for (int i = 0; i < kCols; ++i) xp[i] = xc[i];
          ++j;
        }
      }
      if (!ok) break;
      if (n > 0) {
        if (!(ok = wait_bar_warp(&m->odone, ne_no & 1, m))) break;
        ++ne_no;
      }
      // Epilogue: head h, local dims [128 hc, 128 hc + 128) of this CTA's 256.
      tc_fence_after();
      m->red[0][hc][h] = l_run;  // every use of red[][] by the tile loop is over (odone)
      warp_arrive(&m->sgrp);
      if (!(ok = wait_bar_warp(&m->sgrp, sgrp_phase, m))) break;
      sgrp_phase ^= 1u;
      const float l_tot = l_run + m->red[0][hc ^ 1][h];
      const bool o_live = n > 0;
      const bool head_ok = h < p.H;
      const int d0 = half * kDHalf + hc * 128;  // first output dim of this thread
      const int t = item.t;
      // One split: fold the sink into the denominator and write bf16 out + lse.  Several
      // splits: write the split's normalised fp32 output and sink-free lse.
      float factor = 0.f, lse_v = -INFINITY;
      if (p.S == 1) {
        const float sink_nat = sink_h;
        const float ms = sink_nat * kLog2e;
        const float M = fmaxf(m_ref, ms);
        if (M != -INFINITY) {
          const float den = l_tot * ex2(m_ref - M) + (ms == -INFINITY ? 0.f : ex2(ms - M));
          factor = ex2(m_ref - M) / den;
          // natural-log max from whichever term set it, so a sink-only row gives lse = sink exactly
          lse_v = (M == m_ref ? m_ref * kLn2 : sink_nat) + log2f(den) * kLn2;
        }
      } else if (l_tot > 0.f) {
        factor = 1.f / l_tot;
        lse_v = (m_ref + log2f(l_tot)) * kLn2;
      }
      const int64_t orow_idx = p.S == 1 ? (int64_t)t * p.H + h : ((int64_t)t * p.S + item.split) * p.H + h;
      // Split partials (fp32) go out through a warp-private 4 KB slice of the P buffers
      // (no UMMA reads them once O is final): per 32-dim chunk lane r writes its head's
      // 128 bytes as row r, its 16-byte granules XOR-swizzled by r so that 8 consecutive
      // rows cover all banks; each warp store then writes four whole 128-byte row segments
      // instead of 16 bytes in each of 32 rows.
      if (!pad_warp) {
        uint8_t* wst = sP + warp * 4096;
        const int ln = tid & 31;
        const int head0 = (warp & 3) * 32;
        const int64_t orow0 = orow_idx - ln;  // output row of lane 0's head
        // 32 columns of O (this thread's head) from TMEM; NoPE columns hold dims in the
        // (d0, d2, d1, d3) order of the stage, which is undone here.
        auto load_o_chunk = [&](uint32_t (&o)[32], int col, bool nope) {
          if (o_live) {
            tmem_ld32(tmem + lane_base + kColO + col, o);
            tmem_wait_ld();
            if (nope) {
#pragma unroll
              for (int g4 = 0; g4 < 8; ++g4) {
                const uint32_t t1 = o[4 * g4 + 1];
                o[4 * g4 + 1] = o[4 * g4 + 2];
                o[4 * g4 + 2] = t1;
              }
            }
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = 0u;
          }
        };
        if (p.S == 1) {
          // bf16 out: each lane stores its head's 64 bytes per chunk directly (staging
          // measured no faster for these narrower rows).
#pragma unroll 1
          for (int cc = 0; cc < 4; ++cc) {
            const int dc = d0 + cc * 32;
            uint32_t o[32];
            load_o_chunk(o, hc * 128 + cc * 32, dc < kNope);
            if (head_ok) {
              uint4* dstv = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.out) + (orow_idx * kLatent + dc) * 2);
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                uint32_t wv[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                  wv[e] = bf16x2_bits(__floats2bfloat162_rn(__uint_as_float(o[8 * i + 2 * e]) * factor,
                                                            __uint_as_float(o[8 * i + 2 * e + 1]) * factor));
                dstv[i] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
              }
            }
            __syncwarp();
          }
        } else {
          // fp32 partials: a 128-byte staging row holds one 32-dim chunk.
#pragma unroll 1
          for (int cc = 0; cc < 4; ++cc) {
            const int dc = d0 + cc * 32;  // first output dim of the chunk
            uint32_t o[32];
            load_o_chunk(o, hc * 128 + cc * 32, dc < kNope);
#pragma unroll
            for (int g = 0; g < 8; ++g)
              *reinterpret_cast<float4*>(wst + ln * 128 + ((g ^ (ln & 7)) << 4)) =
                  make_float4(__uint_as_float(o[4 * g]) * factor, __uint_as_float(o[4 * g + 1]) * factor,
                              __uint_as_float(o[4 * g + 2]) * factor, __uint_as_float(o[4 * g + 3]) * factor);
            __syncwarp();
            float4 v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int r = 4 * i + (ln >> 3), g = ln & 7;  // row r, granule g (dims 4g..4g+3)
              v[i] = *reinterpret_cast<const float4*>(wst + r * 128 + ((g ^ (r & 7)) << 4));
            }
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int r = 4 * i + (ln >> 3), g = ln & 7;
              if (head0 + r < p.H) *reinterpret_cast<float4*>(p.o_part + (orow0 + r) * kLatent + dc + 4 * g) = v[i];
            }
          }
        }
      }
      if (head_ok && half == 0 && hc == 0) {
        if (p.S > 1) p.lse_part[orow_idx] = lse_v;
        else if (p.lse != nullptr) p.lse[orow_idx] = lse_v;
      }
      // O, Q and red[] are reused by the next item: every thread's reads end here.
      tc_fence_before();
      warp_arrive(&m->sgrp);
      if (!(ok = wait_bar_warp(&m->sgrp, sgrp_phase, m))) break;
      sgrp_phase ^= 1u;
      tc_fence_after();
    }
    if (!ok) record_abort(m, p.status);
  } else {
    regs_dec<kProducerRegs>();
    // ------------------------------------------------------------ gather + dequant
    const int pt = tid - kSoftmaxThreads;
    if (pt < 32) {
      mma_warp<true>(smem, m, p, cid, items, tmem, pt, peer);
    } else if (pt < 64) {
      mma_warp<false>(smem, m, p, cid, items, tmem, pt - 32, peer);
    } else if (pt < 96) {
      if constexpr (TMA) {
        if (half == 0)
          loader_warp<0>(smem, m, p, &kp.map[0], cid, items, pt - 64);
        else
          loader_warp<1>(smem, m, p, &kp.map[1], cid, items, pt - 64);
      }
    } else if constexpr (TMA) {
      if (half == 0)
        produce_tma<0>(smem, m, p, cid, items, pt - 96);
      else
        produce_tma<1>(smem, m, p, cid, items, pt - 96);
    } else {
      if (half == 0)
        produce_direct<0>(smem, m, p, cid, items, pt - 96);
      else
        produce_direct<1>(smem, m, p, cid, items, pt - 96);
    }
  }

  // Wind down: nobody may leave while the peer can still arrive on this CTA's barriers,
  // and TMEM is freed only after every tcgen05 access of this CTA is done.
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

int attn_ctas_per_split() { return 2; }

int attn_pairs(int64_t items, int sms) {
  const int64_t cap = sms >= 2 ? sms / 2 : 1;
  return (int)(items < cap ? (items > 0 ? items : 1) : cap);
}

size_t attn_xchg_bytes(int pairs) { return (size_t)pairs * 2 * kXchgRegion; }

namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
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

// The cache as a 2-D tensor of u16 whose row y covers bytes [16y, 16y + 576) (every data
// row of the cache starts at a multiple of 16 bytes when P * 584 is one); a gather box
// of one row covers the half's bytes.  False when the view does not apply.
bool make_gather_maps(const AttnParams& p, CUtensorMap* maps) {
  if (((int64_t)p.P * kRowBytes) % 16 != 0 || (reinterpret_cast<uintptr_t>(p.cache) & 15u) != 0) return false;
  const int64_t bytes = p.num_pages * p.P * kRowBytes;
  const int64_t rows = (bytes - kDataBytes) / 16 + 1;
  if (rows < 1 || rows >= ((int64_t)1 << 31)) return false;
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t gdim[2] = {(cuuint64_t)(kDataBytes / 2), (cuuint64_t)rows};
  const cuuint64_t gstride[1] = {16};
  const cuuint32_t estr[2] = {1, 1};
  const cuuint32_t box0[2] = {(cuuint32_t)(RawFmt<0>::DATA / 2), 1};
  const cuuint32_t box1[2] = {(cuuint32_t)(RawFmt<1>::DATA / 2), 1};
  void* base = const_cast<uint8_t*>(p.cache);
  return enc(&maps[0], CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, base, gdim, gstride, box0, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS &&
         enc(&maps[1], CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, base, gdim, gstride, box1, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace

cudaError_t launch_attn(const AttnParams& p, cudaStream_t s) {
  if (p.T == 0) return cudaSuccess;
  KernelParams kp;
  kp.p = p;
  const bool tma = make_gather_maps(p, kp.map);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static bool attr_done[2][64] = {};
  if (dev < 64 && !attr_done[tma][dev]) {
    e = tma ? cudaFuncSetAttribute(attn_pair_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)kSmemBytes)
            : cudaFuncSetAttribute(attn_pair_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_done[tma][dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * p.G, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return tma ? cudaLaunchKernelEx(&cfg, attn_pair_kernel<true>, kp) : cudaLaunchKernelEx(&cfg, attn_pair_kernel<false>, kp);
}

}  // namespace smd
