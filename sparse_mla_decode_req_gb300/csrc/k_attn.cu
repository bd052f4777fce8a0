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
// heads x 512 dims in fp32 would fill all 512 TMEM columns, so a (token, split) work
// item is owned by a cluster of two CTAs, CTA c holding latent dims [256c, 256c+256) of
// K/V and of O:
//
//   TMEM (per CTA, 512 columns): Q half [0,128) as the A operand of QK (bf16 pairs), the
//   S partial [128,256), the O half [256,512).
//   SMEM: 2 stages x [128 rows x 256 dims] bf16 (128B-swizzled, 64 KB each), P as bf16
//   [128 heads x 128 rows] (32 KB, the A operand of PV), and a ring of raw cache rows.
//
// The launch is persistent: G = min(items, SMs / 2) pairs, pair c taking the work items
// c, c + G, ...; the tile sequence (and every barrier phase) runs on across items, so the
// producers prefetch the next item's rows while the current one finishes.
//
// Producers: two groups of four warps, group g owning stage g and the tiles 2x + g of the
// CTA's tile sequence.  A group copies each 32-row chunk of its tile half (the CTA's half
// of every 584-byte row, plus the 8-byte scale row) into a 3-slot raw ring with 16-byte
// cp.async (half a warp per 256-byte row segment, so every warp copy reads whole
// contiguous segments; rows that are masked copy a zero row instead), then dequantises
// the chunk from shared memory into the swizzled stage.
//
// Per 128-row tile j: S_c = Q_c K_c^T (M128 N128 K256, A from TMEM); the softmax threads
// load S_c into registers, which frees the S columns at once so QK of tile j+1 overlaps
// the rest of tile j; they send S_c (in log2 units) to the peer through an L2-resident
// exchange buffer and add the peer's partial, so both CTAs hold the 512-wide scores;
// online softmax; P to shared memory; O_c += P V_c (M128 N256 K128, the stage read
// MN-major).  Every QK flop is done once across the pair.
//
// Exchange format: each thread's 64 partials travel as int16 fixed point scaled by their
// largest magnitude (absolute error <= max|partial| * 2^-16 <= 2^-10 in log2 units) when
// that magnitude is at most 64, and as exact fp32 otherwise (a negative scale flags it).
// The running max only moves when it grows by more than 2^8, so O is rarely rescaled.
//
// Roles: warps 0-7 softmax + epilogue (two threads per head, 64 score columns each;
// thread 0 also issues the UMMAs and warp 0 owns the TMEM allocation), warps 8-15
// gather/dequant.  Every wait is bounded; a wait that gives up records bit 0 in the
// status word and the CTA winds down (draining its UMMAs, freeing TMEM).
#include <cuda.h>

#include "smd_device.cuh"
#include "smd_internal.h"

namespace smd {
namespace {

constexpr int kTile = kTileRows;            // 128 gathered rows per tile
constexpr int kDHalf = 256;                 // latent dims per CTA
constexpr int kSoftmaxThreads = 256;        // warps 0-7
constexpr int kGroupThreads = 128;          // one producer group = 4 warps
constexpr int kThreads = kSoftmaxThreads + 2 * kGroupThreads;
constexpr uint32_t kSoftmaxRegs = 168, kProducerRegs = 88;
static_assert(kSoftmaxThreads * kSoftmaxRegs + 2 * kGroupThreads * kProducerRegs == 65536, "register split");
constexpr int kProducerThreads = 2 * kGroupThreads;  // warps 8-15
constexpr int kChunkRows = 64;              // rows per raw chunk (two per tile)
constexpr int kRingSlots = 3;               // raw chunk slots
constexpr uint32_t kSlab = kTile * 128;     // [128 rows x 64 dims] bf16 = 16 KB
constexpr uint32_t kStageBytes = 4 * kSlab; // 64 KB
constexpr uint32_t kOffP = 2 * kStageBytes;              // P: 2 slabs [128 heads x 64 rows]
constexpr uint32_t kOffRing = kOffP + 2 * kSlab;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColQ = 0, kColS = 128, kColO = 256;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far beyond any legitimate wait
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: p <= 2^8 between rescales
constexpr float kQMax = 32767.f;           // int16 range of the exchanged partials
constexpr float kFixedMax = 64.f;          // largest |partial| (log2 units) sent as int16

// A raw chunk of one half: 64 rows of the half's data bytes (as the TMA gathers write
// them, back to back), then the 64 rows' 8-byte scale rows.
template <int HALF>
struct RawFmt {
  static constexpr int NN = HALF == 0 ? 16 : 12;     // NoPE 16-byte pieces per row
  static constexpr int NR = HALF == 0 ? 0 : 8;       // RoPE pieces per row
  static constexpr int NP = NN + NR;
  static constexpr int DATA = NP * 16;               // 256 / 320 bytes of a row
  static constexpr int SCALES = kChunkRows * DATA;   // offset of the scale rows
  static constexpr int SLOT = SCALES + kChunkRows * 8;
  static constexpr int BYTE0 = HALF == 0 ? 0 : 256;  // first row byte of the half
  static constexpr int CODE0 = HALF == 0 ? 0 : 4;    // first scale code of the half
};
constexpr uint32_t kRingBytes = kRingSlots * RawFmt<1>::SLOT;
constexpr uint32_t kOffMisc = kOffRing + kRingBytes;

// Exchange buffer of one CTA (what its peer writes into): 16 pieces x 256 threads x 16 B
// (int16 mode uses the first 8 pieces), then one scale per thread.
constexpr uint32_t kXchgData = 16u * kSoftmaxThreads * 16u;
constexpr uint32_t kXchgRegion = kXchgData + kSoftmaxThreads * 4u;

struct Misc {
  uint64_t kfull[2];         // producers -> issuer: stage filled (224 converter arrivals)
  uint64_t kempty[2];        // PV commit -> producers: stage consumed
  uint64_t sfull;            // QK commit -> softmax: S partial ready
  uint64_t sfree;            // softmax -> issuer: S loaded into registers (256 arrivals)
  uint64_t pfull;            // softmax -> issuer: P in shared memory, O rescaled (256 arrivals)
  uint64_t pvdone;           // PV commit -> softmax: P buffer and O free again
  uint64_t xfull;            // peer softmax -> softmax: peer partial written (256 remote arrivals)
  uint64_t xempty;           // peer softmax -> softmax: the peer's P slices are free (256 remote)
  uint64_t odone;            // last PV commit of an item -> softmax: O final
  uint64_t drain;            // issuer self-drain before TMEM is freed after a failed wait
  uint64_t sgrp;             // softmax-group rendezvous (256 arrivals per use)
  uint64_t qready;           // softmax -> issuer: an item's Q is in TMEM (256 arrivals)
  uint64_t rawfull[kRingSlots];   // raw chunk landed (loader expect-tx + 32 scale-copy arrivals)
  uint64_t rawempty[kRingSlots];  // raw chunk converted (224 converter arrivals)
  uint64_t hpair[4];         // warps w and w+4 (the two threads of heads 32w..32w+31): 64
  uint32_t tmem_base;
  uint32_t abort;
  uint32_t mask[2][4];              // valid-row bit masks of each stage's 32-row quarters
  uint32_t maskring[kRingSlots][2]; // valid-row masks of each raw chunk
  float red[2][2][128];             // per-column-half tile maxima, then final denominators
  float xscale[kSoftmaxThreads];    // scale of each thread's received partials (< 0: fp32 in L2)
};
// The stages need 1024-byte alignment; dynamic shared memory starts 1024-aligned here
// (checked at run time), so no slack is reserved.
constexpr uint32_t kSmemBytes = kOffMisc + sizeof(Misc);
static_assert(kSmemBytes <= 232448, "shared memory budget");

__device__ __align__(16) uint8_t g_zero_row[320];  // source of the copies of masked rows

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

// The same wait done by a whole warp, with a warp-uniform result, so that a warp never
// splits into lanes that go on and lanes that leave (which would strand the first at the
// next warp-collective instruction).
__device__ __forceinline__ bool wait_bar_warp(uint64_t* bar, uint32_t parity, const Misc* m,
                                              bool cluster_acquire = false) {
  const bool r = wait_bar(bar, parity, m, cluster_acquire);
  return __all_sync(0xffffffffu, r);
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

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async8(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
// Arrive on `bar` once every cp.async this thread issued so far has landed.
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void st_global_v4(void* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// int16 fixed-point codec without conversion instructions.  Encode: adding 1.5 * 2^23
// rounds v (|v| <= 32767) to the nearest integer held in the low mantissa bits, whose low
// 16 bits are then its two's complement.  Decode: flipping the sign bit of a 16-bit field
// and OR-ing 0x4B000000 gives the float 2^23 + q + 32768.
constexpr float kMagicRound = 12582912.0f;      // 1.5 * 2^23
constexpr float kMagicDecode = 8421376.0f;      // 2^23 + 32768
__device__ __forceinline__ uint32_t pack_q16(float a, float b, float enc) {
  const uint32_t ia = __float_as_uint(fmaf(a, enc, kMagicRound));
  const uint32_t ib = __float_as_uint(fmaf(b, enc, kMagicRound));
  return __byte_perm(ia, ib, 0x5410u);
}
__device__ __forceinline__ float q16_lo_biased(uint32_t w) {
  return __uint_as_float(((w & 0xFFFFu) ^ 0x8000u) | 0x4B000000u);
}
__device__ __forceinline__ float q16_hi_biased(uint32_t w) {
  return __uint_as_float(((w >> 16) ^ 0x8000u) | 0x4B000000u);
}

// One (token, split) work item.
struct Item {
  int t, split, tile_begin, n;  // n = tiles of the item (0 for a split past the end)
};
__device__ __forceinline__ Item item_of(const AttnParams& p, int w) {
  Item it;
  it.t = w / p.S;
  it.split = w - it.t * p.S;
  it.tile_begin = it.split * p.tiles_per_split;
  const int ntok = (p.N + kTile - 1) / kTile;
  it.n = max(0, min(ntok, it.tile_begin + p.tiles_per_split) - it.tile_begin);
  return it;
}

// Walks the tiles of the items w0, w0 + G, ... in order, skipping items without tiles.
struct TileCursor {
  int w, k, n, G, items;
  int64_t row0;   // gidx offset of the tile's first row
  int rows;       // rows of the tile inside the token's entry list (1..128)
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

// Walks the 64-row chunks (two per tile) of the CTA's tile sequence.
struct ChunkCursor {
  TileCursor t;
  int c;  // chunk of the tile
  __device__ void init(const AttnParams& p, int w0, int G, int items) {
    t.init(p, w0, G, items);
    c = 0;
  }
  __device__ bool valid() const { return t.valid(); }
  __device__ void next(const AttnParams& p) {
    if (c == 0) {
      c = 1;
    } else {
      c = 0;
      t.next(p);
    }
  }
  // gidx offset of the chunk's first row and the rows it has inside the entry list
  __device__ int64_t row0() const { return t.row0 + c * kChunkRows; }
  __device__ int rows() const { return t.rows - c * kChunkRows; }
};

// Dequantises the 16-byte NoPE piece `k` of a raw row (scale code from its scale row)
// into the stage, or zeros when the row is masked.
// (elements in the (d0, d2, d1, d3) order of dequant16_perm_*; `fast` must be warp-uniform
// and true only when no piece of the warp holds a NaN byte or a code above 134).
template <bool FAST>
__device__ __forceinline__ void convert_nope(uint8_t* stage, int srow, int k, uint4 raw, uint32_t code, bool valid) {
  uint4 lo, hi;
  if (!valid) {
    raw = make_uint4(0, 0, 0, 0);
    code = 0;
  }
  if constexpr (FAST)
    dequant16_perm_fast(raw, code, lo, hi);
  else
    dequant16_perm_exact(raw, code, lo, hi);
  *reinterpret_cast<uint4*>(stage + stage_off(srow, k * 16)) = lo;
  *reinterpret_cast<uint4*>(stage + stage_off(srow, k * 16 + 8)) = hi;
}

// The control warp (warp 8): a non-blocking event loop that (TMA mode) puts the raw
// chunks in flight, four rows per TMA gather, running as far ahead as the 3-slot ring
// allows, and issues every UMMA of the CTA from lane 0: QK of a tile once its stage is
// filled and S is free (or, for an item's first tile, once the item's Q is in TMEM), PV
// of a tile once its P is in shared memory.  Keeping the issue off the softmax warps
// keeps them in step with each other.
constexpr int kConverters = kProducerThreads - 32;

template <int HALF, bool TMA>
__device__ __forceinline__ void control_warp(uint8_t* smem, Misc* m, const AttnParams& p, const CUtensorMap* map,
                                             int cid, int items, uint32_t tmem, int lane) {
  using F = RawFmt<HALF>;
  const CacheView cv = make_cache_view(p.cache, p.P);
  const int64_t n_slots = p.num_pages * p.P;
  uint8_t* ring = smem + kOffRing;
  constexpr uint32_t kIdescQK = idesc_bf16_f32(128, kTile, false, false);
  constexpr uint32_t kIdescPV = idesc_bf16_f32(128, kDHalf, false, true);
  const uint32_t a_stage = smem_u32(smem);
  const uint32_t a_p = smem_u32(smem + kOffP);
  auto issue_qk = [&](int jj) {  // S = Q K^T for tile jj
    const uint32_t base = a_stage + (jj & 1) * kStageBytes;
#pragma unroll
    for (int kk = 0; kk < kDHalf / 16; ++kk)
      umma_ts(tmem + kColS, tmem + kColQ + kk * 8, desc_sw128(base + (kk >> 2) * kSlab + (kk & 3) * 32, 16, 1024),
              kIdescQK, kk > 0 ? 1u : 0u);
    umma_commit(&m->sfull);
  };
  auto issue_pv = [&](int jj, bool first) {  // O += P V for tile jj, then free its stage and P
    const uint32_t base = a_stage + (jj & 1) * kStageBytes;
#pragma unroll
    for (int kk = 0; kk < kTile / 16; ++kk)
      umma_ss(tmem + kColO, desc_sw128(a_p + (kk >> 2) * kSlab + (kk & 3) * 32, 16, 1024),
              desc_sw128(base + kk * 2048, kSlab, 1024), kIdescPV, (!first || kk > 0) ? 1u : 0u);
    umma_commit(&m->kempty[jj & 1]);
    umma_commit(&m->pvdone);
  };
  auto load_gidx = [&](const ChunkCursor& c, int r) -> int32_t {
    if (!c.valid() || r >= c.rows()) return -1;
    const int32_t v = ldg_nc_s32(p.gidx + c.row0() + r);
    return ((int64_t)v >= n_slots) ? -1 : v;
  };
  const int32_t rows_per_page16 = p.P * (kRowBytes / 8) / 2;  // P * 584 / 16 (TMA mode: P even)
  auto row16 = [&](int32_t sl) -> int32_t {  // 16-byte row index of slot sl's data row
    int32_t page, off;
    slot_page_off(cv, sl, page, off);
    return page * rows_per_page16 + off * (kDataBytes / 16);
  };
  auto scale_row = [&](int32_t sl) -> const uint8_t* {
    if (sl < 0) return g_zero_row;
    int32_t page, off;
    slot_page_off(cv, sl, page, off);
    return cv.base + (int64_t)page * cv.page_bytes + cv.scale_start + (int64_t)off * kScaleBytes;
  };

  // chunk issue state (TMA mode): slots of rows lane and lane + 32 of the next two chunks
  ChunkCursor iss, pre;
  iss.init(p, cid, p.G, items);
  pre = iss;
  int32_t ga0 = -1, gb0 = -1, ga1 = -1, gb1 = -1;
  if (TMA) {
    ga0 = load_gidx(pre, lane);
    gb0 = load_gidx(pre, lane + 32);
    pre.next(p);
    ga1 = load_gidx(pre, lane);
    gb1 = load_gidx(pre, lane + 32);
  }
  int q_issue = 0;
  // MMA issue state
  TileCursor qkc, pvc;
  qkc.init(p, cid, p.G, items);
  pvc = qkc;
  int jq = 0, jp = 0;  // tile sequence numbers of the next QK and PV
  int neq = 0;         // index (among items with tiles) of qkc's item
  uint64_t idle_since = 0;

  for (;;) {
    bool progress = false;
    if (TMA && iss.valid()) {
      const int slot = q_issue % kRingSlots;
      bool can = q_issue < kRingSlots || mbar_test_wait(&m->rawempty[slot], (q_issue / kRingSlots - 1) & 1);
      can = __shfl_sync(0xffffffffu, can, 0);
      if (can) {
        const uint32_t base = smem_u32(ring + slot * F::SLOT);
        const bool va = ga0 >= 0, vb = gb0 >= 0;
        const uint32_t ba = __ballot_sync(0xffffffffu, va), bb = __ballot_sync(0xffffffffu, vb);
        if (lane == 0) {
          m->maskring[slot][0] = ba;
          m->maskring[slot][1] = bb;
          mbar_arrive_expect_tx(&m->rawfull[slot], kChunkRows * F::DATA);  // releases maskring
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
        cp_async8(base + F::SCALES + lane * 8, scale_row(ga0));
        cp_async8(base + F::SCALES + (lane + 32) * 8, scale_row(gb0));
        cp_async_arrive(&m->rawfull[slot]);
        ++q_issue;
        iss.next(p);
        ga0 = ga1;
        gb0 = gb1;
        pre.next(p);
        ga1 = load_gidx(pre, lane);
        gb1 = load_gidx(pre, lane + 32);
        progress = true;
      }
    }
    if (qkc.valid()) {
      bool can = false;
      if (lane == 0) {
        can = mbar_test_wait(&m->kfull[jq & 1], (jq >> 1) & 1) &&
              (qkc.k == 0 ? mbar_test_wait(&m->qready, neq & 1) : mbar_test_wait(&m->sfree, (jq - 1) & 1));
        if (can) {
          tc_fence_after();
          issue_qk(jq);
        }
      }
      can = __shfl_sync(0xffffffffu, can, 0);
      if (can) {
        const bool item_end = qkc.k + 1 == qkc.n;
        ++jq;
        qkc.next(p);
        neq += item_end ? 1 : 0;
        progress = true;
      }
    }
    if (pvc.valid() && jp < jq) {
      bool can = false;
      if (lane == 0) {
        can = mbar_test_wait(&m->pfull, jp & 1);
        if (can) {
          tc_fence_after();
          issue_pv(jp, pvc.k == 0);
          if (pvc.k + 1 == pvc.n) umma_commit(&m->odone);
        }
      }
      can = __shfl_sync(0xffffffffu, can, 0);
      if (can) {
        ++jp;
        pvc.next(p);
        progress = true;
      }
    }
    if (!(TMA && iss.valid()) && !qkc.valid() && !pvc.valid()) break;
    if (progress) {
      idle_since = 0;
    } else {
      if (aborted(m)) break;
      const uint64_t now = globaltimer_ns();
      if (idle_since == 0) {
        idle_since = now;
      } else if (now - idle_since > kWaitLimitNs) {
        if (lane == 0) record_abort(m, p.status);
        break;
      }
      // Nothing ready: sleep on the P buffer of the oldest pending PV (the event the
      // critical path waits for), or briefly when no PV is pending.
      if (pvc.valid() && jp < jq)
        (void)mbar_try_wait_hint(&m->pfull, jp & 1, 1000);
      else
        __nanosleep(64);
    }
  }
  if (lane == 0) {
    umma_commit(&m->drain);  // every issued UMMA lands before TMEM is freed
    mbar_wait_bounded(&m->drain, 0, kWaitLimitNs);
  }
  asm volatile("cp.async.wait_all;" ::: "memory");  // no copy may land after the CTA is gone
  __syncwarp();
}

// The converter warps (9-15, ct = 0..223) of the TMA mode: each raw chunk the control
// warp put in flight is dequantised into the stage of its tile.

template <int HALF>
__device__ __forceinline__ void produce_tma(uint8_t* smem, Misc* m, const AttnParams& p, int cid, int items, int ct) {
  using F = RawFmt<HALF>;
  uint8_t* ring = smem + kOffRing;
  ChunkCursor conv;
  conv.init(p, cid, p.G, items);
  for (int q = 0; conv.valid(); ++q) {
    const int slot = q % kRingSlots;
    const int c = conv.c;
    const int j = q >> 1;   // tile sequence number
    const int s = j & 1;    // its stage
    uint8_t* stage = smem + s * kStageBytes;
    // A wait that gives up flags the CTA; the converters still run their remaining chunk
    // sequence without converting, and every later wait returns at once.
    bool live = c != 0 || j < 2 || wait_bar(&m->kempty[s], ((j >> 1) - 1) & 1, m);
    live = live && wait_bar(&m->rawfull[slot], (q / kRingSlots) & 1, m);
    if (!live) record_abort(m, p.status);
    live = live && !aborted(m);
    if (live) {
      const uint8_t* raw = ring + slot * F::SLOT;
      const uint32_t mk0 = m->maskring[slot][0], mk1 = m->maskring[slot][1];
      auto valid_row = [&](int r) { return (((r < 32 ? mk0 : mk1) >> (r & 31)) & 1u) != 0u; };
      // NoPE: 64 rows x NN pieces; consecutive threads take consecutive pieces of a row.
      // The pieces are loaded first, then converted on the fast path unless a piece of
      // the warp needs the exact one.
      constexpr int NI = (kChunkRows * F::NN + kConverters - 1) / kConverters;
      uint4 v[NI];
      uint32_t code[NI];
      bool clean = true;
#pragma unroll
      for (int i = 0; i < NI; ++i) {
        const int pc = ct + kConverters * i;
        const int r = pc / F::NN, k = pc - r * F::NN;
        v[i] = make_uint4(0, 0, 0, 0);
        code[i] = 0;
        if (pc < kChunkRows * F::NN) {
          v[i] = *reinterpret_cast<const uint4*>(raw + r * F::DATA + k * 16);
          code[i] = raw[F::SCALES + r * 8 + F::CODE0 + (k >> 2)];
          clean = clean && code[i] <= 134u && fp8x16_no_nan(v[i]);
        }
      }
      const bool fast = __all_sync(0xffffffffu, clean);
#pragma unroll
      for (int i = 0; i < NI; ++i) {
        const int pc = ct + kConverters * i;
        const int r = pc / F::NN, k = pc - r * F::NN;
        if (pc < kChunkRows * F::NN) {
          if (fast)
            convert_nope<true>(stage, c * kChunkRows + r, k, v[i], code[i], valid_row(r));
          else
            convert_nope<false>(stage, c * kChunkRows + r, k, v[i], code[i], valid_row(r));
        }
      }
      if constexpr (F::NR > 0) {
#pragma unroll
        for (int i = 0; i < (kChunkRows * F::NR + kConverters - 1) / kConverters; ++i) {
          const int pc = ct + kConverters * i;
          if (pc < kChunkRows * F::NR) {
            const int r = pc / F::NR, k = pc - r * F::NR;
            uint4 v = *reinterpret_cast<const uint4*>(raw + r * F::DATA + (F::NN + k) * 16);
            if (!valid_row(r)) v = make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(stage + stage_off(c * kChunkRows + r, 192 + k * 8)) = scrub_bf16x8(v);
          }
        }
      }
      if (ct == 0) {
        m->mask[s][2 * c] = mk0;
        m->mask[s][2 * c + 1] = mk1;
      }
    }
    mbar_arrive(&m->rawempty[slot]);
    if (c == 1) {
      fence_async_smem();
      mbar_arrive(&m->kfull[s]);
    }
    conv.next(p);
  }
}

// Fallback producer for caches whose rows are only 8-byte aligned (pages of an odd slot
// count) or too large for 32-bit TMA row coordinates: every thread loads its pieces
// straight from global memory (no ring), one 64-row chunk at a time.
template <int HALF>
__device__ __forceinline__ void produce_direct(uint8_t* smem, Misc* m, const AttnParams& p, int cid, int items,
                                               int ct) {
  using F = RawFmt<HALF>;
  const CacheView cv = make_cache_view(p.cache, p.P);
  const int64_t n_slots = p.num_pages * p.P;
  ChunkCursor conv;
  conv.init(p, cid, p.G, items);
  for (int q = 0; conv.valid(); ++q) {
    const int c = conv.c;
    const int j = q >> 1;
    const int s = j & 1;
    uint8_t* stage = smem + s * kStageBytes;
    bool live = c != 0 || j < 2 || wait_bar(&m->kempty[s], ((j >> 1) - 1) & 1, m);
    if (!live) record_abort(m, p.status);
    live = live && !aborted(m);
    auto slot_of = [&](int r) -> int32_t {
      if (r >= conv.rows()) return -1;
      const int32_t v = ldg_nc_s32(p.gidx + conv.row0() + r);
      return ((int64_t)v >= n_slots) ? -1 : v;
    };
    if (live) {
      for (int pc = ct; pc < kChunkRows * F::NP; pc += kConverters) {
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
          convert_nope<false>(stage, c * kChunkRows + r, k, v, code, g >= 0);
        else
          *reinterpret_cast<uint4*>(stage + stage_off(c * kChunkRows + r, 192 + (k - F::NN) * 8)) = scrub_bf16x8(v);
      }
      if (ct < 64) {  // valid-row masks of the chunk's two 32-row quarters
        const uint32_t bits = __ballot_sync(0xffffffffu, slot_of(ct) >= 0);
        if ((ct & 31) == 0) m->mask[s][2 * c + (ct >> 5)] = bits;
      }
    }
    if (c == 1) {
      fence_async_smem();
      mbar_arrive(&m->kfull[s]);
    }
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
    if (tid == 0 && p.status != nullptr) atomicOr(p.status, 2u);
    return;
  }

  if (tid == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&m->kfull[s], kConverters);
      mbar_init(&m->kempty[s], 1);
    }
    for (int r = 0; r < kRingSlots; ++r) {
      mbar_init(&m->rawfull[r], 1 + 32);  // the loader's expect-tx + its 32 lanes' scale copies
      mbar_init(&m->rawempty[r], kConverters);
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
    mbar_init(&m->qready, kSoftmaxThreads);
    for (int i = 0; i < 4; ++i) mbar_init(&m->hpair[i], 64);
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

  // Register budget: the launch gives 128 per thread (512 x 128 = the whole file); the
  // softmax warpgroups take 168 and the producer warpgroups keep 88 (2 x 128 x (168 + 88)
  // = 65536).
  if (warp < 8) {
    regs_inc<kSoftmaxRegs>();
    // ------------------------------------------------------------ softmax + UMMA issue
    // Thread (h, hc): head h = TMEM lane h, column half hc of every 128-column tile.
    const int h = tid & 127;
    const int hc = warp >> 2;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float sl2 = p.scale * kLog2e;
    // Exchange regions are recomputed at each use (kernel parameters live in the constant
    // bank), which keeps them out of the register budget.
    auto xregion = [&](uint32_t rank) { return p.xchg + ((size_t)cid * 2 + rank) * kXchgRegion; };
    bool ok = true;
    uint32_t sgrp_phase = 0;
    int j = 0;       // tile sequence number (runs on across items)
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
        if (n > 0) mbar_arrive(&m->qready);  // the issuer may start QK of the item's first tile
      }

      float m_ref = -INFINITY;  // reference max (log2 domain) the weights are taken against
      float l_run = 0.f;        // this thread's share of the denominator relative to m_ref
      for (int k = 0; k < n && ok; ++k, ++j) {
        const int s = j & 1;
        if (!(ok = wait_bar_warp(&m->sfull, j & 1, m))) break;
        tc_fence_after();
        float x[64];
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
          uint32_t r[32];
          tmem_ld32(tmem + lane_base + kColS + hc * 64 + c2 * 32, r);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) x[c2 * 32 + i] = __uint_as_float(r[i]) * sl2;
        }
        // S is in registers: QK of the next tile may go as soon as every thread has
        // loaded S and the next stage is filled.
        tc_fence_before();
        mbar_arrive(&m->sfree);

        // Exchange.  The peer's partials land in this thread's 128-byte slice of the P
        // buffer, which is free from the end of PV of the previous tile until this tile's
        // P is written: say so to the peer, then send this thread's partials (log2 units,
        // int16 fixed point) into the peer's slice of the same thread over DSMEM.  A block
        // beyond the fixed-point range goes through the L2 exchange buffer as fp32.
        if (j > 0 && !(ok = wait_bar_warp(&m->pvdone, (j - 1) & 1, m))) break;
        tc_fence_after();
        mbar_arrive_cluster(mapa(smem_u32(&m->xempty), peer));
        uint8_t* slice = sP + hc * kSlab;
        float amax = 0.f;
#pragma unroll
        for (int c = 0; c < 64; ++c) amax = fmaxf(amax, fabsf(x[c]));
        const bool fixed = amax <= kFixedMax;  // false for NaN too: those go as fp32
        if (!(ok = wait_bar_warp(&m->xempty, j & 1, m, true))) break;
        const uint32_t peer_slice = mapa(smem_u32(slice), peer);
        if (fixed) {
          const float enc = amax > 0.f ? kQMax / amax : 0.f;
#pragma unroll
          for (int i = 0; i < 8; ++i)
            st_cluster_v4(peer_slice + sw128_off(h, i), pack_q16(x[8 * i], x[8 * i + 1], enc),
                          pack_q16(x[8 * i + 2], x[8 * i + 3], enc), pack_q16(x[8 * i + 4], x[8 * i + 5], enc),
                          pack_q16(x[8 * i + 6], x[8 * i + 7], enc));
        } else {
          uint8_t* dst = xregion(peer) + tid * 16;
#pragma unroll
          for (int i = 0; i < 16; ++i)
            st_global_v4(dst + i * (kSoftmaxThreads * 16), __float_as_uint(x[4 * i]), __float_as_uint(x[4 * i + 1]),
                         __float_as_uint(x[4 * i + 2]), __float_as_uint(x[4 * i + 3]));
        }
        asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(mapa(smem_u32(&m->xscale[tid]), peer)),
                     "f"(fixed ? amax / kQMax : -1.f)
                     : "memory");
        mbar_arrive_cluster(mapa(smem_u32(&m->xfull), peer));

        // Receive the peer's partials and add them.
        if (!(ok = wait_bar_warp(&m->xfull, j & 1, m, true))) break;
        {
          const float dec = m->xscale[tid];
          if (dec >= 0.f) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const uint4 v = *reinterpret_cast<const uint4*>(slice + sw128_off(h, i));
              const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
              for (int qq = 0; qq < 4; ++qq) {  // (biased - magic) is the integer exactly
                x[8 * i + 2 * qq] = fmaf(q16_lo_biased(wv[qq]) - kMagicDecode, dec, x[8 * i + 2 * qq]);
                x[8 * i + 2 * qq + 1] = fmaf(q16_hi_biased(wv[qq]) - kMagicDecode, dec, x[8 * i + 2 * qq + 1]);
              }
            }
          } else {
            // fp32 partials from the L2 buffer, staged through the slice 8 pieces at a time
            const uint8_t* src = xregion(half) + tid * 16;
#pragma unroll
            for (int hb = 0; hb < 2; ++hb) {
#pragma unroll
              for (int i = 0; i < 8; ++i)
                cp_async16(smem_u32(slice + sw128_off(h, i)), src + (8 * hb + i) * (kSoftmaxThreads * 16));
              asm volatile("cp.async.wait_all;" ::: "memory");
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const uint4 v = *reinterpret_cast<const uint4*>(slice + sw128_off(h, i));
                x[32 * hb + 4 * i] += __uint_as_float(v.x);
                x[32 * hb + 4 * i + 1] += __uint_as_float(v.y);
                x[32 * hb + 4 * i + 2] += __uint_as_float(v.z);
                x[32 * hb + 4 * i + 3] += __uint_as_float(v.w);
              }
            }
          }
        }

        // The stage's valid-row masks (published by the producers before kfull).
        if (!(ok = wait_bar_warp(&m->kfull[s], (j >> 1) & 1, m))) break;
        const uint32_t mk0 = m->mask[s][2 * hc], mk1 = m->mask[s][2 * hc + 1];
        // Online softmax over this thread's 64 columns; both threads of head h agree on m_ref.
        float lmax = -INFINITY;
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const uint32_t bits = c < 32 ? mk0 : mk1;
          const float v = ((bits >> (c & 31)) & 1u) ? x[c] : -INFINITY;
          x[c] = v;
          lmax = fmaxf(lmax, v);
        }
        m->red[s][hc][h] = lmax;
        mbar_arrive(&m->hpair[warp & 3]);
        if (!(ok = wait_bar_warp(&m->hpair[warp & 3], j & 1, m))) break;
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
        // P buffer and O are free (PV of the previous tile is done, waited above).
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<uint4*>(sP + hc * kSlab + sw128_off(h, c)) =
              make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        if (k > 0 && __any_sync(0xffffffffu, upd)) {
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
        ok = !aborted(m);
      }
      if (!ok) break;
      if (n > 0) {
        if (!(ok = wait_bar_warp(&m->odone, ne_no & 1, m))) break;
        ++ne_no;
      }
      // Epilogue: head h, local dims [128 hc, 128 hc + 128) of this CTA's 256.
      tc_fence_after();
      m->red[0][hc][h] = l_run;  // every use of red[][] by the tile loop is over (odone)
      mbar_arrive(&m->sgrp);
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
        const float sink_nat = (p.sink != nullptr && head_ok) ? __ldg(p.sink + h) : -INFINITY;
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
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t o[32];
        if (o_live) {
          tmem_ld32(tmem + lane_base + kColO + hc * 128 + cc * 32, o);
          tmem_wait_ld();
          // NoPE columns hold dims in the (d0, d2, d1, d3) order of the stage
          if (d0 + cc * 32 < kNope) {
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
        if (!head_ok) continue;
        if (p.S == 1) {
          uint4* dstv = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.out) + (orow_idx * kLatent + d0 + cc * 32) * 2);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint32_t wv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              wv[e] = bf16x2_bits(__floats2bfloat162_rn(__uint_as_float(o[8 * i + 2 * e]) * factor,
                                                        __uint_as_float(o[8 * i + 2 * e + 1]) * factor));
            dstv[i] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
          }
        } else {
          float4* dstv = reinterpret_cast<float4*>(p.o_part + orow_idx * kLatent + d0 + cc * 32);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            dstv[i] = make_float4(__uint_as_float(o[4 * i]) * factor, __uint_as_float(o[4 * i + 1]) * factor,
                                  __uint_as_float(o[4 * i + 2]) * factor, __uint_as_float(o[4 * i + 3]) * factor);
        }
      }
      if (head_ok && half == 0 && hc == 0) {
        if (p.S > 1) p.lse_part[orow_idx] = lse_v;
        else if (p.lse != nullptr) p.lse[orow_idx] = lse_v;
      }
      // O, Q and red[] are reused by the next item: every thread's reads end here.
      tc_fence_before();
      mbar_arrive(&m->sgrp);
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
      if (half == 0)
        control_warp<0, TMA>(smem, m, p, &kp.map[0], cid, items, tmem, pt);
      else
        control_warp<1, TMA>(smem, m, p, &kp.map[1], cid, items, tmem, pt);
    } else if constexpr (TMA) {
      if (half == 0)
        produce_tma<0>(smem, m, p, cid, items, pt - 32);
      else
        produce_tma<1>(smem, m, p, cid, items, pt - 32);
    } else {
      if (half == 0)
        produce_direct<0>(smem, m, p, cid, items, pt - 32);
      else
        produce_direct<1>(smem, m, p, cid, items, pt - 32);
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
  const dim3 grid(2 * p.G, 1);
  if (tma)
    attn_pair_kernel<true><<<grid, kThreads, kSmemBytes, s>>>(kp);
  else
    attn_pair_kernel<false><<<grid, kThreads, kSmemBytes, s>>>(kp);
  return cudaGetLastError();
}

}  // namespace smd
