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
constexpr int kChunkRows = 32;
constexpr int kRingSlots = 3;               // raw chunk slots per producer group
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

// Raw ring row format of each half: the half's data bytes, then the 8-byte scale row,
// padded to a multiple of 16 bytes so that consecutive rows start 4 banks apart.
template <int HALF>
struct RawFmt {
  static constexpr int NN = HALF == 0 ? 16 : 12;     // NoPE 16-byte pieces per row
  static constexpr int NR = HALF == 0 ? 0 : 8;       // RoPE pieces per row
  static constexpr int NP = NN + NR;
  static constexpr int STRIDE = NP * 16 + 16;        // 272 / 336
  static constexpr int CHUNK = kChunkRows * STRIDE;  // 8704 / 10752
  static constexpr int BYTE0 = HALF == 0 ? 0 : 256;  // first row byte of the half
  static constexpr int CODE0 = HALF == 0 ? 0 : 4;    // first scale code of the half
};
constexpr uint32_t kRingBytes = 2 * kRingSlots * RawFmt<1>::CHUNK;
constexpr uint32_t kOffMisc = kOffRing + kRingBytes;

// Exchange buffer of one CTA (what its peer writes into): 16 pieces x 256 threads x 16 B
// (int16 mode uses the first 8 pieces), then one scale per thread.
constexpr uint32_t kXchgData = 16u * kSoftmaxThreads * 16u;
constexpr uint32_t kXchgRegion = kXchgData + kSoftmaxThreads * 4u;

struct Misc {
  uint64_t kfull[2];         // producer group g -> issuer: stage g filled (128 arrivals)
  uint64_t kempty[2];        // PV commit -> producer group: stage consumed
  uint64_t sfull;            // QK commit -> softmax: S partial ready
  uint64_t sfree;            // softmax -> issuer: S loaded into registers (256 arrivals)
  uint64_t pfull;            // softmax -> issuer: P in shared memory, O rescaled (256 arrivals)
  uint64_t pvdone;           // PV commit -> softmax: P buffer and O free again
  uint64_t xfull;            // peer softmax -> softmax: peer partial written (256 remote arrivals)
  uint64_t xempty;           // peer softmax -> softmax: peer read our last partial (256 remote)
  uint64_t odone;            // last PV commit of an item -> softmax: O final
  uint64_t drain;            // issuer self-drain before TMEM is freed after a failed wait
  uint64_t sgrp;             // softmax-group rendezvous (256 arrivals per use)
  uint64_t rawfull[2][kRingSlots];  // cp.async completion of a raw chunk (128 arrivals)
  uint64_t hpair[4];         // warps w and w+4 (the two threads of heads 32w..32w+31): 64
  uint32_t tmem_base;
  uint32_t abort;
  uint32_t mask[2][4];              // valid-row bit masks of each stage's four chunks
  uint32_t maskring[2][kRingSlots]; // valid-row mask of each raw chunk
  int32_t gbuf[2][kTile];           // converted slots of each group's next tile
  float red[2][2][128];             // per-column-half tile maxima, then final denominators
};
// The stages need 1024-byte alignment; dynamic shared memory starts 1024-aligned here
// (checked at run time), so no slack is reserved.
constexpr uint32_t kSmemBytes = kOffMisc + sizeof(Misc);
static_assert(kSmemBytes <= 232448, "shared memory budget");

__device__ __align__(16) uint8_t g_zero_row[16];  // source of the copies of masked rows

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
// Arrive on `bar` once every cp.async this thread issued so far has landed.
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void st_global_v4(void* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ float ld_global_cg_f32(const void* p) {
  float v;
  asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
  return v;
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

// A 16-byte piece of a cache row into shared memory: one copy when the row is 16-byte
// aligned, two 8-byte copies otherwise (pages of an odd slot count).
template <bool ALIGN16>
__device__ __forceinline__ void cp_piece(uint32_t dst, const uint8_t* src) {
  if constexpr (ALIGN16) {
    cp_async16(dst, src);
  } else {
    cp_async8(dst, src);
    cp_async8(dst + 8, src + 8);
  }
}

// The producer role of group `g` (128 threads, gt = 0..127) for this CTA's half.
template <int HALF, bool ALIGN16>
__device__ __forceinline__ void produce(uint8_t* smem, Misc* m, const AttnParams& p, int cid, int items, int g,
                                        int gt) {
  using F = RawFmt<HALF>;
  const CacheView cv = make_cache_view(p.cache, p.P);
  const int64_t n_slots = p.num_pages * p.P;
  const int gw = gt >> 5, lane = gt & 31;
  const uint32_t bar_id = 1 + g;
  uint8_t* ring = smem + kOffRing + g * kRingSlots * F::CHUNK;
  uint8_t* stage = smem + g * kStageBytes;

  // Tiles of this group: the CTA's tiles g, g+2, g+4, ...
  TileCursor conv, iss, pre;
  conv.init(p, cid, p.G, items);
  if (g == 1 && conv.valid()) conv.next(p);
  iss = conv;
  pre = conv;
  auto skip2 = [&](TileCursor& c) {
    if (c.valid()) c.next(p);
    if (c.valid()) c.next(p);
  };
  auto load_gidx = [&](const TileCursor& c) -> int32_t {
    if (!c.valid() || gt >= c.rows) return -1;
    const int32_t v = ldg_nc_s32(p.gidx + c.row0 + gt);
    return ((int64_t)v >= n_slots) ? -1 : v;
  };
  if (!conv.valid()) return;

  // Prologue: this tile's slots into gbuf, the next tile's in a register.
  m->gbuf[g][gt] = load_gidx(conv);
  skip2(pre);
  int32_t gpre = load_gidx(pre);
  named_bar_sync(bar_id, kGroupThreads);

  int iss_chunk = 0;  // chunk of `iss` the next issue copies
  int q_issue = 0;    // group-local chunk sequence number of the next issue
  auto issue = [&]() {
    const int slot = q_issue % kRingSlots;
    const uint32_t dst = smem_u32(ring + slot * F::CHUNK);
    const int32_t* gb = m->gbuf[g] + iss_chunk * kChunkRows;
    auto src_row = [&](int r, const uint8_t*& d, const uint8_t*& sc) {
      const int32_t s = gb[r];
      d = g_zero_row;
      sc = g_zero_row;
      if (s >= 0) {
        int32_t page, off;
        slot_page_off(cv, s, page, off);
        const uint8_t* pg = cv.base + (int64_t)page * cv.page_bytes;
        d = pg + (int64_t)off * kDataBytes + F::BYTE0;
        sc = pg + cv.scale_start + (int64_t)off * kScaleBytes;
      }
    };
#pragma unroll
    for (int i = 0; i < 4; ++i) {  // pieces 0..15: half a warp per 256-byte row segment
      const int r = gw * 8 + 2 * i + (lane >> 4), k = lane & 15;
      const uint8_t *d, *sc;
      src_row(r, d, sc);
      cp_piece<ALIGN16>(dst + r * F::STRIDE + k * 16, d == g_zero_row ? d : d + k * 16);
    }
    if (F::NP > 16) {  // pieces 16..19 of the second half: a quarter warp per row
      const int r = gw * 8 + (lane >> 2), k = 16 + (lane & 3);
      const uint8_t *d, *sc;
      src_row(r, d, sc);
      cp_piece<ALIGN16>(dst + r * F::STRIDE + k * 16, d == g_zero_row ? d : d + k * 16);
    }
    if (gw == 0) {  // scale rows, and the chunk's valid-row mask
      const uint8_t *d, *sc;
      src_row(lane, d, sc);
      cp_async8(dst + lane * F::STRIDE + F::NP * 16, sc);
      const uint32_t bits = __ballot_sync(0xffffffffu, gb[lane] >= 0);
      if (lane == 0) m->maskring[g][slot] = bits;
    }
    cp_async_arrive(&m->rawfull[g][slot]);
    ++q_issue;
    if (++iss_chunk == kTile / kChunkRows) {
      iss_chunk = 0;
      skip2(iss);
    }
  };

  // Up to kRingSlots chunks in flight (they all belong to the first tile).
  for (int i = 0; i < kRingSlots && iss.valid(); ++i) issue();

  const int cr = gt >> 2, cs = gt & 3;  // converter: row of the chunk, quarter of the row
  int q = 0;                            // group-local chunk sequence number
  for (int x = 0; conv.valid(); ++x) {
    for (int c = 0; c < kTile / kChunkRows; ++c, ++q) {
      const int slot = q % kRingSlots;
      // A wait that gives up flags the CTA; the group still runs its remaining chunk
      // sequence (without converting), so that every thread keeps meeting the group's
      // named barriers, and every later wait returns at once.
      bool live = c != 0 || x == 0 || wait_bar(&m->kempty[g], (x - 1) & 1, m);
      live = live && wait_bar(&m->rawfull[g][slot], (q / kRingSlots) & 1, m);
      if (!live) record_abort(m, p.status);
      live = live && !aborted(m);
      // Dequantise chunk c (rows 32c + cr) into the stage.
      if (live) {
      const uint8_t* rrow = ring + slot * F::CHUNK + cr * F::STRIDE;
      const int row = c * kChunkRows + cr;
      const uint2 codes = *reinterpret_cast<const uint2*>(rrow + F::NP * 16);
      constexpr int PN = F::NN / 4;  // NoPE pieces per thread: 4 or 3
      uint4 v[PN];
#pragma unroll
      for (int i = 0; i < PN; ++i) v[i] = *reinterpret_cast<const uint4*>(rrow + (cs * PN + i) * 16);
      uint4 rp[2];
      if (F::NR > 0) {
#pragma unroll
        for (int i = 0; i < 2; ++i) rp[i] = *reinterpret_cast<const uint4*>(rrow + (F::NN + cs * 2 + i) * 16);
      }
#pragma unroll
      for (int i = 0; i < PN; ++i) {
        const int k = cs * PN + i;
        const int ci = F::CODE0 + (k >> 2);
        const uint32_t code = ((ci < 4 ? codes.x : codes.y) >> (8 * (ci & 3))) & 0xFFu;
        uint4 lo, hi;
        dequant16_fast(v[i], code, lo, hi);
        *reinterpret_cast<uint4*>(stage + stage_off(row, k * 16)) = lo;
        *reinterpret_cast<uint4*>(stage + stage_off(row, k * 16 + 8)) = hi;
      }
      if (F::NR > 0) {
#pragma unroll
        for (int i = 0; i < 2; ++i)
          *reinterpret_cast<uint4*>(stage + stage_off(row, 192 + (cs * 2 + i) * 8)) = scrub_bf16x8(rp[i]);
      }
      if (gt == 0) m->mask[g][c] = m->maskring[g][slot];
      }
      named_bar_sync(bar_id, kGroupThreads);  // every thread is done with raw slot `slot`
      if (c == 1) {
        // The issues of this tile's chunks are all done: gbuf takes the next tile's slots.
        m->gbuf[g][gt] = gpre;
        skip2(pre);
        gpre = load_gidx(pre);
        named_bar_sync(bar_id, kGroupThreads);
      }
      if (iss.valid()) issue();
    }
    fence_async_smem();
    mbar_arrive(&m->kfull[g]);
    skip2(conv);
  }
  asm volatile("cp.async.wait_all;" ::: "memory");  // no copy may land after the CTA is gone
}

}  // namespace

template <bool ALIGN16>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1) attn_pair_kernel(AttnParams p) {
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
      mbar_init(&m->kfull[s], kGroupThreads);
      mbar_init(&m->kempty[s], 1);
      for (int r = 0; r < kRingSlots; ++r) mbar_init(&m->rawfull[s][r], kGroupThreads);
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
    const bool issuer = tid == 0;
    constexpr uint32_t kIdescQK = idesc_bf16_f32(128, kTile, false, false);
    constexpr uint32_t kIdescPV = idesc_bf16_f32(128, kDHalf, false, true);
    const uint32_t a_stage = smem_u32(smem);
    const uint32_t a_p = smem_u32(sP);
    // Exchange regions and the peer's barriers are recomputed at each use (kernel
    // parameters live in the constant bank), which keeps them out of the register budget.
    auto xregion = [&](uint32_t rank) { return p.xchg + ((size_t)cid * 2 + rank) * kXchgRegion; };
    const float sl2 = p.scale * kLog2e;
    bool ok = true;
    uint32_t sgrp_phase = 0;
    int j = 0;       // tile sequence number (runs on across items)
    int it_no = 0;   // items taken by this pair so far

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

    for (int w = cid; w < items && ok; w += p.G, ++it_no) {
      const Item item = item_of(p, w);
      const int n = item.n;
      {  // this thread's half of head h's Q half -> TMEM columns [64 hc, 64 hc + 64) of lane h
        const uint8_t* qrow = static_cast<const uint8_t*>(p.q) + ((int64_t)item.t * p.H + h) * (kLatent * 2) +
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
        ok = wait_bar_warp(&m->sgrp, sgrp_phase, m);
        sgrp_phase ^= 1u;
        tc_fence_after();
      }
      if (ok && issuer && n > 0) {
        if ((ok = wait_bar(&m->kfull[j & 1], (j >> 1) & 1, m))) {
          tc_fence_after();
          issue_qk(j);
        } else {
          record_abort(m, p.status);
        }
      }
      ok = __all_sync(0xffffffffu, ok);

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
        // loaded S and the next stage is filled.  The issuer only probes here and at
        // the later checkpoints, so its own exchange traffic never waits on producers.
        tc_fence_before();
        mbar_arrive(&m->sfree);
        bool qk_pending = issuer && k + 1 < n;
        auto try_qk_next = [&]() {
          if (qk_pending && mbar_test_wait(&m->sfree, j & 1) &&
              mbar_test_wait(&m->kfull[(j + 1) & 1], ((j + 1) >> 1) & 1)) {
            tc_fence_after();
            issue_qk(j + 1);
            qk_pending = false;
          }
        };
        try_qk_next();
        __syncwarp();

        // Send this thread's 64 partials (log2 units) to the peer.
        float amax = 0.f;
#pragma unroll
        for (int c = 0; c < 64; ++c) amax = fmaxf(amax, fabsf(x[c]));
        const bool fixed = amax <= kFixedMax;  // false for NaN too: those go as fp32
        if (j > 0 && !(ok = wait_bar_warp(&m->xempty, (j - 1) & 1, m, true))) break;
        uint8_t* xpeer = xregion(peer);
        uint8_t* dst = xpeer + tid * 16;
        if (fixed) {
          const float enc = amax > 0.f ? kQMax / amax : 0.f;
#pragma unroll
          for (int i = 0; i < 8; ++i)
            st_global_v4(dst + i * (kSoftmaxThreads * 16), pack_q16(x[8 * i], x[8 * i + 1], enc),
                         pack_q16(x[8 * i + 2], x[8 * i + 3], enc), pack_q16(x[8 * i + 4], x[8 * i + 5], enc),
                         pack_q16(x[8 * i + 6], x[8 * i + 7], enc));
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i)
            st_global_v4(dst + i * (kSoftmaxThreads * 16), __float_as_uint(x[4 * i]), __float_as_uint(x[4 * i + 1]),
                         __float_as_uint(x[4 * i + 2]), __float_as_uint(x[4 * i + 3]));
        }
        reinterpret_cast<float*>(xpeer + kXchgData)[tid] = fixed ? amax / kQMax : -1.f;
        mbar_arrive_cluster(mapa(smem_u32(&m->xfull), peer));
        try_qk_next();
        __syncwarp();

        // Receive the peer's partials.  This thread's 128-byte slice of the P buffer is
        // free once PV of the previous tile is done, until it takes this tile's P: the
        // slice stages the peer's int16 partials (cp.async from L2), so the exchange buffer
        // is released at once and the decode holds one piece in registers at a time.
        if (j > 0 && !(ok = wait_bar_warp(&m->pvdone, (j - 1) & 1, m))) break;
        tc_fence_after();
        if (!(ok = wait_bar_warp(&m->xfull, j & 1, m, true))) break;
        {
          const uint8_t* xown = xregion(half);
          const uint8_t* src = xown + tid * 16;
          uint8_t* slice = sP + hc * kSlab;
#pragma unroll
          for (int i = 0; i < 8; ++i) cp_async16(smem_u32(slice + sw128_off(h, i)), src + i * (kSoftmaxThreads * 16));
          const float dec = ld_global_cg_f32(xown + kXchgData + tid * 4);
          asm volatile("cp.async.wait_all;" ::: "memory");
          if (dec >= 0.f) {
            mbar_arrive_cluster(mapa(smem_u32(&m->xempty), peer));
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
            // fp32 partials (a block beyond the fixed-point range): the staged first half
            // holds columns 0..31; the slice then stages columns 32..63.
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const uint4 v = *reinterpret_cast<const uint4*>(slice + sw128_off(h, i));
              x[4 * i] += __uint_as_float(v.x);
              x[4 * i + 1] += __uint_as_float(v.y);
              x[4 * i + 2] += __uint_as_float(v.z);
              x[4 * i + 3] += __uint_as_float(v.w);
            }
#pragma unroll
            for (int i = 0; i < 8; ++i)
              cp_async16(smem_u32(slice + sw128_off(h, i)), src + (8 + i) * (kSoftmaxThreads * 16));
            asm volatile("cp.async.wait_all;" ::: "memory");
            mbar_arrive_cluster(mapa(smem_u32(&m->xempty), peer));
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const uint4 v = *reinterpret_cast<const uint4*>(slice + sw128_off(h, i));
              x[32 + 4 * i] += __uint_as_float(v.x);
              x[32 + 4 * i + 1] += __uint_as_float(v.y);
              x[32 + 4 * i + 2] += __uint_as_float(v.z);
              x[32 + 4 * i + 3] += __uint_as_float(v.w);
            }
          }
        }
        try_qk_next();
        __syncwarp();

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
        if (issuer) {
          try_qk_next();
          if ((ok = wait_bar(&m->pfull, j & 1, m))) {
            tc_fence_after();
            issue_pv(j, k == 0);
            if (k + 1 == n) umma_commit(&m->odone);
          }
          // PV of this tile frees its stage for the producers first; then QK of the next
          // tile, if it is still pending, waits for its stage here.
          if (ok && qk_pending) {
            if ((ok = wait_bar(&m->sfree, j & 1, m)) &&
                (ok = wait_bar(&m->kfull[(j + 1) & 1], ((j + 1) >> 1) & 1, m))) {
              tc_fence_after();
              issue_qk(j + 1);
              qk_pending = false;
            }
          }
          if (!ok) record_abort(m, p.status);
        }
        ok = __all_sync(0xffffffffu, ok && !aborted(m));
      }
      if (!ok) break;
      if (issuer && n == 0) mbar_arrive(&m->odone);
      if (!(ok = wait_bar_warp(&m->odone, it_no & 1, m))) break;
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
    if (!ok) {
      record_abort(m, p.status);
      if (issuer) {
        umma_commit(&m->drain);  // let issued UMMAs land before TMEM is freed
        mbar_wait_bounded(&m->drain, 0, kWaitLimitNs);
      }
    }
  } else {
    regs_dec<kProducerRegs>();
    // ------------------------------------------------------------ gather + dequant
    const int pt = tid - kSoftmaxThreads;
    const int g = pt >> 7;
    if (half == 0)
      produce<0, ALIGN16>(smem, m, p, cid, items, g, pt & 127);
    else
      produce<1, ALIGN16>(smem, m, p, cid, items, g, pt & 127);
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
  const dim3 grid(2 * p.G, 1);
  if (align16)
    attn_pair_kernel<true><<<grid, kThreads, kSmemBytes, s>>>(p);
  else
    attn_pair_kernel<false><<<grid, kThreads, kSmemBytes, s>>>(p);
  return cudaGetLastError();
}

}  // namespace smd
