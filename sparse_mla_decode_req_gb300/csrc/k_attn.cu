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
// GB300 mapping.  A work item is (token, split, group of 64 heads); one CTA owns it alone
// (no cluster, no exchange between CTAs), so 128 heads take two CTAs that gather the same
// rows (the second read is an L2 hit when both run at once, which the item order arranges).
//   QK:  S = Q K^T, UMMA M = 64 heads, N = 64 rows, K = 512 (A = Q and B = the bf16 tile,
//        both K-major 128B-swizzled shared memory).  S lands in TMEM lanes 0-15 of each
//        32-lane quarter (the M = 64 accumulator layout), 64 columns.
//   PV:  O^T = V^T P^T, four UMMAs of M = 128 latent dims, N = 64 heads, K = 64 rows: A is
//        the same bf16 tile read MN-major, B is P^T (bf16, K-major).  O^T takes 4 x 64
//        TMEM columns, lane = latent dim, column = head.  Holding O transposed is what lets
//        a 64-head x 512-dim fp32 accumulator (128 KB) share one SM's TMEM with the S
//        buffers; the M = 128 PV runs at full tensor rate.
// TMEM: O^T in columns [0, 256), two S buffers at [256, 320) and [320, 384).
// SMEM: Q [64 heads x 512] (64 KB, loaded by TMA), two stages [64 rows x 512] bf16
// (64 KB each), two P^T buffers (8 KB each).
//
// The launch is persistent: G = min(items, SMs) CTAs, CTA c taking items c, c + G, ...;
// the tile sequence (and every barrier phase) runs on across items, so the converters
// prefetch the next item's rows while the current one finishes.
//
// Roles (512 threads, four warpgroups):
//   warps 0-3, softmax + epilogue: thread (n, half) owns head n (TMEM lane 32(n/16) +
//     n%16) and 32 of the tile's 64 score columns; it writes the head's P^T row, and the
//     warp rescales O^T (its 32 latent-dim lanes, all heads) when a head's running max
//     moved, and writes the output rows.
//   warps 4 and 5: issue the QK UMMAs and Q loads, and the PV UMMAs (converged warps,
//     one elected lane issuing); warps 6 and 7 idle.
//   warps 8-15, the converters, two groups of four taking alternate tiles: each warp owns
//     16 rows of its group's tiles; it loads them straight from the cache (a tile ahead),
//     dequantises and scrubs them and writes them into the tile's 128B-swizzled stage.
//
// Every wait is bounded (AttnParams::wait_limit_ns); a wait that gives up records bit 0 in
// the status word and the CTA winds down (draining its UMMAs and Q loads, freeing TMEM).
// The kernel is launched as a programmatic dependent of the previous kernel in the stream
// and waits for it after its own set-up, before any global access.
#include <cuda.h>

#include "smd_device.cuh"
#include "smd_internal.h"

namespace smd {
namespace {

constexpr int kTile = 64;                       // gathered rows per tile
constexpr int kHeads = 64;                      // heads per CTA
constexpr int kStages = 2;
constexpr int kSoftmaxWarps = 4;                // warpgroup 0: warps 0-3
constexpr int kQkWarp = 4;                      // warpgroup 1: warps 4-7 (6 and 7 idle)
constexpr int kPvWarp = 5;
constexpr int kConvWarp0 = 8;
constexpr int kConvWarps = 8;                   // warpgroups 2-3: warps 8-15, two groups of four
constexpr int kThreads = (kConvWarp0 + kConvWarps) * 32;
// Register split (per thread): the launch gives 128 (512 x 128 = the whole file); the
// issue warpgroup (fully unrolled descriptor arithmetic) drops to 96 and the converter
// warpgroups, which hold two tiles of gathered rows in flight, rise to 136
// (128 x 128 + 128 x 96 + 256 x 136 <= 65536); nothing spills at this split.
constexpr uint32_t kIssueRegs = 96, kConvRegs = 136;
static_assert(128 * 128 + 128 * kIssueRegs + 256 * kConvRegs <= 65536, "register split");
constexpr uint32_t kSlab = kTile * 128;         // [64 rows x 64 dims] bf16, 128B-swizzled
constexpr uint32_t kStageBytes = 8 * kSlab;     // [64 rows x 512 dims]
constexpr uint32_t kQBytes = 8 * kSlab;         // [64 heads x 512 dims]
constexpr uint32_t kPBytes = kSlab;             // P^T [64 heads x 64 rows]
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffStage = kOffQ + kQBytes;
constexpr uint32_t kOffP = kOffStage + kStages * kStageBytes;
constexpr uint32_t kOffEpi = kOffP + 2 * kPBytes;    // output staging: 4 KB per softmax warp
constexpr uint32_t kEpiWarpBytes = 4096;
constexpr uint32_t kOffMisc = kOffEpi + 4 * kEpiWarpBytes;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0;
constexpr uint32_t kColS = 256;
constexpr uint64_t kDrainLimitNs = 2000000000ull;  // waits for work already in flight
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: weights stay <= 2^8 between rescales

struct Misc {
  uint64_t kfull[kStages];   // converters (one arrival per warp) -> MMA, softmax: stage filled
  uint64_t kempty[kStages];  // PV commit -> converters: stage consumed
  uint64_t sfull[2];         // QK commit -> softmax: S buffer filled
  uint64_t sfree[2];         // softmax (4 warps) -> MMA: S buffer in registers
  uint64_t pfull[2];         // softmax (4 warps) -> MMA: P^T written, O^T rescaled
  uint64_t pvdone[2];        // PV commit -> softmax: P^T buffer read, O^T updated
  uint64_t rdv;              // softmax rendezvous of a tile's rescale decision (4 warps)
  uint64_t erdv;             // softmax rendezvous of an item's output factors (4 warps)
  uint64_t qfull;            // Q of an item landed (TMA transaction bytes)
  uint64_t qfree;            // QK of an item's last tile done: the Q buffer may be reloaded
  uint64_t odone;            // last PV of an item done: O^T final
  uint64_t ofree;            // epilogue (4 warps) read O^T: the next item may overwrite it
  uint64_t drain[2];         // each issuer's own UMMAs, before TMEM is freed
  uint32_t tmem_base;
  uint32_t abort;
  uint32_t rescale_seq[2];   // tile j + 1 when tile j needs an O^T rescale
  alignas(16) float mask[kStages][kTile];  // per row of each stage: 0 (valid) or -inf (read as 16-byte vectors)
  alignas(16) float alpha[2][kHeads];   // per-head rescale factor of a tile (read as 16-byte vectors)
  alignas(16) float factor[2][kHeads];  // per-head output factor of an item (read as 16-byte vectors)
};
static_assert(offsetof(Misc, mask) % 16 == 0, "mask[] is read with 16-byte loads");
constexpr uint32_t kSmemBytes = kOffMisc + sizeof(Misc);
constexpr uint32_t kSmemLaunch = kSmemBytes + 1024;  // slack for aligning the base to 1 KB
static_assert(kSmemLaunch <= 232448, "shared memory budget");

__device__ __forceinline__ bool aborted(const Misc* m) {
  return *reinterpret_cast<const volatile uint32_t*>(&m->abort) != 0u;
}
__device__ __forceinline__ void record_abort(Misc* m, uint32_t* status) {
  atomicExch(&m->abort, 1u);
  if (status != nullptr) atomicOr(status, kStatusTimeout);
}

// One probe of a phase: the suspending try_wait normally; a non-blocking test when the
// bound is shorter than try_wait's suspend time (a bound that short is only set to make
// the waits give up, and a suspending probe could outlast it by finding the phase done).
__device__ __forceinline__ bool probe(uint64_t* bar, uint32_t parity, uint64_t limit) {
  return limit < kSuspendHintNs ? mbar_test(bar, parity) : mbar_try_wait(bar, parity);
}
// Bounded wait that also gives up once another role of this CTA has aborted.
__device__ __forceinline__ bool wait_slow(uint64_t* bar, uint32_t parity, const Misc* m, uint64_t limit) {
  const uint64_t t0 = globaltimer_ns();
  while (!probe(bar, parity, limit)) {
    if (aborted(m) || globaltimer_ns() - t0 > limit) return false;
  }
  return true;
}
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, const Misc* m, uint64_t limit) {
  if (probe(bar, parity, limit)) return true;
  return wait_slow(bar, parity, m, limit);
}
// The same wait done by a whole warp, with a warp-uniform result, so that a warp never
// splits into lanes that go on and lanes that leave (which would strand the first at the
// next warp-collective instruction).
__device__ __forceinline__ bool wait_warp(uint64_t* bar, uint32_t parity, const Misc* m, uint64_t limit) {
  return __all_sync(0xffffffffu, wait_bar(bar, parity, m, limit));
}
// One arrival per warp, after the warp's lanes converge (which orders their earlier
// memory accesses before lane 0's release).
__device__ __forceinline__ void warp_arrive(uint64_t* bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

// One work item: (token t, split, head group g); tiles [tile_begin, tile_begin + n) of the
// token's entries (n = 0 for a split past the end).  The token attends to its first ntot
// converted entries, the first kmain of them in the main cache and the rest in the window
// cache (the call's K and N, or the per-token counts of a compacted conversion).
struct Item {
  int t, split, g, tile_begin, n, kmain, ntot;
};
__device__ __forceinline__ Item item_of(const AttnParams& p, int w) {
  Item it;
  const int ts = w / p.HG;  // head group fastest: a token's groups run side by side
  it.g = w - ts * p.HG;
  it.t = ts / p.S;
  it.split = ts - it.t * p.S;
  it.tile_begin = it.split * p.tiles_per_split;
  it.kmain = p.K;
  it.ntot = p.N;
  if (p.counts != nullptr) {
    it.ntot = min(max(__ldg(p.counts + 2 * it.t + 1), 0), p.N);
    it.kmain = min(max(__ldg(p.counts + 2 * it.t), 0), it.ntot);
  }
  const int ntok = (it.ntot + kTile - 1) / kTile;
  it.n = max(0, min(ntok, it.tile_begin + p.tiles_per_split) - it.tile_begin);
  return it;
}

__device__ __forceinline__ int num_items(const AttnParams& p) { return p.T * p.S * p.HG; }

// Walks the tiles of the items w0, w0 + G, ... in order, skipping items without tiles.
struct TileCursor {
  int w, k;
  Item it;
  __device__ void settle(const AttnParams& p) {
    const int items = num_items(p);
    while (w < items) {
      it = item_of(p, w);
      if (k < it.n) return;
      w += p.G;
      k = 0;
    }
  }
  __device__ void init(const AttnParams& p, int w0) {
    w = w0;
    k = 0;
    settle(p);
  }
  __device__ bool valid(const AttnParams& p) const { return w < num_items(p); }
  __device__ bool first() const { return k == 0; }
  __device__ bool last() const { return k == it.n - 1; }
  __device__ int64_t row0(const AttnParams& p) const { return (int64_t)it.t * p.N + (int64_t)(it.tile_begin + k) * kTile; }
  __device__ int rows(const AttnParams& p) const { return min(kTile, it.ntot - (it.tile_begin + k) * kTile); }
  // first entry index of the tile within the token's list
  __device__ int entry0() const { return (it.tile_begin + k) * kTile; }
  __device__ void next(const AttnParams& p) {
    ++k;
    settle(p);
  }
  __device__ void next_item(const AttnParams& p) {
    k = it.n;
    settle(p);
  }
};

// ------------------------------------------------------------------ UMMA issuers
// Two warps issue every UMMA of the CTA, each after blocking waits for its inputs (a PV,
// which waits for the softmax, never queues behind a QK, which waits for the converters,
// which in turn wait for PV to free a stage).  Each warp runs its issue loop converged
// and unrolled, one elected lane issuing:
//   QK warp (4):  QK(j) once stage j is converted, S buffer j&1 was read (tile j-2) and
//     the item's Q landed; its commit fills S buffer j&1.  After an item's last QK it
//     waits for that QK to complete (the Q buffer is then free) and loads the next item's
//     Q with TMA (prefetched into L2 when the item started).
//   PV warp (5):  PV(j) once P^T(j) is written (and, for an item's first tile, once the
//     previous item's epilogue has read O^T); its commit frees stage j and P^T buffer
//     j&1, and the item's last PV signals O^T final.
__device__ void qk_warp(uint8_t* smem, Misc* m, const AttnParams& p, const CUtensorMap* qmap, int cid,
                        uint32_t tmem, int lane) {
  constexpr uint32_t kIdQK = idesc_bf16_f32(64, kTile, false, false);
  const uint32_t sQ = smem_u32(smem + kOffQ);
  const uint64_t dQ = desc_sw128(sQ, 16, 1024);                          // A: Q, K-major
  const uint64_t dK = desc_sw128(smem_u32(smem + kOffStage), 16, 1024);  // B: the tile, K-major
  const uint64_t limit = p.wait_limit_ns;
  TileCursor qc;
  qc.init(p, cid);
  auto q_row = [&](const TileCursor& c) { return c.it.t * p.H + c.it.g * kHeads; };
  auto load_q = [&](const TileCursor& c) {
    if (lane == 0) {
      mbar_arrive_expect_tx(&m->qfull, kQBytes);
#pragma unroll
      for (int s = 0; s < 8; ++s) tma_load_2d(sQ + s * kSlab, qmap, s * 64, q_row(c), &m->qfull);
    }
    __syncwarp();
  };
  int nq = 0;   // Q loads issued (= items started)
  bool ok = true;
  if (qc.valid(p)) {
    load_q(qc);
    ++nq;
  }
  for (int j = 0; qc.valid(p) && ok; ++j) {
    if (qc.first()) {
      ok = wait_warp(&m->qfull, (nq - 1) & 1, m, limit);
      TileCursor nx = qc;  // the next item's Q into L2
      nx.next_item(p);
      if (ok && nx.valid(p) && lane < 8) tma_prefetch_2d(qmap, lane * 64, q_row(nx));
    }
    ok = ok && wait_warp(&m->kfull[j & 1], (j >> 1) & 1, m, limit);
    ok = ok && (j < 2 || wait_warp(&m->sfree[j & 1], ((j >> 1) - 1) & 1, m, limit));
    if (!ok) break;
    tc_fence_after();
    const uint32_t d = tmem + kColS + (j & 1) * kTile;
    const uint64_t b = dK + (uint64_t)(((j & 1) * kStageBytes) >> 4);
#pragma unroll
    for (int kk = 0; kk < kLatent / 16; ++kk) {
      constexpr uint32_t kSlab16 = kSlab >> 4;
      const uint64_t off = (uint64_t)((kk >> 2) * kSlab16 + (kk & 3) * 2);
      umma_ss_elect(d, dQ + off, b + off, kIdQK, kk > 0 ? 1u : 0u);
    }
    umma_commit_elect(&m->sfull[j & 1]);
    const bool last = qc.last();
    qc.next(p);
    if (last && qc.valid(p)) {  // the next item's Q, once this item's QKs have read Q
      umma_commit_elect(&m->qfree);
      ok = wait_warp(&m->qfree, (nq - 1) & 1, m, limit);
      if (!ok) break;
      load_q(qc);
      ++nq;
    }
  }
  if (!ok && lane == 0) record_abort(m, p.status);
  // Every UMMA issued lands before TMEM is freed, and the last Q load before the shared
  // memory is released.
  umma_commit_elect(&m->drain[0]);
  if (lane == 0) {
    (void)mbar_wait_bounded(&m->drain[0], 0, kDrainLimitNs);
    if (nq > 0) (void)mbar_wait_bounded(&m->qfull, (nq - 1) & 1, kDrainLimitNs);
  }
  __syncwarp();
}

__device__ void pv_warp(uint8_t* smem, Misc* m, const AttnParams& p, int cid, uint32_t tmem, int lane) {
  constexpr uint32_t kIdPV = idesc_bf16_f32(128, kHeads, true, false);
  const uint64_t dV = desc_sw128(smem_u32(smem + kOffStage), kSlab, 1024);  // A: the tile read MN-major
  const uint64_t dP = desc_sw128(smem_u32(smem + kOffP), 16, 1024);         // B: P^T, K-major
  const uint64_t limit = p.wait_limit_ns;
  TileCursor pc;
  pc.init(p, cid);
  int ip = 0;  // items whose PVs were all issued
  bool ok = true;
  for (int j = 0; pc.valid(p) && ok; ++j) {
    const bool first = pc.first();
    ok = !first || ip == 0 || wait_warp(&m->ofree, (ip - 1) & 1, m, limit);
    ok = ok && wait_warp(&m->pfull[j & 1], (j >> 1) & 1, m, limit);
    if (!ok) break;
    tc_fence_after();
    const uint64_t a = dV + (uint64_t)(((j & 1) * kStageBytes) >> 4);
    const uint64_t b = dP + (uint64_t)(((j & 1) * kPBytes) >> 4);
    const uint32_t acc0 = first ? 0u : 1u;
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
      for (int kk = 0; kk < kTile / 16; ++kk)
        umma_ss_elect(tmem + kColO + c * kHeads, a + (uint64_t)((c * 2 * kSlab + kk * 2048) >> 4),
                      b + (uint64_t)((kk * 32) >> 4), kIdPV, kk > 0 ? 1u : acc0);
    umma_commit_elect(&m->kempty[j & 1]);
    umma_commit_elect(&m->pvdone[j & 1]);
    if (pc.last()) {
      umma_commit_elect(&m->odone);
      ++ip;
    }
    pc.next(p);
  }
  if (!ok && lane == 0) record_abort(m, p.status);
  umma_commit_elect(&m->drain[1]);
  if (lane == 0) (void)mbar_wait_bounded(&m->drain[1], 0, kDrainLimitNs);
  __syncwarp();
}

// ------------------------------------------------------------------ converters
// All eight converter warps take every tile: warp cw owns rows 8cw .. 8cw+7, lanes
// 4q..4q+3 row 8cw + q, moved in 9 steps of one 64-byte segment (lane m taking bytes
// 16m .. 16m+15 of it): steps 0-6 the NoPE segments (step st = dims 64st..64st+63, all
// under scale code st), steps 7-8 the two RoPE halves.  At each step a group of four lanes
// reads 64 contiguous bytes (whole sectors; a row is fetched by one warp within a few
// instructions, which keeps DRAM pages open: a layout that spread each row over nine warps
// gathered at half the rate).  Each lane reads its row's slot and scale row itself.  The
// eight rows of one store instruction hit eight different 16-byte bank groups of the
// 128B-swizzled stage (row r's chunks are XORed with r & 7).
//
// Every warp keeps two tiles of gathered rows in registers (buffers A and B, for the even
// and the odd tiles): right after converting a tile into its stage it issues the gathers
// of the tile two ahead into the same registers, so each warp has one tile of gathers in
// flight while it converts the other, and a tile's conversion is spread over all warps.
constexpr int kRowsPerConvWarp = kTile / kConvWarps;  // 8
static_assert(kRowsPerConvWarp == 8, "one 8-row set per converter warp");

// A row's converted slot and the scope (cache) it lives in.
struct SlotRef {
  int32_t g;      // -1: masked or past the end
  int32_t scope;  // 0: main cache, 1: window cache
};
__device__ __forceinline__ CacheDesc scope_cache(const AttnParams& p, int32_t scope) {
  CacheDesc c;
  c.base = scope ? p.cache2.base : p.cache.base;
  c.num_pages = scope ? p.cache2.num_pages : p.cache.num_pages;
  c.P = scope ? p.cache2.P : p.cache.P;
  c.log2P = scope ? p.cache2.log2P : p.cache.log2P;
  return c;
}
// Issues the read of the slot of entry row `r` of tile `c` (the value is validated where
// it is used, so the read stays in flight meanwhile).
__device__ __forceinline__ SlotRef read_slot(const AttnParams& p, const TileCursor& c, bool v, int r) {
  SlotRef s{-1, 0};
  if (v && r < c.rows(p) && in_range(c.row0(p) + r < (int64_t)p.T * p.N, p.status)) {
    s.g = ldg_nc_s32(p.gidx + c.row0(p) + r);
    s.scope = c.entry0() + r >= c.it.kmain ? 1 : 0;
  }
  return s;
}

template <bool ALIGN16>
struct Converter {
  int q, m, row;  // q = lane / 4: the lane's row in the warp's 8; m = lane % 4: its piece; row: in the tile
  __device__ Converter(int lane, int cw) : q(lane >> 2), m(lane & 3), row(kRowsPerConvWarp * cw + (lane >> 2)) {}
  struct Raw {
    uint4 v[9];          // v[st]: bytes 64 st + 16 m .. +15 of the lane's row
    uint2 sc;            // its scale row
    const uint8_t* rp;   // its data
    bool ok;             // the row is valid
  };
  __device__ SlotRef slot(const AttnParams& p, const TileCursor& c, bool v) const { return read_slot(p, c, v, row); }
  __device__ void load(const AttnParams& p, SlotRef sl, Raw& d) const {
    const CacheDesc cd = scope_cache(p, sl.scope);
    d.ok = false;
    d.sc = make_uint2(0, 0);
    d.rp = cd.base;
    if (sl.g >= 0 && (int64_t)sl.g < cd.num_pages * cd.P) {
      const CacheView cv = make_cache_view(cd.base, cd.P, cd.log2P);
      int32_t page, o;
      slot_page_off(cv, sl.g, page, o);
      if (in_range(page >= 0 && page < cd.num_pages && o >= 0 && o < cd.P, p.status)) {
        const uint8_t* pg = cv.base + (int64_t)page * cv.page_bytes;
        d.rp = pg + (int64_t)o * kDataBytes;
        d.sc = ldg_nc_v2(pg + cv.scale_start + (int64_t)o * kScaleBytes);
        d.ok = true;
      }
    }
#pragma unroll
    for (int st = 0; st < 9; ++st) {
      d.v[st] = make_uint4(0, 0, 0, 0);
      if (d.ok) d.v[st] = ldg16<ALIGN16>(d.rp + st * 64 + m * 16);
    }
  }
  // Straight-line conversion of every piece on the fast path (no NaN byte, code <= 134);
  // the rare pieces outside that case are read again (an L1/L2 hit) and redone on the
  // exact path afterwards, overwriting their fast result.
  __device__ void store(uint8_t* stage, const Raw& d) const {
    uint32_t redo = 0;
    uint8_t* rrow = stage + row * 128;
#pragma unroll
    for (int st = 0; st < 7; ++st) {  // NoPE: slab st, chunks 2m and 2m + 1
      const uint32_t code = ((st < 4 ? d.sc.x : d.sc.y) >> (8 * (st & 3))) & 0xFFu;
      uint8_t* rb = rrow + st * kSlab;
      uint4 lo, hi;
      dequant_fast(d.v[st], code, lo, hi);
      redo |= needs_exact(d.v[st], code) ? 1u << st : 0u;
      *reinterpret_cast<uint4*>(rb + (((2 * m) ^ q) << 4)) = lo;
      *reinterpret_cast<uint4*>(rb + (((2 * m + 1) ^ q) << 4)) = hi;
    }
#pragma unroll
    for (int st = 7; st < 9; ++st)  // RoPE: slab 7, chunk 4(st - 7) + m
      *reinterpret_cast<uint4*>(rrow + 7 * kSlab + (((4 * (st - 7) + m) ^ q) << 4)) = scrub_bf16x8(d.v[st]);
    if (__any_sync(0xffffffffu, redo != 0u)) {  // rare: NaN bytes or codes above 134
#pragma unroll 1
      for (int st = 0; st < 7; ++st) {
        if ((redo >> st) & 1u) {
          const uint4 raw = ldg16<ALIGN16>(d.rp + st * 64 + m * 16);
          const uint32_t code = ((st < 4 ? d.sc.x : d.sc.y) >> (8 * (st & 3))) & 0xFFu;
          uint4 lo, hi;
          dequant_piece(raw, code, lo, hi);
          uint8_t* rb = rrow + st * kSlab;
          *reinterpret_cast<uint4*>(rb + (((2 * m) ^ q) << 4)) = lo;
          *reinterpret_cast<uint4*>(rb + (((2 * m + 1) ^ q) << 4)) = hi;
        }
      }
    }
  }
};

template <bool ALIGN16>
__device__ void converter_warps(uint8_t* smem, Misc* m, const AttnParams& p, int cid, int cw, int lane) {
  using Cv = Converter<ALIGN16>;
  const Cv cv(lane, cw);
  const uint64_t limit = p.wait_limit_ns;
  typename Cv::Raw a, b;  // even and odd tiles
  TileCursor c;           // the tile whose slot is read next
  c.init(p, cid);
  auto take = [&](bool& v, SlotRef& sl) {  // slot of the cursor's tile, then advance
    v = c.valid(p);
    sl = cv.slot(p, c, v);
    if (v) c.next(p);
  };
  bool va, vb, va2, vb2;
  SlotRef sa, sb, sa2, sb2;
  take(va, sa);    // tile 0
  take(vb, sb);    // tile 1
  take(va2, sa2);  // tile 2
  take(vb2, sb2);  // tile 3
  if (va) cv.load(p, sa, a);
  if (vb) cv.load(p, sb, b);
  // One tile into its stage: wait for the stage (PV of the tile two before it), convert,
  // publish, then gathers of the tile two ahead into the same registers and the slot read
  // of the tile after that.
  auto step = [&](typename Cv::Raw& d, int st_, int k, bool& vnext, SlotRef& snext) -> bool {
    if (k >= 1 && !wait_warp(&m->kempty[st_], (k - 1) & 1, m, limit)) {
      if (lane == 0) record_abort(m, p.status);
      return false;
    }
    cv.store(smem + kOffStage + st_ * kStageBytes, d);
    if (cv.m == 0) m->mask[st_][cv.row] = d.ok ? 0.f : -INFINITY;
    fence_async_smem();
    warp_arrive(&m->kfull[st_]);
    const bool v = vnext;
    if (v) cv.load(p, snext, d);
    take(vnext, snext);
    return v;
  };
  for (int k = 0; va; ++k) {  // tiles 2k (buffer a) and 2k + 1 (buffer b)
    const bool na = step(a, 0, k, va2, sa2);
    if (!vb) break;
    const bool nb = step(b, 1, k, vb2, sb2);
    if (aborted(m)) return;
    va = na;
    vb = nb;
  }
}

// bf16 latent rows (1024 bytes: 512 little-endian bf16, NoPE then RoPE): nothing to
// dequantise, only the non-finite elements to zero.  All eight converter warps take every
// tile, warp cw owning rows 8cw .. 8cw+7, moved in 16 steps of one 64-byte segment per
// row (step st = dims 32st .. 32st+31: slab st/2, chunks 4(st&1) .. +3), lanes 4q..4q+3
// owning row q as on the fp8 path.  A tile's rows stay in registers while the warp waits
// for their stage, so the gathers of tile j + 1 are in flight during the wait for the PV
// of tile j - 1.
constexpr int kBf16RowBytes = 1024;
__device__ void converter_warps_bf16(uint8_t* smem, Misc* m, const AttnParams& p, int cid, int cw, int lane) {
  const int q = lane >> 2, mm = lane & 3;
  const uint64_t limit = p.wait_limit_ns;
  uint4 v[16];
  bool ok = false;
  auto slot = [&](const TileCursor& c, bool valid) -> SlotRef { return read_slot(p, c, valid, 8 * cw + q); };
  auto load = [&](SlotRef sl) {
    const CacheDesc cd = scope_cache(p, sl.scope);
    ok = sl.g >= 0 && (int64_t)sl.g < cd.num_pages * cd.P &&
         in_range(((int64_t)sl.g + 1) * kBf16RowBytes <= cd.num_pages * cd.P * kBf16RowBytes, p.status);
    // pages hold P rows of 1024 bytes back to back, so slot g sits at byte 1024 g
    const uint8_t* r = cd.base + (ok ? (int64_t)sl.g * kBf16RowBytes : 0);
#pragma unroll
    for (int st = 0; st < 16; ++st) {
      v[st] = make_uint4(0, 0, 0, 0);
      if (ok) v[st] = ldg_nc_v4(r + st * 64 + mm * 16);
    }
  };
  TileCursor c;
  c.init(p, cid);
  bool v0 = c.valid(p);
  SlotRef s0 = slot(c, v0);
  if (v0) c.next(p);
  bool v1 = c.valid(p);
  SlotRef s1 = slot(c, v1);
  if (v1) c.next(p);
  load(s0);
  for (int j = 0; v0; ++j) {
    const int st_ = j & 1;
    if (j >= kStages && !wait_warp(&m->kempty[st_], ((j >> 1) - 1) & 1, m, limit)) {
      if (lane == 0) record_abort(m, p.status);
      return;
    }
    uint8_t* rrow = smem + kOffStage + st_ * kStageBytes + (8 * cw + q) * 128;
#pragma unroll
    for (int st = 0; st < 16; ++st)
      *reinterpret_cast<uint4*>(rrow + (st >> 1) * kSlab + (((4 * (st & 1) + mm) ^ q) << 4)) = scrub_bf16x8(v[st]);
    if (mm == 0) m->mask[st_][8 * cw + q] = ok ? 0.f : -INFINITY;
    fence_async_smem();
    warp_arrive(&m->kfull[st_]);
    v0 = v1;
    s0 = s1;
    if (v0) load(s0);  // gathers before the next slot reads, as on the fp8 path
    v1 = c.valid(p);
    s1 = slot(c, v1);
    if (v1) c.next(p);
  }
}

// ------------------------------------------------------------------ softmax + epilogue
__device__ void softmax_warps(uint8_t* smem, Misc* m, const AttnParams& p, const CUtensorMap* omap, int cid,
                              uint32_t tmem, int warp, int lane) {
  const int n = 16 * warp + (lane & 15);  // head within the group (TMEM lane 32 warp + lane % 16)
  const int half = lane >> 4;             // score columns [32 half, 32 half + 32)
  const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
  const float sl2 = p.scale * kLog2e;
  const uint64_t limit = p.wait_limit_ns;
  const int items = num_items(p);
  bool ok = true;
  int j = 0;          // tile sequence number
  int nitem = 0;      // items with tiles done
  int nrdv = 0, nerdv = 0;
  for (int w = cid; w < items && ok; w += p.G) {
    const Item it = item_of(p, w);
    const int h = it.g * kHeads + n;
    const bool head_ok = h < p.H;
    const float sink_nat = (p.S == 1 && p.sink != nullptr && head_ok) ? __ldg(p.sink + h) : -INFINITY;
    const int64_t orow = p.S == 1 ? (int64_t)it.t * p.H + h : ((int64_t)it.t * p.S + it.split) * p.H + h;
    if (it.n == 0) {  // no entries: out = 0 and lse = sink (one split), or an empty split
      if (head_ok && half == 0 && in_range(orow < (int64_t)p.T * p.S * p.H, p.status)) {
        if (p.S > 1) p.lse_part[orow] = -INFINITY;
        else if (p.lse != nullptr) p.lse[orow] = sink_nat;
      }
      if (p.S == 1) {
        const int d = 32 * warp + lane;
        for (int hh = 0; hh < kHeads && it.g * kHeads + hh < p.H; ++hh)
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int64_t off = ((int64_t)it.t * p.H + it.g * kHeads + hh) * kLatent + 128 * c + d;
            if (in_range(off < (int64_t)p.T * p.H * kLatent, p.status))
              reinterpret_cast<__nv_bfloat16*>(p.out)[off] = __float2bfloat16_rn(0.f);
          }
      }
      continue;
    }
    float m_ref = -INFINITY;  // running reference max (log2 units) the weights are taken against
    float l_run = 0.f;        // this thread's share of the denominator relative to m_ref
    for (int k = 0; k < it.n; ++k, ++j) {
      const int b = j & 1;
      if (!(ok = wait_warp(&m->sfull[b], (j >> 1) & 1, m, limit))) break;
      tc_fence_after();
      uint32_t r[32];
      tmem_ld16x2_32(tmem + lane_base + kColS + b * kTile, r);
      tmem_wait_ld();
      tc_fence_before();
      warp_arrive(&m->sfree[b]);  // QK of tile j + 2 may overwrite the buffer
      // row masks of the tile (published with the stage): 0, or -inf for an invalid row,
      // whose gathered row is zero so its score is too
      if (!(ok = wait_warp(&m->kfull[b], (j >> 1) & 1, m, limit))) break;
      float mk[32];
#pragma unroll
      for (int k4 = 0; k4 < 8; ++k4) {
        const uint4 v4 = ld_shared_v4(smem_u32(&m->mask[b][32 * half + 4 * k4]));
        mk[4 * k4] = __uint_as_float(v4.x);
        mk[4 * k4 + 1] = __uint_as_float(v4.y);
        mk[4 * k4 + 2] = __uint_as_float(v4.z);
        mk[4 * k4 + 3] = __uint_as_float(v4.w);
      }
      float x[32];
      float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};  // four chains, not one of 32
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        x[i] = fmaf(__uint_as_float(r[i]), sl2, mk[i]);
        mx[i & 3] = fmaxf(mx[i & 3], x[i]);
      }
      float tmax = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
      tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 16));
      float alpha = 1.f;
      const bool upd = tmax > m_ref + kRescaleThreshold;  // false while everything is masked
      if (upd) {
        alpha = fast_exp2(m_ref - tmax);  // 0 when m_ref is -inf
        m_ref = tmax;
      }
      float psum = 0.f;
      uint32_t pk[16];
      if (m_ref == -INFINITY) {
#pragma unroll
        for (int i = 0; i < 16; ++i) pk[i] = 0u;
      } else {
        float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float p0 = fast_exp2(x[2 * i] - m_ref), p1 = fast_exp2(x[2 * i + 1] - m_ref);
          ps[i & 3] += p0 + p1;  // the denominator keeps the unrounded weights
          pk[i] = bf16x2_bits(__floats2bfloat162_rn(p0, p1));
        }
        psum = (ps[0] + ps[1]) + (ps[2] + ps[3]);
      }
      l_run = l_run * alpha + psum;
      // P^T buffer b was last read by PV of tile j - 2
      if (j >= 2 && !(ok = wait_warp(&m->pvdone[b], ((j >> 1) - 1) & 1, m, limit))) break;
      const uint32_t pbase = smem_u32(smem + kOffP + b * kPBytes);
#pragma unroll
      for (int c = 0; c < 4; ++c)
        st_shared_v4(pbase + sw128_off(n, 4 * half + c), make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]));
      if (k > 0) {
        // O^T holds the item's PV up to tile j - 1; a head whose max moved needs its
        // column rescaled by every warp (each owns 32 latent-dim lanes of all heads).
        if (half == 0) m->alpha[b][n] = alpha;
        if (upd) m->rescale_seq[b] = (uint32_t)j + 1u;
        warp_arrive(&m->rdv);
        if (!(ok = wait_warp(&m->rdv, nrdv & 1, m, limit))) break;
        ++nrdv;
        if (*reinterpret_cast<volatile uint32_t*>(&m->rescale_seq[b]) == (uint32_t)j + 1u) {
          if (!(ok = wait_warp(&m->pvdone[b ^ 1], ((j - 1) >> 1) & 1, m, limit))) break;
          tc_fence_after();
#pragma unroll 1
          for (int cc = 0; cc < 8; ++cc) {
            uint32_t o[32];
            const uint32_t col = kColO + cc * 32;  // block cc/2, heads 32(cc&1)..+31
            tmem_ld32(tmem + lane_base + col, o);
            float al[32];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const uint4 a4 = ld_shared_v4(smem_u32(&m->alpha[b][32 * (cc & 1) + 4 * k]));
              al[4 * k] = __uint_as_float(a4.x);
              al[4 * k + 1] = __uint_as_float(a4.y);
              al[4 * k + 2] = __uint_as_float(a4.z);
              al[4 * k + 3] = __uint_as_float(a4.w);
            }
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * al[i]);
            tmem_st32(tmem + lane_base + col, o);
          }
          tmem_wait_st();
        }
      }
      fence_async_smem();
      tc_fence_before();
      warp_arrive(&m->pfull[b]);
    }
    if (!ok) break;
    // ---------------------------------------------------------------- epilogue
    const float l_tot = l_run + __shfl_xor_sync(0xffffffffu, l_run, 16);
    // One split: fold the sink into the denominator and write bf16 out + lse.  Several
    // splits: the split's normalised fp32 output and sink-free lse.
    float factor = 0.f, lse_v = -INFINITY;
    if (p.S == 1) {
      const float ms = sink_nat * kLog2e;
      const float M = fmaxf(m_ref, ms);
      if (M != -INFINITY) {
        const float den = l_tot * fast_exp2(m_ref - M) + (ms == -INFINITY ? 0.f : fast_exp2(ms - M));
        factor = fast_exp2(m_ref - M) / den;
        // natural-log max from whichever term set it, so a sink-only row gives lse = sink exactly
        lse_v = (M == m_ref ? m_ref * kLn2 : sink_nat) + log2f(den) * kLn2;
      }
    } else if (l_tot > 0.f) {
      factor = 1.f / l_tot;
      lse_v = (m_ref + log2f(l_tot)) * kLn2;
    }
    const int fb = nitem & 1;
    if (half == 0) {
      m->factor[fb][n] = factor;
      if (head_ok && in_range(orow < (int64_t)p.T * p.S * p.H, p.status)) {
        if (p.S > 1) p.lse_part[orow] = lse_v;
        else if (p.lse != nullptr) p.lse[orow] = lse_v;
      }
    }
    if (!(ok = wait_warp(&m->odone, nitem & 1, m, limit))) break;
    ++nitem;
    warp_arrive(&m->erdv);
    if (!(ok = wait_warp(&m->erdv, nerdv & 1, m, limit))) break;
    ++nerdv;
    tc_fence_after();
    // O^T (lane = latent dim, column = head) leaves by TMA stores, which take no slot in the
    // load/store pipeline that the gathers keep busy.  Per block of 128 dims the warp loads
    // its 32 dim-lanes of all 64 heads from TMEM (two loads in flight together), scales them
    // and writes them as [heads][32 dims] boxes into its two alternating 4 KB staging
    // buffers (a slice of the P^T buffers, free once O is final, and a slice of the staging
    // region): one box of 64 heads in bf16, or two of 32 heads in fp32; one lane stores each
    // box to out[t, heads, dims] (or o_part[t, split, heads, dims]), the tensor map clipping
    // heads past H.
    const int zc = p.S == 1 ? it.t : it.t * p.S + it.split;
    uint8_t* const buf0 = smem + kOffP + warp * kEpiWarpBytes;
    uint8_t* const buf1 = smem + kOffEpi + warp * kEpiWarpBytes;
    const bool odd = lane & 1;
    int nbox = 0;  // boxes committed by this warp in this item
    auto next_buffer = [&]() -> uint8_t* {  // once the store two boxes back has read it
      if (lane == 0 && nbox >= 2) bulk_wait_read<1>();
      __syncwarp();
      return (nbox & 1) ? buf1 : buf0;
    };
    auto store_box = [&](uint8_t* sb, int x, int y) {
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        // a box wholly past H is not stored, but still closes a (then empty) group, so
        // that the wait in next_buffer always counts the store of the other buffer
        if (y < p.H) tma_store_3d(omap, smem_u32(sb), x, y, zc);
        bulk_commit();
      }
      ++nbox;
    };
    // the 32 heads' factors from h0 into registers first: loads interleaved with the
    // staging stores would be kept in order behind them (they may alias) and serialise it
    auto factors = [&](int h0, float (&fac)[32]) {
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint4 f4 = ld_shared_v4(smem_u32(&m->factor[fb][h0 + 4 * k]));
        fac[4 * k] = __uint_as_float(f4.x);
        fac[4 * k + 1] = __uint_as_float(f4.y);
        fac[4 * k + 2] = __uint_as_float(f4.z);
        fac[4 * k + 3] = __uint_as_float(f4.w);
      }
    };
    // bf16 rows h0 .. h0+31 of a [64 heads][32 dims] box: lanes 2k and 2k + 1 (dims 2k,
    // 2k + 1) trade one value per pair of heads (i, i + 1), so that lane 2k stores head
    // i's bf16 pair and lane 2k + 1 head i + 1's
    auto stage_bf16 = [&](uint8_t* sb, const uint32_t (&o)[32], int h0) {
      float fac[32];
      factors(h0, fac);
#pragma unroll
      for (int i = 0; i < 32; i += 2) {
        const float v0 = __uint_as_float(o[i]) * fac[i], v1 = __uint_as_float(o[i + 1]) * fac[i + 1];
        const float keep = odd ? v1 : v0, give = odd ? v0 : v1;
        const float got = __shfl_xor_sync(0xffffffffu, give, 1);
        const uint32_t pair = bf16x2_bits(odd ? __floats2bfloat162_rn(got, keep) : __floats2bfloat162_rn(keep, got));
        *reinterpret_cast<uint32_t*>(sb + (h0 + i + (odd ? 1 : 0)) * 64 + (lane & ~1) * 2) = pair;
      }
    };
    auto stage_f32 = [&](uint8_t* sb, const uint32_t (&o)[32], int h0) {  // a [32 heads][32 dims] box
      float fac[32];
      factors(h0, fac);
#pragma unroll
      for (int i = 0; i < 32; ++i) *reinterpret_cast<float*>(sb + (i * 32 + lane) * 4) = __uint_as_float(o[i]) * fac[i];
    };
#pragma unroll 1
    for (int blk = 0; blk < 4; ++blk) {
      uint32_t oa[32], ob[32];
      tmem_ld32(tmem + lane_base + kColO + blk * kHeads, oa);       // heads 0-31
      tmem_ld32(tmem + lane_base + kColO + blk * kHeads + 32, ob);  // heads 32-63
      tmem_wait_ld();
      const int x = blk * 128 + 32 * warp, y = it.g * kHeads;
      if (p.S == 1) {
        uint8_t* sb = next_buffer();
        stage_bf16(sb, oa, 0);
        stage_bf16(sb, ob, 32);
        store_box(sb, x, y);
      } else {
        uint8_t* sb = next_buffer();
        stage_f32(sb, oa, 0);
        store_box(sb, x, y);
        sb = next_buffer();
        stage_f32(sb, ob, 32);
        store_box(sb, x, y + 32);
      }
    }
    if (lane == 0) bulk_wait_read<0>();  // the next item writes P^T into the staging
    __syncwarp();
    tc_fence_before();
    warp_arrive(&m->ofree);  // the next item's first PV may overwrite O^T
  }
  if (!ok) record_abort(m, p.status);
  if (lane == 0) bulk_wait_all();  // every output store performed before the CTA exits
  __syncwarp();
}

}  // namespace

// Kernel parameters: the call's parameters and the tensor map of q as [T*H rows, 512] bf16.
struct KernelParams {
  AttnParams p;
  CUtensorMap qmap;  // the type carries the 64-byte alignment of a tensor map
  CUtensorMap omap;  // out [T, H, 512] bf16 (one split) or o_part [T*S, H, 512] fp32
};

template <bool ALIGN16, int FMT>
__global__ void __launch_bounds__(kThreads, 1) attn_kernel(const __grid_constant__ KernelParams kp) {
  const AttnParams& p = kp.p;
  extern __shared__ uint8_t smem_raw[];
  // 1 KB alignment for the swizzled tiles (the launch reserves the slack)
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Misc* m = reinterpret_cast<Misc*>(smem + kOffMisc);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int cid = blockIdx.x;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      // every converter warp fills its rows of every stage
      mbar_init(&m->kfull[s], kConvWarps);
      mbar_init(&m->kempty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&m->sfull[b], 1);
      mbar_init(&m->sfree[b], kSoftmaxWarps);
      mbar_init(&m->pfull[b], kSoftmaxWarps);
      mbar_init(&m->pvdone[b], 1);
      m->rescale_seq[b] = 0;
    }
    mbar_init(&m->rdv, kSoftmaxWarps);
    mbar_init(&m->erdv, kSoftmaxWarps);
    mbar_init(&m->qfull, 1);
    mbar_init(&m->qfree, 1);
    mbar_init(&m->odone, 1);
    mbar_init(&m->ofree, kSoftmaxWarps);
    mbar_init(&m->drain[0], 1);
    mbar_init(&m->drain[1], 1);
    m->abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&m->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = m->tmem_base;
  grid_dep_wait();  // the conversion kernel's slots (and any earlier reader of our outputs)

  if (warp < kSoftmaxWarps) {
    softmax_warps(smem, m, p, &kp.omap, cid, tmem, warp, lane);
  } else if (warp < kConvWarp0) {
    regs_dec<kIssueRegs>();
    if (warp == kQkWarp) qk_warp(smem, m, p, &kp.qmap, cid, tmem, lane);
    else if (warp == kPvWarp) pv_warp(smem, m, p, cid, tmem, lane);
  } else {
    regs_inc<kConvRegs>();
    if constexpr (FMT == 0)
      converter_warps<ALIGN16>(smem, m, p, cid, warp - kConvWarp0, lane);
    else
      converter_warps_bf16(smem, m, p, cid, warp - kConvWarp0, lane);
  }

  // TMEM is freed only after every tcgen05 access of this CTA is done.
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

int attn_ctas_per_split(int H) { return (H + kHeads - 1) / kHeads; }

int attn_ctas(int64_t items, int sms) {
  const int64_t cap = sms >= 1 ? sms : 1;
  return (int)(items < cap ? (items > 0 ? items : 1) : cap);
}

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

// q [T*H rows, 512] bf16 viewed by boxes of 64 heads x 64 dims (128-byte swizzle), so that
// each box lands as one K-major slab of the Q tile.  Rows past T*H read as zeros.
bool make_q_map(const AttnParams& p, CUtensorMap* map) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t gdim[2] = {(cuuint64_t)kLatent, (cuuint64_t)p.T * (cuuint64_t)p.H};
  const cuuint64_t gstride[1] = {(cuuint64_t)kLatent * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)kHeads};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(p.q), gdim, gstride, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The output as [rows of one token (and split)] x [H heads] x [512 dims], stored by boxes of
// 32 dims x 64 heads (bf16) or 32 dims x 32 heads (fp32) from the epilogue's staging (no
// swizzle).
bool make_out_map(const AttnParams& p, CUtensorMap* map) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  const bool one = p.S == 1;
  const cuuint64_t esize = one ? 2 : 4;
  const cuuint64_t gdim[3] = {(cuuint64_t)kLatent, (cuuint64_t)p.H, (cuuint64_t)p.T * (one ? 1 : (cuuint64_t)p.S)};
  const cuuint64_t gstride[2] = {(cuuint64_t)kLatent * esize, (cuuint64_t)p.H * kLatent * esize};
  const cuuint32_t box[3] = {32, one ? 64u : 32u, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  void* base = one ? p.out : static_cast<void*>(p.o_part);
  return enc(map, one ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, gdim, gstride, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool A16, int FMT>
cudaError_t set_smem_attr() {
  // once per thread and device (the attribute is per function and device; setting it again
  // with the same value from another thread is harmless)
  static thread_local bool done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(attn_kernel<A16, FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemLaunch);
  if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = true;
  return e;
}

template <bool A16, int FMT>
cudaError_t launch_variant(const KernelParams& kp, cudaStream_t s) {
  cudaError_t e = set_smem_attr<A16, FMT>();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kp.p.G, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemLaunch;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attn_kernel<A16, FMT>, kp);
}
}  // namespace

cudaError_t launch_attn(const AttnParams& p, cudaStream_t s) {
  if (p.T == 0) return cudaSuccess;
  KernelParams kp;
  kp.p = p;
  if (!make_q_map(p, &kp.qmap) || !make_out_map(p, &kp.omap)) return cudaErrorInvalidValue;
  if (p.fmt == 1) return launch_variant<true, 1>(kp, s);
  // fp8 data rows are 16-byte aligned when both caches' pages hold an even number of slots
  const bool a16 = ((int64_t)p.cache.P * kRowBytes) % 16 == 0 && ((int64_t)p.cache2.P * kRowBytes) % 16 == 0;
  return a16 ? launch_variant<true, 0>(kp, s) : launch_variant<false, 0>(kp, s);
}

}  // namespace smd
