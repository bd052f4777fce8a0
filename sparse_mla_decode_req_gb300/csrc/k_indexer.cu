// The indexer step: the per-token choice of the top-k cached positions that the sparse
// decode then attends to.  Two kernels here (the logits kernel is in k_indexer_logits.cu):
//
//   indexer_gather_kernel: the pages' key gather from the paged fp8 key cache (vLLM PR
//     #52212 report, "关键源码片段", _cp_gather_indexer_quant_cache_gfx950_kernel): token
//     tid of a ragged batch belongs to sequence token_to_seq[tid] (valid in [0, B)) and
//     must lie in [cu_seqlen[b], cu_seqlen[b + 1]); its position in the sequence selects a
//     block-table entry whose page must lie in [0, num_pages); the position's D key bytes
//     go to k_out[tid] and its float32 scale to scale_out[tid] (0, with the key bytes left
//     as they are, for an invalid page; nothing for an invalid token).  Block offsets are
//     64-bit.  Layout 0 with 16-byte aligned rows: 32 tokens per warp when head_dim / 16 is
//     a power of two (indexer_gather_warp_kernel), else a group of head_dim / 16 lanes per
//     token (indexer_gather16_kernel); otherwise one warp per token in 4-byte words.
//
//   indexer_topk_kernel: per token the K positions of the largest finite logits among its
//     first ctx_lens[t]: a radix select over order-preserving keys (a 12-bit pass fused
//     with the one read of the row; a 10-bit pass that also compacts the keys under the
//     chosen 12-bit digit; the last 10 bits over those keys alone) finds the K-th largest
//     logit, then one ordered pass writes the positions above it (ascending) followed by
//     the lowest positions equal to it; -1 pads a token with fewer than K finite logits.  One CTA of 512 threads per token, the row's keys
//     in shared memory when it holds up to 40 K positions; when the tokens are fewer than
//     half the SMs, a cluster of four CTAs per token instead (rows up to 64 K positions),
//     each CTA a quarter of the row, merging their counts through distributed shared memory.
//     The histograms are shared-memory atomics.
#include <cuda.h>

#include <utility>

#include "smd_device.cuh"
#include "smd_internal.h"

namespace smd {
namespace {

// ------------------------------------------------------------------ key gather
constexpr int kGatherThreads = 256;

// Where token tid's key lives: its page base and in-page position, or nullptr when the
// token writes nothing (nullptr with `bad_page` when it writes only its zero scale).
struct GatherSrc {
  const uint8_t* page;
  int32_t off;
  bool bad_page;
};
__device__ __forceinline__ GatherSrc gather_src(const IndexerGatherParams& p, int64_t tid) {
  GatherSrc g{nullptr, 0, false};
  const int32_t b = __ldg(p.token_to_seq + tid);
  if (b < 0 || b >= p.B) return g;
  const int32_t start = __ldg(p.cu_seqlen + b), end = __ldg(p.cu_seqlen + b + 1);
  if (tid < start || tid >= end) return g;
  const int64_t pos = tid - start;
  const int64_t blk = pos / p.P;
  const int32_t page = blk < p.W ? __ldg(p.block_table + (int64_t)b * p.bt_stride + blk) : -1;
  if (page < 0 || page >= p.num_pages) {
    g.bad_page = true;
    return g;
  }
  g.page = p.cache + (int64_t)page * ((int64_t)p.P * (p.D + 4));
  g.off = (int32_t)(pos - blk * p.P);
  return g;
}

// Any layout and head_dim (a multiple of 4): one warp per token, 4-byte words.
__global__ void __launch_bounds__(kGatherThreads) indexer_gather_kernel(IndexerGatherParams p) {
  grid_dep_wait();  // launched as a programmatic dependent of the previous kernel
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (kGatherThreads / 32);
  for (int64_t tid = (int64_t)blockIdx.x * (kGatherThreads / 32) + (threadIdx.x >> 5); tid < p.n; tid += warps) {
    const GatherSrc g = gather_src(p, tid);
    if (g.page == nullptr) {
      if (g.bad_page && lane == 0) p.scale_out[tid] = 0.f;
      continue;
    }
    const int64_t vo = p.layout == 0 ? (int64_t)g.off * p.D : (int64_t)g.off * (p.D + 4);
    const int64_t so = p.layout == 0 ? (int64_t)p.P * p.D + 4 * g.off : vo + p.D;
    const uint32_t* src = reinterpret_cast<const uint32_t*>(g.page + vo);
    uint32_t* dst = reinterpret_cast<uint32_t*>(p.k_out + tid * p.D);
    for (int w = lane; w < p.D / 4; w += 32) dst[w] = __ldg(src + w);
    if (lane == 0) p.scale_out[tid] = __ldg(reinterpret_cast<const float*>(g.page + so));
  }
}

// Layout 0 with 16-byte aligned rows (head_dim a multiple of 16, at most 512): a group of
// head_dim / 16 lanes per token, one 16-byte load and store each, two tokens per group in
// flight.
__global__ void __launch_bounds__(kGatherThreads) indexer_gather16_kernel(IndexerGatherParams p) {
  grid_dep_wait();
  const int lanes = p.D >> 4;                 // lanes per token
  const int groups = 32 / lanes;              // tokens per warp at a time
  const int lane = threadIdx.x & 31;
  const int grp = lane / lanes, c = lane - grp * lanes;
  const bool active = grp < groups;
  const int64_t per_step = ((int64_t)gridDim.x * (kGatherThreads / 32)) * groups;
  int64_t tid = ((int64_t)blockIdx.x * (kGatherThreads / 32) + (threadIdx.x >> 5)) * groups + grp;
  for (; tid < p.n; tid += 2 * per_step) {
    const int64_t t2 = tid + per_step;
    const GatherSrc g1 = active ? gather_src(p, tid) : GatherSrc{nullptr, 0, false};
    const GatherSrc g2 = active && t2 < p.n ? gather_src(p, t2) : GatherSrc{nullptr, 0, false};
    uint4 v1 = make_uint4(0, 0, 0, 0), v2 = make_uint4(0, 0, 0, 0);
    float s1 = 0.f, s2 = 0.f;
    if (g1.page != nullptr) {
      v1 = ldg_nc_v4(g1.page + (int64_t)g1.off * p.D + 16 * c);
      if (c == 0) s1 = __ldg(reinterpret_cast<const float*>(g1.page + (int64_t)p.P * p.D + 4 * g1.off));
    }
    if (g2.page != nullptr) {
      v2 = ldg_nc_v4(g2.page + (int64_t)g2.off * p.D + 16 * c);
      if (c == 0) s2 = __ldg(reinterpret_cast<const float*>(g2.page + (int64_t)p.P * p.D + 4 * g2.off));
    }
    if (g1.page != nullptr) *reinterpret_cast<uint4*>(p.k_out + tid * p.D + 16 * c) = v1;
    if (g2.page != nullptr) *reinterpret_cast<uint4*>(p.k_out + t2 * p.D + 16 * c) = v2;
    if (c == 0 && active) {
      if (g1.page != nullptr || g1.bad_page) p.scale_out[tid] = s1;
      if (t2 < p.n && (g2.page != nullptr || g2.bad_page)) p.scale_out[t2] = s2;
    }
  }
}

// Layout 0 with 16-byte aligned rows and PIECES = head_dim / 16 a power of two (head_dim
// 16 .. 512): each warp takes 32 consecutive tokens per step.  Lane l resolves token l's
// page and in-page position (the index reads coalesced across the warp) and moves its
// scale; then the warp copies the 32 rows as 32 * PIECES 16-byte pieces, lane l taking
// pieces l, l + 32, ... (consecutive lanes on consecutive bytes of consecutive rows), up to
// eight of them in flight per lane, each piece's row pointer passed by a shuffle from the
// lane that resolved it.  Four CTAs per SM (64 registers a thread): the bytes in flight,
// not the instructions, set its rate (three CTAs at 78 registers moved 0.80 of the measured
// copy bandwidth on the large-batch indexer shape, four 0.89, six, spilling, 0.77).
template <int PIECES>
__global__ void __launch_bounds__(kGatherThreads, 4) indexer_gather_warp_kernel(IndexerGatherParams p) {
  static_assert(PIECES >= 1 && PIECES <= 32 && (PIECES & (PIECES - 1)) == 0, "a power of two up to 32");
  grid_dep_wait();
  constexpr int kRound = PIECES < 8 ? PIECES : 8;  // pieces per lane in flight
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (int64_t)gridDim.x * (kGatherThreads / 32);
  for (int64_t t0 = ((int64_t)blockIdx.x * (kGatherThreads / 32) + (threadIdx.x >> 5)) * 32; t0 < p.n;
       t0 += nwarps * 32) {
    const int64_t tid = t0 + lane;
    const GatherSrc g = tid < p.n ? gather_src(p, tid) : GatherSrc{nullptr, 0, false};
    const uint8_t* row = g.page != nullptr ? g.page + (int64_t)g.off * p.D : nullptr;
    float sc = 0.f;
    if (g.page != nullptr) sc = __ldg(reinterpret_cast<const float*>(g.page + (int64_t)p.P * p.D + 4 * g.off));
    const unsigned long long rp = reinterpret_cast<unsigned long long>(row);
#pragma unroll 1
    for (int j0 = 0; j0 < PIECES; j0 += kRound) {
      uint4 v[kRound];
      uint32_t have = 0u;  // bit j: piece j's row is valid
#pragma unroll
      for (int j = 0; j < kRound; ++j) {
        const int q = lane + 32 * (j0 + j);  // piece q: row q / PIECES, piece q % PIECES of it
        const uint8_t* src = reinterpret_cast<const uint8_t*>(__shfl_sync(0xffffffffu, rp, q / PIECES));
        v[j] = make_uint4(0, 0, 0, 0);
        if (src != nullptr) {
          v[j] = ldg_nc_v4(src + 16 * (q % PIECES));
          have |= 1u << j;
        }
      }
#pragma unroll
      for (int j = 0; j < kRound; ++j) {
        const int q = lane + 32 * (j0 + j);
        if ((have >> j) & 1u) *reinterpret_cast<uint4*>(p.k_out + (t0 + q / PIECES) * p.D + 16 * (q % PIECES)) = v[j];
      }
    }
    if (tid < p.n && (g.page != nullptr || g.bad_page)) p.scale_out[tid] = sc;
  }
}

// ------------------------------------------------------------------ top-k
constexpr int kTopkThreads = 512;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kTopkChunk = 8192;                     // positions per ordered-pass step (512 per warp)
constexpr int kTopkSmemKeys = 40 * 1024;             // rows up to this length keep their keys in shared memory
constexpr int kTopkCand = 8192;                      // candidates kept after the first radix pass (long rows)
constexpr int kTopkBins1 = 4096;                     // first pass: the keys' top 12 bits

// Order-preserving key of a logit: larger logit, larger key; -inf and NaN map to 0 and are
// never selected; -0 is read as +0 (adding +0 turns it into +0).  A negative value's bits
// all flip, a positive one's sign bit sets.  Every finite key is at least 2^23, so the top
// 12 bits of key 0 (bin 0 of the first histogram) hold no finite logit.
__device__ __forceinline__ uint32_t order_key(float x) {
  const uint32_t u = __float_as_uint(x + 0.0f);
  const uint32_t k = u ^ ((uint32_t)((int32_t)u >> 31) | 0x80000000u);
  return x > -INFINITY ? k : 0u;
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
  // every warp scans the warps' totals with shuffles (lane w holding warp w's)
  int xa = lane < kTopkWarps ? wsum[lane][0] : 0, xb = lane < kTopkWarps ? wsum[lane][1] : 0;
#pragma unroll
  for (int o = 1; o < kTopkWarps; o <<= 1) {
    const int va = __shfl_up_sync(0xffffffffu, xa, o), vb = __shfl_up_sync(0xffffffffu, xb, o);
    if (lane >= o) {
      xa += va;
      xb += vb;
    }
  }
  const int wa = __shfl_sync(0xffffffffu, xa, warp > 0 ? warp - 1 : 0);
  const int wb = __shfl_sync(0xffffffffu, xb, warp > 0 ? warp - 1 : 0);
  pa = (warp > 0 ? wa : 0) + ia - a;
  pb = (warp > 0 ? wb : 0) + ib - b;
  ta = __shfl_sync(0xffffffffu, xa, kTopkWarps - 1);
  tb = __shfl_sync(0xffffffffu, xb, kTopkWarps - 1);
  __syncthreads();  // wsum is reused by the next call
}

// Counts keys into `hist` by the digit (k >> shift) & (bins - 1) among those with
// (k & mask) == prefix (shared-memory atomics; aggregating equal digits within a warp with
// a match instruction first measured slower on GB300: 26.6 against 20.5 µs on the
// mid-batch indexer shape).
__device__ __forceinline__ void count_digit(uint32_t k, bool in, uint32_t mask, uint32_t prefix, int shift,
                                            uint32_t bins, uint32_t* hist) {
  // prefix holds a finite key's top digit (>= 8), so key 0 never matches
  if (in && (k & mask) == prefix) atomicAdd(&hist[(k >> shift) & (bins - 1u)], 1u);
}

// The digit holding the remaining-th largest counted key, scanning `bins` bins from the top,
// and the rank left inside it (set only when there are at least `remaining` keys); returns
// the number of keys counted.  Every thread of the block calls it.
__device__ __forceinline__ int pick_digit(const uint32_t* hist, uint32_t bins, uint32_t remaining, int (*wsum)[2],
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
  return total;
}

// One pass over the keys [0, m) that load4(i, k) gives four at a time (k[j] = the key at
// i + j, 0 past m): the histogram of the digit (key >> 10) & 1023 of the keys with
// (key & mask) == prefix into hist (1024 bins, zeroed by the caller), and those keys
// appended, unordered, to cand while fewer than cap of them (*ncand, zeroed by the caller,
// ends at their number, which may exceed cap).  A warp makes its appends of a step with one
// shared-memory atomic, and only in steps where one of its lanes has a key to append.
// Every thread of the block calls it.
template <class Load4>
__device__ __forceinline__ void count_and_compact(Load4 load4, int m, uint32_t mask, uint32_t prefix, uint32_t* hist,
                                                  uint32_t* cand, uint32_t cap, uint32_t* ncand) {
  const int lane = threadIdx.x & 31;
  constexpr int kStep = kTopkThreads * 4;
  const int m_round = (m + kStep - 1) / kStep * kStep;  // warp-uniform bound
  for (int i0 = threadIdx.x * 4; i0 < m_round; i0 += kStep) {
    uint32_t k[4];
    load4(i0, k);
    uint32_t hit = 0u;  // bit j: key j is under the prefix
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if ((k[j] & mask) == prefix) {  // a finite digit is >= 8, so key 0 never matches
        hit |= 1u << j;
        atomicAdd(&hist[(k[j] >> 10) & 1023u], 1u);
      }
    }
    if (__ballot_sync(0xffffffffu, hit != 0u) == 0u) continue;
    const int c = __popc(hit);
    int incl = c;  // inclusive scan of the lanes' counts
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    uint32_t base = 0u;
    if (lane == 31) base = atomicAdd(ncand, (uint32_t)incl);
    uint32_t at = __shfl_sync(0xffffffffu, base, 31) + (uint32_t)(incl - c);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if ((hit >> j) & 1u) {
        if (at < cap) cand[at] = k[j];
        ++at;
      }
    }
  }
}

// Ordered output over the positions [0, m) of a row (or of a CTA's slice of it, position
// pos0 + i for index i): those whose key is above tau go to out[base_gt + rank] in
// ascending position, those equal to tau (tau != 0) to out[n_gt + base_eq + rank] while
// that rank is below need_eq.  Per step each warp owns kTopkChunk / kTopkWarps consecutive
// positions and lane l takes every 32nd of them from l (shared-memory reads free of bank
// conflicts); a position's rank is its warp's offset (one block-wide scan of the warps'
// counts per step) plus the warp ballots of the positions before it.  base_gt and base_eq
// come back advanced by the counts of [0, m).  ONE_TIE: at most one key of the whole row
// equals tau (the usual case), so its position goes straight to out[n_gt] and the ties take
// no ballots (base_eq then comes back unchanged).  Every thread of the block calls it.
template <bool ONE_TIE, class KeyAt>
__device__ __forceinline__ void ordered_pass(KeyAt key_at, int m, uint32_t tau, int need_eq, int n_gt, int pos0,
                                             int32_t* out, int& base_gt, int& base_eq, int (*wsum)[2]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t before = (1u << lane) - 1u;
  constexpr int kPerWarp = kTopkChunk / kTopkWarps;
  for (int c0 = 0; c0 < m; c0 += kTopkChunk) {
    const int w0 = c0 + warp * kPerWarp;
    constexpr int kSteps = kPerWarp / 32;
    uint32_t bg[kSteps], be[kSteps];  // the warp's ballots, kept for the writes
    int cg = 0, ce = 0;               // the warp's counts (warp-uniform)
#pragma unroll
    for (int k = 0; k < kSteps; ++k) {
      const int i = w0 + 32 * k + lane;
      const uint32_t key = i < m ? key_at(i) : 0u;
      bg[k] = __ballot_sync(0xffffffffu, key > tau);  // key 0 (not finite) is never above tau
      cg += __popc(bg[k]);
      if constexpr (ONE_TIE) {
        if (tau != 0u && key == tau) out[n_gt] = pos0 + i;
      } else {
        be[k] = __ballot_sync(0xffffffffu, tau != 0u && key == tau);
        ce += __popc(be[k]);
      }
    }
    int og, oe, tg, te;
    block_scan2(lane == 0 ? cg : 0, lane == 0 ? ce : 0, og, oe, tg, te, wsum);
    og = __shfl_sync(0xffffffffu, og, 0) + base_gt;
    oe = __shfl_sync(0xffffffffu, oe, 0) + base_eq;
#pragma unroll
    for (int k = 0; k < kSteps; ++k) {
      const int i = w0 + 32 * k + lane;
      if ((bg[k] >> lane) & 1u) out[og + __popc(bg[k] & before)] = pos0 + i;
      og += __popc(bg[k]);
      if constexpr (!ONE_TIE) {
        if ((be[k] >> lane) & 1u) {
          const int r = oe + __popc(be[k] & before);
          if (r < need_eq) out[n_gt + r] = pos0 + i;
        }
        oe += __popc(be[k]);
      }
    }
    base_gt += tg;
    base_eq += te;
  }
}

// IN_SMEM: the row's keys are kept in shared memory (rows up to kTopkSmemKeys positions);
// otherwise every pass reads the row from global memory again.
template <bool IN_SMEM>
__global__ void __launch_bounds__(kTopkThreads, 2) indexer_topk_kernel(IndexerTopkParams p) {
  grid_dep_wait();  // the logits kernel before it, launched as its programmatic dependent
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
  const int tid = threadIdx.x;
  constexpr bool in_smem = IN_SMEM;  // the launch gives L keys of shared memory then
  auto key_at = [&](int i) -> uint32_t { return in_smem ? skey[i] : order_key(__ldg(row + i)); };

  for (int i = tid; i < kTopkBins1; i += kTopkThreads) hist[i] = 0u;
  if (tid == 0) s_ncand = 0u;
  __syncthreads();
  // one read of the row (four vector loads in flight per thread where aligned): keys into
  // shared memory and the first pass's histogram (top 12 bits) of the finite logits
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
      uint32_t kk[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {  // past the row: -inf, key 0, not counted
        kk[k] = order_key(v[u][k]);
        if (kk[k] != 0u) atomicAdd(&hist[kk[k] >> 20], 1u);
      }
      if (in_smem) {  // one 16-byte store where all four are in the row
        if (i0 + 4 <= n) *reinterpret_cast<uint4*>(skey + i0) = make_uint4(kk[0], kk[1], kk[2], kk[3]);
        else
#pragma unroll
          for (int k = 0; k < 4; ++k)
            if (i0 + k < n) skey[i0 + k] = kk[k];
      }
    }
  }
  __syncthreads();
  // the finite logits' count, and the 12-bit digit holding the K-th largest when above K
  const int total = pick_digit(hist, kTopkBins1, (uint32_t)p.K, wsum, &s_digit, &s_left);

  uint32_t tau = 0u;      // key of the K-th largest logit (0: take every finite one)
  int need_eq = 0;        // positions equal to tau to take
  int n_tie = 0;          // positions equal to tau in the row
  if (total > p.K) {
    uint32_t prefix = s_digit << 20, mask = 0xFFF00000u;
    uint32_t remaining = s_left;
    // the next 10 bits: one pass over the row counts them for the keys under the chosen
    // 12-bit digit and compacts those keys (unordered) while they fit
    for (int i = tid; i < 1024; i += kTopkThreads) hist[i] = 0u;
    __syncthreads();
    const bool vec_row = (reinterpret_cast<uintptr_t>(row) & 15u) == 0;
    count_and_compact(
        [&](int i0, uint32_t (&k)[4]) {
          if (in_smem && i0 + 4 <= n) {
            const uint4 v = *reinterpret_cast<const uint4*>(skey + i0);
            k[0] = v.x; k[1] = v.y; k[2] = v.z; k[3] = v.w;
          } else if (!in_smem && vec_row && i0 + 4 <= n) {
            const float4 f = __ldg(reinterpret_cast<const float4*>(row + i0));
            k[0] = order_key(f.x); k[1] = order_key(f.y); k[2] = order_key(f.z); k[3] = order_key(f.w);
          } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) k[j] = i0 + j < n ? key_at(i0 + j) : 0u;
          }
        },
        n, mask, prefix, hist, cand, (uint32_t)kTopkCand, &s_ncand);
    __syncthreads();
    const uint32_t ncand = s_ncand;
    (void)pick_digit(hist, 1024u, remaining, wsum, &s_digit, &s_left);
    prefix |= s_digit << 10;
    mask |= 1023u << 10;
    remaining = s_left;
    // the last 10 bits over the candidates (or the whole row if they did not fit)
    for (int i = tid; i < 1024; i += kTopkThreads) hist[i] = 0u;
    __syncthreads();
    const bool compact = ncand <= (uint32_t)kTopkCand;
    const int m = compact ? (int)ncand : n;
    const int m_round = (m + kTopkThreads - 1) / kTopkThreads * kTopkThreads;
    for (int i = tid; i < m_round; i += kTopkThreads) {
      const uint32_t k = i < m ? (compact ? cand[i] : key_at(i)) : 0u;
      count_digit(k, i < m, mask, prefix, 0, 1024u, hist);
    }
    __syncthreads();
    (void)pick_digit(hist, 1024u, remaining, wsum, &s_digit, &s_left);
    tau = prefix | s_digit;
    need_eq = (int)s_left;
    n_tie = (int)hist[s_digit];  // keys equal to tau: all 32 bits chosen
  }
  const int n_gt = total > p.K ? p.K - need_eq : total;  // positions strictly above tau (all finite if none)
  // ordered pass: positions above tau ascending into [0, n_gt), then the lowest positions
  // equal to tau into [n_gt, K)
  int base_gt = 0, base_eq = 0;
  if (n_tie <= 1) {
    ordered_pass<true>(key_at, n, tau, need_eq, n_gt, 0, out, base_gt, base_eq, wsum);
    base_eq = n_tie;
  } else {
    ordered_pass<false>(key_at, n, tau, need_eq, n_gt, 0, out, base_gt, base_eq, wsum);
  }
  const int written = n_gt + (need_eq < base_eq ? need_eq : base_eq);
  for (int i = written + tid; i < p.K; i += kTopkThreads) out[i] = -1;
}

// Four CTAs per token as a cluster, for rows up to 64 K positions: CTA r takes a quarter of
// the row (its keys and candidates in its own shared memory); the histograms, finite counts
// and ordered-pass counts are merged by reading the other CTAs' shared memory, so every CTA
// picks the same digits and writes its own positions at the right offsets.
constexpr int kTkCluster = 4;
constexpr int kTkSliceMax = 16 * 1024;   // keys per CTA

__global__ void __launch_bounds__(kTopkThreads, 2) indexer_topk_cluster_kernel(IndexerTopkParams p) {
  grid_dep_wait();
  extern __shared__ uint32_t dyn[];        // [slice keys][candidates], kTkSliceMax each at most
  __shared__ uint32_t hist[kTopkBins1];    // this CTA's counts
  __shared__ uint32_t mhist[kTopkBins1];   // the cluster's counts
  __shared__ int wsum[kTopkWarps][2];
  __shared__ int s_cnt[2];                 // this CTA's published counts
  __shared__ uint32_t s_digit, s_left, s_ncand;
  const uint32_t rank = cluster_ctarank();
  const int t = blockIdx.x / kTkCluster;
  const int n = max(0, min(__ldg(p.ctx_lens + t), p.L));
  const int chunk = ((n + kTkCluster - 1) / kTkCluster + 3) & ~3;   // a multiple of 4 positions
  const int s0 = min(n, (int)rank * chunk), s1 = min(n, s0 + chunk);
  const int m = s1 - s0;                                             // this CTA's positions
  const int cap = p.slice_cap;
  uint32_t* const skey = dyn;
  uint32_t* const cand = dyn + cap;
  const float* row = p.logits + (int64_t)t * p.stride + s0;
  int32_t* out = p.topk + (int64_t)t * p.K;
  const int tid = threadIdx.x;
  auto merged = [&](uint32_t* local, int bins) {  // mhist[i] = sum over the cluster of local[i]
    for (int i = tid; i < bins; i += kTopkThreads) {
      const uint32_t a = smem_u32(local + i);
      uint32_t v = 0u;
#pragma unroll
      for (int r = 0; r < kTkCluster; ++r) v += ld_cluster_u32(mapa_shared(a, (uint32_t)r));
      mhist[i] = v;
    }
  };
  // the two counts every CTA published in s_cnt (after a cluster barrier): the sums over
  // the CTAs ranked below this one and over all of them
  auto cluster_sum2 = [&](int& below_a, int& below_b, int& all_a, int& all_b) {
    below_a = below_b = all_a = all_b = 0;
    for (int r = 0; r < kTkCluster; ++r) {
      const int x = (int)ld_cluster_u32(mapa_shared(smem_u32(&s_cnt[0]), (uint32_t)r));
      const int y = (int)ld_cluster_u32(mapa_shared(smem_u32(&s_cnt[1]), (uint32_t)r));
      if (r < (int)rank) {
        below_a += x;
        below_b += y;
      }
      all_a += x;
      all_b += y;
    }
  };

  for (int i = tid; i < kTopkBins1; i += kTopkThreads) hist[i] = 0u;
  __syncthreads();
  // one read of the slice: keys into shared memory and the 12-bit histogram of the finite logits
  const bool vec = (reinterpret_cast<uintptr_t>(row) & 15u) == 0;
  constexpr int kU = 4;
  for (int b0 = 0; b0 < m; b0 += kTopkThreads * 4 * kU) {
    float v[kU][4];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int i0 = b0 + (u * kTopkThreads + tid) * 4;
      if (vec && i0 + 4 <= m) {
        const float4 f = __ldg(reinterpret_cast<const float4*>(row + i0));
        v[u][0] = f.x; v[u][1] = f.y; v[u][2] = f.z; v[u][3] = f.w;
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) v[u][k] = i0 + k < m ? __ldg(row + i0 + k) : -INFINITY;
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int i0 = b0 + (u * kTopkThreads + tid) * 4;
      uint32_t kk[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {  // past the slice: -inf, key 0, not counted
        kk[k] = order_key(v[u][k]);
        if (kk[k] != 0u) atomicAdd(&hist[kk[k] >> 20], 1u);
      }
      if (i0 + 4 <= m) *reinterpret_cast<uint4*>(skey + i0) = make_uint4(kk[0], kk[1], kk[2], kk[3]);
      else
#pragma unroll
        for (int k = 0; k < 4; ++k)
          if (i0 + k < m) skey[i0 + k] = kk[k];
    }
  }
  cluster_sync();  // every CTA's histogram complete
  merged(hist, kTopkBins1);
  cluster_sync();  // every CTA has read the others' histograms
  // the cluster's finite count, and the 12-bit digit holding the K-th largest when above K
  const int total = pick_digit(mhist, kTopkBins1, (uint32_t)p.K, wsum, &s_digit, &s_left);

  uint32_t tau = 0u;
  int need_eq = 0;
  int n_tie = 0;  // positions of the row equal to tau
  if (total > p.K) {  // the same decision in every CTA of the cluster
    uint32_t prefix = s_digit << 20, mask = 0xFFF00000u;
    uint32_t remaining = s_left;
    // the next 10 bits: one pass over the slice counts them for the keys under the chosen
    // 12-bit digit and compacts those keys; the last 10 bits are counted over those alone
    for (int i = tid; i < 1024; i += kTopkThreads) hist[i] = 0u;
    if (tid == 0) s_ncand = 0u;
    __syncthreads();
    count_and_compact(
        [&](int i0, uint32_t (&k)[4]) {
          if (i0 + 4 <= m) {
            const uint4 v = *reinterpret_cast<const uint4*>(skey + i0);
            k[0] = v.x; k[1] = v.y; k[2] = v.z; k[3] = v.w;
          } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) k[j] = i0 + j < m ? skey[i0 + j] : 0u;
          }
        },
        m, mask, prefix, hist, cand, (uint32_t)cap, &s_ncand);
    __syncthreads();
    const int nc = (int)s_ncand;  // <= m <= cap
    const int nc_round = (nc + kTopkThreads - 1) / kTopkThreads * kTopkThreads;
    for (int shift = 10; shift >= 0; shift -= 10) {
      if (shift == 0) {
        for (int i = tid; i < 1024; i += kTopkThreads) hist[i] = 0u;
        __syncthreads();
        for (int i = tid; i < nc_round; i += kTopkThreads)
          count_digit(i < nc ? cand[i] : 0u, i < nc, mask, prefix, 0, 1024u, hist);
      }
      cluster_sync();
      merged(hist, 1024);
      cluster_sync();
      (void)pick_digit(mhist, 1024u, remaining, wsum, &s_digit, &s_left);
      prefix |= s_digit << shift;
      mask |= 1023u << shift;
      remaining = s_left;
      if (shift == 0) n_tie = (int)mhist[s_digit];  // all 32 bits chosen: the keys equal to tau
      __syncthreads();
    }
    tau = prefix;
    need_eq = (int)remaining;
  }
  // this CTA's counts above and at tau, then its offsets among the cluster's
  int lg = 0, le = 0;
  for (int i = tid; i < m; i += kTopkThreads) {
    const uint32_t k = skey[i];
    lg += k != 0u && k > tau;
    le += tau != 0u && k == tau;
  }
  {
    int pa, pb, ta, tb;
    block_scan2(lg, le, pa, pb, ta, tb, wsum);
    if (tid == 0) {
      s_cnt[0] = ta;
      s_cnt[1] = tb;
    }
  }
  cluster_sync();
  int base_gt, base_eq, n_gt, n_eq;
  cluster_sum2(base_gt, base_eq, n_gt, n_eq);
  cluster_sync();  // the counts are read; the CTAs may now leave once done with their own memory
  // ordered pass over the slice: positions above tau at [base_gt, ...), the lowest equal ones
  // at n_gt + [base_eq, ...) while below need_eq
  if (n_tie <= 1)
    ordered_pass<true>([&](int i) { return skey[i]; }, m, tau, need_eq, n_gt, s0, out, base_gt, base_eq, wsum);
  else
    ordered_pass<false>([&](int i) { return skey[i]; }, m, tau, need_eq, n_gt, s0, out, base_gt, base_eq, wsum);
  if (rank == 0) {
    const int written = n_gt + (need_eq < n_eq ? need_eq : n_eq);
    for (int i = written + tid; i < p.K; i += kTopkThreads) out[i] = -1;
  }
}

// Launch as a programmatic dependent of the previous kernel in the stream: the grid may be
// scheduled while that kernel finishes and waits for it (grid_dep_wait) before its first
// global access.
template <typename... Args, typename... Act>
cudaError_t launch_dependent(void (*kernel)(Args...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                             Act&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Act>(args)...);
}

}  // namespace

cudaError_t launch_indexer_gather(const IndexerGatherParams& p, cudaStream_t s) {
  if (p.n == 0) return cudaSuccess;
  const bool fast = p.layout == 0 && p.D % 16 == 0 && p.D <= 512 && ((int64_t)p.P * (p.D + 4)) % 16 == 0 &&
                    (reinterpret_cast<uintptr_t>(p.cache) & 15u) == 0 &&
                    (reinterpret_cast<uintptr_t>(p.k_out) & 15u) == 0;
  const int pieces = p.D / 16;
  if (fast && (pieces & (pieces - 1)) == 0) {  // 32 tokens per warp
    int64_t blocks = (p.n + (kGatherThreads / 32) * 32 - 1) / ((kGatherThreads / 32) * 32);
    if (blocks > 65535 * 16) blocks = 65535 * 16;
    switch (pieces) {
      case 1: return launch_dependent(indexer_gather_warp_kernel<1>, dim3((unsigned)blocks), dim3(kGatherThreads), 0, s, p);
      case 2: return launch_dependent(indexer_gather_warp_kernel<2>, dim3((unsigned)blocks), dim3(kGatherThreads), 0, s, p);
      case 4: return launch_dependent(indexer_gather_warp_kernel<4>, dim3((unsigned)blocks), dim3(kGatherThreads), 0, s, p);
      case 8: return launch_dependent(indexer_gather_warp_kernel<8>, dim3((unsigned)blocks), dim3(kGatherThreads), 0, s, p);
      case 16: return launch_dependent(indexer_gather_warp_kernel<16>, dim3((unsigned)blocks), dim3(kGatherThreads), 0, s, p);
      default: return launch_dependent(indexer_gather_warp_kernel<32>, dim3((unsigned)blocks), dim3(kGatherThreads), 0, s, p);
    }
  }
  const int64_t per = (kGatherThreads / 32) * (fast ? 32 / (p.D / 16) * 2 : 1);  // tokens per CTA per step
  int64_t blocks = (p.n + per - 1) / per;
  if (blocks > 65535 * 16) blocks = 65535 * 16;
  if (fast) return launch_dependent(indexer_gather16_kernel, dim3((unsigned)blocks), dim3(kGatherThreads), 0, s, p);
  return launch_dependent(indexer_gather_kernel, dim3((unsigned)blocks), dim3(kGatherThreads), 0, s, p);
}

cudaError_t launch_indexer_topk(const IndexerTopkParams& p, cudaStream_t s) {
  if (p.T == 0 || p.K == 0) return cudaSuccess;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int slice = ((p.L + kTkCluster - 1) / kTkCluster + 3) & ~3;
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) sms = 1;
  if (slice <= kTkSliceMax && 2 * p.T <= sms) {
    // few tokens (one CTA each would leave most SMs idle): a cluster of four CTAs per token,
    // each with its quarter of the row in shared memory
    static thread_local bool done_c[64] = {};
    if (dev < 0 || dev >= 64 || !done_c[dev]) {
      e = cudaFuncSetAttribute(indexer_topk_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               2 * kTkSliceMax * 4);
      if (e != cudaSuccess) return e;
      if (dev >= 0 && dev < 64) done_c[dev] = true;
    }
    IndexerTopkParams q = p;
    q.slice_cap = slice;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.T * kTkCluster, 1, 1);
    cfg.blockDim = dim3(kTopkThreads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)2 * slice * 4;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kTkCluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // a dependent of the logits kernel
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, indexer_topk_cluster_kernel, q);
  }
  // many tokens, or rows too long for the clusters: one CTA per token (rows up to 40 K
  // positions in shared memory, longer ones re-read from global memory on every pass)
  static thread_local bool done[64] = {};
  if (dev < 0 || dev >= 64 || !done[dev]) {
    e = cudaFuncSetAttribute(indexer_topk_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (kTopkCand + kTopkSmemKeys) * 4);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(indexer_topk_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kTopkCand * 4);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) done[dev] = true;
  }
  if (p.L <= kTopkSmemKeys)
    return launch_dependent(indexer_topk_kernel<true>, dim3((unsigned)p.T), dim3(kTopkThreads),
                            (size_t)(kTopkCand + p.L) * 4, s, p);
  return launch_dependent(indexer_topk_kernel<false>, dim3((unsigned)p.T), dim3(kTopkThreads), (size_t)kTopkCand * 4,
                          s, p);
}

}  // namespace smd
