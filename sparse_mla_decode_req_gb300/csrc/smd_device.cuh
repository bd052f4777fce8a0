// Device-side building blocks for libsmd (sm_103a): the fp8_ds_mla row format, the row
// dequantiser shared by the attention kernel and the gather export, and thin inline-PTX
// wrappers for mbarrier, TMA, tcgen05 (TMEM allocation, MMA, loads/stores, fences) and
// the UMMA descriptors.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace smd {

// ---------------------------------------------------------------- row format
// SGLang PR #26208 report, "关键源码片段": 448 fp8 NoPE + 64 bf16 RoPE = 576 data bytes,
// 7 UE8M0 scales + 1 pad = 8 scale bytes; a page holds its data rows, then its scale rows.
constexpr int kLatent = 512;
constexpr int kNope = 448;
constexpr int kRope = 64;
constexpr int kDataBytes = 576;
constexpr int kScaleBytes = 8;
constexpr int kRowBytes = kDataBytes + kScaleBytes;
constexpr int kNopePieces = kNope / 16;    // 28 pieces of 16 fp8 bytes
constexpr int kRowPieces = kDataBytes / 16;  // 36 pieces of 16 bytes per data row

struct CacheView {
  const uint8_t* base;
  int64_t page_bytes;   // P * 584
  int64_t scale_start;  // P * 576: offset of the scale rows inside a page
  int32_t P;
  int32_t log2P;        // log2(P) when P is a power of two, else -1
};

__host__ __device__ inline int32_t log2_if_pow2(int32_t P) {
  if (P <= 0 || (P & (P - 1)) != 0) return -1;
  int32_t l = 0;
  while ((1 << l) < P) ++l;
  return l;
}

__device__ __forceinline__ CacheView make_cache_view(const uint8_t* base, int32_t P) {
  return CacheView{base, (int64_t)P * kRowBytes, (int64_t)P * kDataBytes, P, log2_if_pow2(P)};
}
// The same with log2(P) already known (-1: not a power of two).
__device__ __forceinline__ CacheView make_cache_view(const uint8_t* base, int32_t P, int32_t log2P) {
  return CacheView{base, (int64_t)P * kRowBytes, (int64_t)P * kDataBytes, P, log2P};
}

// Page and in-page offset of a global slot (shifts for power-of-two page sizes).
__device__ __forceinline__ void slot_page_off(const CacheView& c, int32_t slot, int32_t& page, int32_t& off) {
  if (c.log2P >= 0) {
    page = slot >> c.log2P;
    off = slot & (c.P - 1);
  } else {
    page = slot / c.P;
    off = slot - page * c.P;
  }
}
__device__ __forceinline__ const uint8_t* row_data(const CacheView& c, int32_t slot) {
  int32_t page, off;
  slot_page_off(c, slot, page, off);
  return c.base + (int64_t)page * c.page_bytes + (int64_t)off * kDataBytes;
}
__device__ __forceinline__ const uint8_t* row_scales(const CacheView& c, int32_t slot) {
  int32_t page, off;
  slot_page_off(c, slot, page, off);
  return c.base + (int64_t)page * c.page_bytes + c.scale_start + (int64_t)off * kScaleBytes;
}

// ---------------------------------------------------------------- dequantisation
// Zero every bf16 lane whose exponent field is all ones (inf or NaN).
__device__ __forceinline__ uint32_t scrub_bf16x2(uint32_t v) {
  const uint32_t t = v & 0x7F807F80u;
  const uint32_t bad_lo = (t & 0xFFFFu) == 0x7F80u ? 0x0000FFFFu : 0u;
  const uint32_t bad_hi = (t >> 16) == 0x7F80u ? 0xFFFF0000u : 0u;
  return v & ~(bad_lo | bad_hi);
}
__device__ __forceinline__ uint4 scrub_bf16x8(uint4 v) {
  return make_uint4(scrub_bf16x2(v.x), scrub_bf16x2(v.y), scrub_bf16x2(v.z), scrub_bf16x2(v.w));
}

__device__ __forceinline__ uint32_t bf16x2_bits(__nv_bfloat162 v) { return *reinterpret_cast<uint32_t*>(&v); }

// Zero the bytes of w that encode e4m3 NaN (low 7 bits all ones).  Adding one to each
// byte's low 7 bits sets its bit 7 exactly for those bytes (no carry leaves a byte); a
// byte permute whose selectors have bit 3 set copies each byte's bit 7 over the byte.
__device__ __forceinline__ uint32_t zero_fp8_nans(uint32_t w) {
  const uint32_t hit = (w & 0x7F7F7F7Fu) + 0x01010101u;
  uint32_t mask;
  asm("prmt.b32 %0, %1, 0, 0xBA98;" : "=r"(mask) : "r"(hit));
  return w & ~mask;
}

// Dequantisation without conversion instructions.  Placing an e4m3 byte s.eeee.mmm into
// bf16 bits as s.0000eeee.mmm0000 gives a bf16 whose value times 2^120 is exactly the
// e4m3 value, for normal and subnormal encodings alike (2^(e-127)(1+m/8) * 2^120 =
// 2^(e-7)(1+m/8); m*2^-129 * 2^120 = m*2^-9).  `sel` picks two bytes of w into the low
// bytes of the two 16-bit halves (0x4140: bytes 0 and 1; 0x4342: bytes 2 and 3).
__device__ __forceinline__ uint32_t place_fp8x2(uint32_t w, uint32_t sel) {
  const uint32_t y = __byte_perm(w, 0u, sel);  // 0x00bb00aa
  // y * 16 puts each byte at bits 4..11 of its half, sign at bit 11; adding sign * 240
  // moves that bit to 15 (+ sign << 8, - sign << 4), with no carry out of a half
  const uint32_t sgn = y & 0x00800080u;
  return y * 16u + sgn * 240u;
}
__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// One 16-byte NoPE piece: 16 e4m3 bytes times 2^(code-127) -> 16 bf16 in element order
// (lo = elements 0..7, hi = 8..15).  NaN bytes become 0; so does every product that is
// not finite in bf16 (code 255 decodes to a NaN scale; codes >= 247 can overflow).
//
// dequant_fast handles the common case without a branch: no NaN byte and code <= 134,
// where one exact multiply by 2^(code-7) carries both the 2^120 of the placement and the
// scale, rounded once (exact unless the product leaves bf16's range at the bottom).
// needs_exact tells whether a piece is outside that case; dequant_piece handles any
// piece: NaN bytes zeroed, then for code > 134 2^120 first (exact), then the scale, then
// the non-finite scrub.  Both routes round the same exact product once, so they agree
// wherever both apply.
__device__ __forceinline__ bool needs_exact(uint4 in, uint32_t code) {
  const uint32_t hit = (((in.x & 0x7F7F7F7Fu) + 0x01010101u) | ((in.y & 0x7F7F7F7Fu) + 0x01010101u) |
                        ((in.z & 0x7F7F7F7Fu) + 0x01010101u) | ((in.w & 0x7F7F7F7Fu) + 0x01010101u)) &
                       0x80808080u;
  return hit != 0u || code > 134u;
}
__device__ __forceinline__ void dequant_fast(uint4 in, uint32_t code, uint4& lo, uint4& hi) {
  const uint32_t sb = (code + 120u) << 7;  // bf16 2^(code - 7)
  const uint32_t sc = sb | (sb << 16);
  const uint32_t w[4] = {in.x, in.y, in.z, in.w};
  uint32_t r[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    r[2 * i] = mul_bf16x2(place_fp8x2(w[i], 0x4140u), sc);
    r[2 * i + 1] = mul_bf16x2(place_fp8x2(w[i], 0x4342u), sc);
  }
  lo = make_uint4(r[0], r[1], r[2], r[3]);
  hi = make_uint4(r[4], r[5], r[6], r[7]);
}
__device__ __forceinline__ void dequant_piece(uint4 in, uint32_t code, uint4& lo, uint4& hi) {
  const uint32_t w[4] = {zero_fp8_nans(in.x), zero_fp8_nans(in.y), zero_fp8_nans(in.z), zero_fp8_nans(in.w)};
  if (code <= 134u) {
    dequant_fast(make_uint4(w[0], w[1], w[2], w[3]), code, lo, hi);
    return;
  }
  constexpr uint32_t k2p120 = 0x7B807B80u;        // bf16x2 (2^120, 2^120)
  const uint32_t sb = code << 7;                  // bf16 2^(code - 127); 255 -> inf
  const uint32_t sc = sb | (sb << 16);
  uint32_t r[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    r[2 * i] = scrub_bf16x2(mul_bf16x2(mul_bf16x2(place_fp8x2(w[i], 0x4140u), k2p120), sc));
    r[2 * i + 1] = scrub_bf16x2(mul_bf16x2(mul_bf16x2(place_fp8x2(w[i], 0x4342u), k2p120), sc));
  }
  lo = make_uint4(r[0], r[1], r[2], r[3]);
  hi = make_uint4(r[4], r[5], r[6], r[7]);
}

// ---------------------------------------------------------------- debug range checks
// Status-word bits: a bounded wait gave up (bit 0), a range check of the SMD_DEBUG build
// failed (bit 1).
constexpr uint32_t kStatusTimeout = 1u;
constexpr uint32_t kStatusDeviceCheck = 2u;
// In a build with SMD_DEBUG defined, in_range(cond, status) records a failed check in the
// status word (bit 1) and returns false, so that the caller skips the access; otherwise it
// is `true` and costs nothing.  The checks restate each address's bounds from the buffer
// sizes, independently of the masking that already keeps accesses in range.
#ifdef SMD_DEBUG
__device__ __forceinline__ bool in_range(bool cond, uint32_t* status) {
  if (!cond && status != nullptr) atomicOr(status, kStatusDeviceCheck);
  return cond;
}
#else
__device__ __forceinline__ constexpr bool in_range(bool, uint32_t*) { return true; }
#endif

// ---------------------------------------------------------------- global loads
// Loads through the read-only path as volatile PTX: the compiler keeps them in program
// order and cannot sink them to their first use, so a batch of them is in flight at once.
__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}
__device__ __forceinline__ uint2 ldg_nc_v2(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}
__device__ __forceinline__ int32_t ldg_nc_s32(const void* p) {
  int32_t v;
  asm volatile("ld.global.nc.s32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}
// 16 bytes; ALIGN16 = false splits them into two 8-byte loads (pages with an odd slot
// count leave data rows only 8-byte aligned).
template <bool ALIGN16>
__device__ __forceinline__ uint4 ldg16(const uint8_t* p) {
  if constexpr (ALIGN16) {
    return ldg_nc_v4(p);
  } else {
    const uint2 a = ldg_nc_v2(p), b = ldg_nc_v2(p + 8);
    return make_uint4(a.x, a.y, b.x, b.y);
  }
}

// 2^x with the hardware approximation (relative error about 2^-22); -inf gives 0.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------- misc PTX
__device__ __forceinline__ uint32_t smem_u32(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
               : "memory");
  return v;
}

// ---------------------------------------------------------------- dependent launches
// A grid launched with programmatic stream serialization may start before the previous
// kernel in the stream has finished; it must wait here before it touches memory that
// kernel reads or writes.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
// try_wait with a suspend-time hint: a waiting thread sleeps until the phase completes or
// about 0.1 ms passes, instead of spinning on the issue slots its neighbours need.
constexpr uint32_t kSuspendHintNs = 100000;
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}
// Non-blocking probe of a phase: true once the phase with `parity` has completed.
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait: gives up after `limit_ns` of wall time and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
  return true;
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

// ---------------------------------------------------------------- clusters
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// The shared::cluster address, in CTA `rank` of the cluster, of this CTA's shared::cta
// address `local` (the same offset in the other CTA's shared memory).
__device__ __forceinline__ uint32_t mapa_shared(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}
// 32-bit load from shared::cluster address `addr` (possibly another CTA's).
__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
// Every thread of every CTA of the cluster (all threads execute it): the CTAs' shared
// memory writes before it are visible to the cluster after it.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Per-warpgroup register budget changes (all four warps of a warpgroup execute them).
template <uint32_t N>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// ---------------------------------------------------------------- TMA
// 2-D tiled tensor load into shared memory, completing on `bar` (transaction bytes).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
          "r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// 3-D tiled tensor load into shared memory, completing on `bar` (transaction bytes).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

// Prefetch of the same 2-D box into L2 (no shared memory, no completion to wait for).
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(map), "r"(x), "r"(y)
               : "memory");
}

// Store of a 3-D box from shared memory (the tensor map clips it at the tensor's bounds),
// tracked by the issuing thread's bulk async-groups.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int x, int y, int z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(map),
               "r"(src), "r"(x), "r"(y), "r"(z)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until at most N of this thread's bulk groups still read their shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Waits until all of this thread's bulk groups are complete (their writes performed).
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// Generic-proxy shared-memory writes -> visible to the async proxy (UMMA operand reads).
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, kind::f16 (bf16 in, f32 accumulate), issued
// by one elected lane of a converged warp.  The whole warp runs the issue loop, so its
// descriptor arithmetic stays warp-uniform (uniform registers) and, unrolled with constant
// offsets, an MMA issues at the tensor core's pace (a loop run by one divergent lane with
// per-iteration descriptor math took ~90 cycles per MMA on GB300).
__device__ __forceinline__ void umma_ss_elect(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                              uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive (once) on `bar` when every MMA issued so far has completed, from one elected lane
// of a converged warp (the lane that issued the MMAs with umma_ss_elect: elect.sync picks
// the same lane for the same member mask).
__device__ __forceinline__ void umma_commit_elect(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

#define SMD_R32_OUT(r)                                                                                           \
  "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),    \
      "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),     \
      "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),    \
      "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
#define SMD_R32_IN(r)                                                                                             \
  "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),   \
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), \
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), \
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
#define SMD_R32_LIST                                                                                          \
  "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27," \
  "%28,%29,%30,%31}"

// 32 consecutive 32-bit columns of this thread's TMEM lane (warp w reads lanes
// 32(w%4)..32(w%4)+31, thread i lane 32(w%4)+i).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 " SMD_R32_LIST ", [%32];" : SMD_R32_OUT(r) : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%32], " SMD_R32_LIST ";" ::SMD_R32_IN(r), "r"(taddr)
               : "memory");
}
// 16 lanes of the warp's TMEM quarter, twice: threads 0-15 read lanes base+0..15 at
// columns [c, c+32), threads 16-31 the same lanes at columns [c+32, c+64).  This is the
// access pattern of an M=64 accumulator, whose rows sit in lanes 0-15 of each quarter.
__device__ __forceinline__ void tmem_ld16x2_32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile("tcgen05.ld.sync.aligned.16x32bx2.x32.b32 " SMD_R32_LIST ", [%32], 32;"
               : SMD_R32_OUT(r)
               : "r"(taddr));
}

// UMMA shared-memory matrix descriptor, 128-byte swizzle (sm_100 family layout:
// start >> 4 in bits [0,14), leading-dimension byte offset >> 4 in [16,30), stride-
// dimension byte offset >> 4 in [32,46), version 1 in [46,48), swizzle mode 2 in [61,64)).
// The tile base must be 1024-byte aligned (base-offset field 0).
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor for kind::f16 with bf16 A/B and f32 accumulator.
// a_mn / b_mn select MN-major (transposed) operands.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4)                          // D format: f32
         | (1u << 7)                        // A format: bf16
         | (1u << 10)                       // B format: bf16
         | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17)         // N / 8
         | ((uint32_t)(M >> 4) << 24);      // M / 16
}

// Instruction descriptor for kind::f8f6f4 with e4m3 A/B (both K-major) and f32 accumulator.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
  return (1u << 4)                          // D format: f32
         | (0u << 7)                        // A format: e4m3
         | (0u << 10)                       // B format: e4m3
         | ((uint32_t)(N >> 3) << 17)       // N / 8
         | ((uint32_t)(M >> 4) << 24);      // M / 16
}
// D[tmem] (+)= A[smem desc] * B[smem desc]^T, kind::f8f6f4 (8-bit in, f32 accumulate),
// issued by one elected lane of a converged warp.
__device__ __forceinline__ void umma_f8_elect(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                              uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Byte offset of 16-byte chunk `chunk` (0..7) of row `row` inside a 128B-swizzled slab
// whose rows are 128 bytes apart (8-row atoms of 1024 bytes).
__host__ __device__ __forceinline__ uint32_t sw128_off(uint32_t row, uint32_t chunk) {
  return row * 128u + ((chunk ^ (row & 7u)) << 4);
}

}  // namespace smd
