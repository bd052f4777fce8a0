// Stand-alone row gather + dequantisation (a test/debug export of the stage that the
// attention kernel fuses): gidx[i] -> bf16 latent row kv_out[i, 0:512].
//
// SGLang PR #26208 report, "关键源码片段", _gather_dequant_dsv4_kernel: page = slot // P,
// offset = slot % P, data at page * stride + offset * 576, scales at page * stride +
// P * 576 + offset * 8, int64 address arithmetic; invalid slots give zero rows.
//
// One warp per row.  Lane L writes output dims [16L, 16L+16): lanes 0..27 read 16 NoPE
// bytes and one scale code, lanes 28..31 read 32 RoPE bytes; every load and store is
// 16 bytes wide and a warp's output row is one contiguous 1 KB write.  The NoPE pieces go
// through dequant_piece and the RoPE pieces through scrub_bf16x8, the same routines the
// attention kernel's converters run, so this export pins the hot path's dequantisation.
// A bf16 cache (1024-byte rows) is copied with scrub_bf16x8 on every piece, as the
// attention kernel's bf16 converters do.
#include "smd_device.cuh"
#include "smd_internal.h"

namespace smd {

template <bool ALIGN16>
__global__ void __launch_bounds__(256) gather_dequant_kernel(GatherParams p) {
  const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= p.rows) return;
  const int32_t slot = __ldg(p.gidx + row);
  uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
  if (p.fmt == 1) {
    if (slot >= 0 && (int64_t)slot < p.num_pages * p.P) {
      const uint8_t* src = p.cache + (int64_t)slot * (kLatent * 2) + lane * 32;
      lo = scrub_bf16x8(ldg16<true>(src));
      hi = scrub_bf16x8(ldg16<true>(src + 16));
    }
  } else if (slot >= 0 && (int64_t)slot < p.num_pages * p.P) {
    const CacheView c = make_cache_view(p.cache, p.P);
    const uint8_t* data = row_data(c, slot);
    if (lane < 28) {
      const uint4 raw = ldg16<ALIGN16>(data + lane * 16);
      dequant_piece(raw, __ldg(row_scales(c, slot) + (lane >> 2)), lo, hi);
    } else {
      lo = scrub_bf16x8(ldg16<ALIGN16>(data + kNope + (lane - 28) * 32));
      hi = scrub_bf16x8(ldg16<ALIGN16>(data + kNope + (lane - 28) * 32 + 16));
    }
  }
  uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.kv_out) + row * (kLatent * 2)) + lane * 2;
  dst[0] = lo;
  dst[1] = hi;
}

cudaError_t launch_gather_dequant(const GatherParams& p, cudaStream_t s) {
  if (p.rows == 0) return cudaSuccess;
  const unsigned blocks = (unsigned)((p.rows + 7) / 8);
  if (p.fmt == 1 || ((int64_t)p.P * kRowBytes) % 16 == 0)
    gather_dequant_kernel<true><<<blocks, 256, 0, s>>>(p);
  else
    gather_dequant_kernel<false><<<blocks, 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace smd
