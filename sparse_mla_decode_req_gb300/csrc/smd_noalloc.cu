// smd_sparse_mla_decode_static_scratch: the decode step with its scratch memory in a
// fixed array that the library itself holds, so the call allocates nothing.
//
// Why it exists: the regular entry point wants a caller-provided workspace, which most
// callers get from cudaMalloc or a caching allocator.  Some callers cannot do that: a
// serving engine that has handed nearly all HBM to its paged KV cache at start-up and
// forbids further device allocations, a plugin loaded into a host process whose own
// allocator owns the device memory, or a latency-critical loop that cannot afford
// cudaMalloc's implicit device synchronisation.  They call this entry point instead.
//
// The scratch (status word, converted slots and split partials) lives in the file-scope
// device array g_scratch below, SMD_STATIC_SCRATCH_BYTES long.  Every GPU that loads the
// library keeps that array until the process exits.  Host code cannot pass g_scratch
// itself to a kernel (in host code the name is only a host-side stand-in), so the first
// call on each device looks up its device address with cudaGetSymbolAddress while that
// device is current and caches it; make that first call before any stream capture.  The
// cached address belongs to the device's primary context, so it is stale after
// cudaDeviceReset.  smd_read_static_scratch_status reads the status word at its start.
#include <cuda_runtime.h>

#include <mutex>

#include "smd.h"
#include "smd_internal.h"

namespace {

static __device__ __align__(256) uint8_t g_scratch[SMD_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_scratch on the current device (looked up once per device).
int scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return smd::set_error(SMD_ERR_CUDA, "cudaGetDevice failed: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return smd::set_error(SMD_ERR_UNSUPPORTED, "device index %d >= %d", dev, kMaxDevices);
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess || p == nullptr)
      return smd::set_error(SMD_ERR_CUDA, "cudaGetSymbolAddress(scratch) failed on device %d: %s", dev,
                            cudaGetErrorString(e));
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return SMD_OK;
}

}  // namespace

extern "C" SMD_API int smd_sparse_mla_decode_static_scratch(const smd_dims* dims, const void* q,
                                                            const uint8_t* kv_cache, const int32_t* block_table,
                                                            const int32_t* req_id, const int32_t* topk_idx,
                                                            const int32_t* swa_idx, const float* sink, float scale,
                                                            void* out, float* lse, int num_splits,
                                                            smd_stream_t stream) {
  const size_t need = smd_workspace_size(dims, num_splits, 0);
  if (need == 0) return SMD_ERR_INVALID_ARG;  // smd_workspace_size left the message
  if (need > (size_t)SMD_STATIC_SCRATCH_BYTES)
    return smd::set_error(SMD_ERR_WORKSPACE,
                          "this step needs %zu bytes of scratch, more than the %zu-byte static scratch array; "
                          "use fewer tokens or splits, or smd_sparse_mla_decode with a caller workspace",
                          need, (size_t)SMD_STATIC_SCRATCH_BYTES);
  void* scratch = nullptr;
  const int rc = scratch_for_current_device(&scratch);
  if (rc != SMD_OK) return rc;
  // The decode resets the status word at the start of the array itself; every other byte
  // it reads (converted slots, split partials) is written earlier in the same call.
  return smd_sparse_mla_decode(dims, q, kv_cache, block_table, req_id, topk_idx, swa_idx, sink, scale, out, lse,
                               num_splits, scratch, (size_t)SMD_STATIC_SCRATCH_BYTES, stream);
}

extern "C" SMD_API int smd_read_static_scratch_status(int32_t* device_status, smd_stream_t stream) {
  if (device_status == nullptr) return smd::set_error(SMD_ERR_INVALID_ARG, "device_status is NULL");
  int dev = 0;
  const cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return smd::set_error(SMD_ERR_CUDA, "cudaGetDevice failed: %s", cudaGetErrorString(e));
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (dev >= 0 && dev < kMaxDevices) scratch = g_scratch_ptr[dev];
  }
  if (scratch == nullptr)
    return smd::set_error(SMD_ERR_INVALID_ARG, "no static-scratch decode was made on device %d yet", dev);
  return smd_read_status(scratch, device_status, stream);
}
