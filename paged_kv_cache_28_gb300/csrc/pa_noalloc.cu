// pa_noalloc.cu -- split-KV decode for callers that cannot allocate device memory.
//
// pa_decode_splitkv needs a caller-supplied workspace.  Some callers cannot
// provide one: a plugin running inside a host framework that owns all device
// memory through its own pool, a latency-critical path where cudaMalloc's
// implicit device-wide synchronisation is not acceptable, or a deployment whose
// device-memory budget is fixed at start-up.  This file gives them
// pa_decode_splitkv_noalloc, which runs the same split-KV decode and merge with
// its scratch in a fixed array that lives in the library's own device image.
//
// The array below is reserved on every GPU that loads the library, until the
// process exits.  In host code its name is only a host-side stand-in, never a
// device address, so the host looks up the real address once per device with
// cudaGetSymbolAddress and hands that to the kernels.
#include <cuda_runtime.h>

#include <mutex>

#include "pa.h"
#include "pa_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up on first use.
cudaError_t scratch_address(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_addr[dev]) {
    void *ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = ptr;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" pa_status pa_decode_splitkv_noalloc(const pa_shape *shape, float *out,
                                               int32_t num_splits, const void *q,
                                               const void *k_pool, const void *v_pool,
                                               const float *k_scale, const float *v_scale,
                                               const int32_t *block_tables,
                                               const int32_t *seq_lens, float sm_scale,
                                               int32_t *err_flag, pa_stream_t stream) {
  if (!shape) return PA_ERR_INVALID_ARG;
  const size_t need = pa_splitkv_workspace_bytes(shape, num_splits);
  if (need == 0 || need > static_cast<size_t>(PA_NOALLOC_SCRATCH_BYTES))
    return PA_ERR_INVALID_ARG;
  if (shape->B == 0) return PA_OK;
  void *scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return PA_ERR_CUDA;
  pa_status st = pa_decode_splitkv(shape, out, scratch, PA_NOALLOC_SCRATCH_BYTES, num_splits, q,
                                   k_pool, v_pool, k_scale, v_scale, block_tables, seq_lens,
                                   /*opts=*/nullptr, sm_scale, err_flag, stream);
  if (st != PA_OK) return st;
  return pa_merge_lse(shape, out, scratch, num_splits, stream);
}
