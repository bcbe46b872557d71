// pa_noalloc.cu -- split-KV decode for callers that cannot allocate device memory.
//
// pa_decode's load-balanced split decode needs a caller-supplied workspace.  Some
// callers cannot provide one: a plugin running inside a host framework that owns
// all device memory through its own pool, a latency-critical path where
// cudaMalloc's implicit device-wide synchronisation is not acceptable, or a
// deployment whose device-memory budget is fixed at start-up.  This file gives them
// pa_decode_splitkv_noalloc, which runs the same split decode and merge with its
// scratch in a fixed array that lives in the library's own device image.
//
// The array below is reserved on every GPU that loads the library, until the
// process exits.  In host code its name is only a host-side stand-in, never a
// device address, so the host looks up the real address on the current device with
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

// Device address of the scratch array on the current device.  Looked up again on
// every call outside stream capture (cheap once the module is loaded, and right
// after a device reset); a call whose stream is being captured reuses the address the
// last lookup on this device found.
cudaError_t scratch_address(cudaStream_t stream, void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  e = cudaStreamIsCapturing(stream, &cap);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (cap == cudaStreamCaptureStatusNone || !g_scratch_addr[dev]) {
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
                                               int32_t num_segments, const void *q,
                                               const void *k_pool, const void *v_pool,
                                               const float *k_scale, const float *v_scale,
                                               const int32_t *block_tables,
                                               const int32_t *seq_lens, float sm_scale,
                                               int32_t *err_flag, pa_stream_t stream) {
  if (!shape) return PA_ERR_INVALID_ARG;
  pa_decode_opts opts = {};
  if (shape->B == 0)   // nothing to do: the shape checks of pa_decode decide the status
    return pa_decode(shape, out, q, k_pool, v_pool, k_scale, v_scale, block_tables, seq_lens,
                     &opts, sm_scale, err_flag, stream);
  if (num_segments < 0) return PA_ERR_INVALID_ARG;
  if (num_segments == 0) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return PA_ERR_CUDA;
    num_segments = pa_default_num_segments(shape, sms);
  }
  const size_t need = pa_decode_workspace_bytes(shape, num_segments);
  if (need == 0 || need > static_cast<size_t>(PA_NOALLOC_SCRATCH_BYTES))
    return PA_ERR_INVALID_ARG;
  void *scratch = nullptr;
  if (scratch_address(reinterpret_cast<cudaStream_t>(stream), &scratch) != cudaSuccess)
    return PA_ERR_CUDA;
  opts.workspace = scratch;
  opts.workspace_bytes = PA_NOALLOC_SCRATCH_BYTES;
  opts.num_segments = num_segments;
  return pa_decode(shape, out, q, k_pool, v_pool, k_scale, v_scale, block_tables, seq_lens,
                   &opts, sm_scale, err_flag, stream);
}
