// A wait that runs out, for the failure-handling test: one CTA waits, through the
// library's own bounded mbarrier wait, on a barrier nothing arrives at.  The wait
// gives up, the kernel records PA_DEVERR_TIMEOUT in the error flag and returns; the
// host then checks the flag and that the context still runs work.  Nothing traps,
// nothing faults and no wait is endless.
#include "pa_common.cuh"

namespace {

__global__ void wait_nothing_arrives(int32_t *err, int32_t *finished) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    pa::mbar_init(pa::smem_u32(&bar), 1);
    pa::fence_mbar_init();
  }
  __syncthreads();
  if (!pa::mbar_wait<4096>(pa::smem_u32(&bar), 0)) pa::set_err(err, PA_DEVERR_TIMEOUT);
  __syncthreads();
  if (threadIdx.x == 0) atomicAdd(finished, 1);
}

}  // namespace

// Launches the kernel on the default stream and waits for it; returns the CUDA error.
extern "C" int run_wait_nothing_arrives(int32_t *err, int32_t *finished) {
  wait_nothing_arrives<<<1, 32>>>(err, finished);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  return static_cast<int>(e);
}
