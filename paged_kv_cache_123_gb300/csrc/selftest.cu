// Self-test of the bounded mbarrier wait every asynchronous kernel here uses
// (tma.cuh mbar_wait_bounded): a wait on a barrier phase that nothing
// completes must give up after its cycle limit, raise the CTA's abort flag,
// and let a second waiter with a far longer limit leave through that flag —
// the path a CTA takes when a copy it waits for never lands. Nothing here
// faults or spins without a limit: both waits end by themselves.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pagedattn.h"
#include "tma.cuh"

namespace {

__global__ void bounded_wait_selftest_kernel(int* status, long long timeout_cycles) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    pa::mbar_init(pa::smem_u32(&bar), 1);   // one arrival expected; none comes
    abort_flag = 0;
    pa::mbar_fence_init();
  }
  __syncthreads();
  if (lane == 0) {
    // warp 0: the short limit; warp 1: 1000x longer, so it can only leave
    // early through the abort flag warp 0 raises
    const long long limit = warp == 0 ? timeout_cycles : timeout_cycles * 1000;
    const bool done = pa::mbar_wait_bounded(pa::smem_u32(&bar), 0, &abort_flag, limit);
    status[warp] = done ? PA_OK : PA_ERR_TIMEOUT;
  }
  __syncthreads();
  if (threadIdx.x == 0) status[2] = abort_flag;
}

}  // namespace

extern "C" PA_API int pa_selftest_bounded_wait(int* status, long long timeout_cycles,
                                               void* stream) {
  if (!status) return PA_ERR_NULL;
  if (timeout_cycles <= 0 || timeout_cycles > (1ll << 40) / 1000) return PA_ERR_SHAPE;
  bounded_wait_selftest_kernel<<<1, 64, 0, (cudaStream_t)stream>>>(status, timeout_cycles);
  const cudaError_t e = cudaGetLastError();
  if (e == cudaErrorNoKernelImageForDevice || e == cudaErrorInvalidDeviceFunction)
    return PA_ERR_DEVICE;
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
