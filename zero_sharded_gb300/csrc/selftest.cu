// Self-test of the device-side failure detection.
//
// The step's kernels never wait without a limit: every mbarrier wait gives up
// after a bounded time, records CZ_ERR_TIMEOUT in the workspace status word and
// lets the kernel return, so a stuck pipeline surfaces as an error status
// instead of a hung GPU.  This entry point exercises exactly that mechanism
// (mbar_wait from ptx.cuh) on a barrier that nothing ever completes.

#include <cuda_runtime.h>

#include "cz.h"
#include "ptx.cuh"

namespace {

__global__ void bounded_wait_probe(int* status, int64_t timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    cz::mbar_init(&bar, 1);      // one arrival expected; none will come
    abort_flag = 0;
    cz::fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const bool done = cz::mbar_wait(&bar, 0, &abort_flag, status, timeout_ns);
    if (done) cz::record_status(status, CZ_ERR_DEVICE_CHECK);   // cannot happen: nobody arrives
  }
}

}  // namespace

extern "C" int cz_selftest_bounded_wait(int64_t timeout_ns, void* workspace, void* stream) {
  if (!workspace || timeout_ns < 0 || timeout_ns > 2000000000LL) return CZ_ERR_INVALID;
  bounded_wait_probe<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(static_cast<int*>(workspace), timeout_ns);
  return cudaGetLastError() == cudaSuccess ? CZ_OK : CZ_ERR_CUDA;
}
