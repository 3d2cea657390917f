// diag.cu -- self-test of the kernels' bounded waits.
//
// A CTA waits on an mbarrier that nothing arrives on, through the same bounded
// wait every tcgen05 kernel uses, with a short limit.  The wait must run out,
// record H3DIT_ERR_TIMEOUT in the workspace status word and let the kernel
// return, leaving the context usable.  No trap, assert or bad address is used.
#include "internal.h"
#include "ptx.cuh"

namespace h3 {
namespace {

__global__ void unsignalled_wait_kernel(int* status, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // phase 0 never completes: no thread arrives on this barrier
    mbar_wait(&bar, 0, &abort_flag, status, limit_ns);
  }
  __syncthreads();
}

}  // namespace
}  // namespace h3

extern "C" h3dit_status h3dit_selftest_timeout(void* workspace, size_t ws_bytes, int limit_ms,
                                               void* stream) {
  if (!workspace || ws_bytes < 256 || limit_ms < 1 || limit_ms > 10000) return H3DIT_ERR_ARG;
  h3::unsignalled_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<int*>(workspace), (unsigned long long)limit_ms * 1000000ull);
  return cudaGetLastError() == cudaSuccess ? H3DIT_OK : H3DIT_ERR_CUDA;
}
