// Failure detection without a GPU fault: a self-test of the bounded waits.
//
// Every wait in the library's tcgen05 kernels (on an mbarrier, or on a flag another CTA
// sets) gives up after a fixed limit without progress: the waiting thread records
// XMOD_ERR_TIMEOUT in the caller's status word, raises its CTA's abort flag and returns
// false, and the kernel winds down and returns, so the CUDA context stays usable. The
// self-test runs that path for real: one thread waits, through the kernels' own
// mbar_wait, on an mbarrier phase that nothing completes (no thread arrives and no copy
// is in flight), until the limit expires.

#include <cuda_runtime.h>

#include "internal.h"
#include "tc_common.cuh"

namespace xmod {

namespace {

using namespace tc;

__global__ void wait_selftest_kernel(int* status, int* result) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // phase 0 of a one-arrival barrier that nobody arrives at
    const bool ok = mbar_wait(b, 0, (volatile int*)&abort_flag, status);
    result[0] = ok ? 1 : 0;
    result[1] = abort_flag;
  }
}

}  // namespace

}  // namespace xmod

extern "C" int xmod_selftest_wait_timeout(void* ws, size_t ws_bytes, void* stream) {
  if (!ws || ((uintptr_t)ws & 15u) || ws_bytes < 256) return XMOD_ERR_INVALID_ARG;
  int* w = (int*)ws;   // the status word at offset 0; the wait's outcome at words 1, 2
  xmod::wait_selftest_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(w, w + 1);
  xmod::count_launch();
  return cudaGetLastError() == cudaSuccess ? XMOD_OK : XMOD_ERR_CUDA;
}
