// Tensor-core (tcgen05 / TMEM / TMA) kernels for sm_103a.
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"

namespace fbob {

namespace {

// One thread waits on an mbarrier whose phase nothing completes; the bounded
// wait gives up after limit_ns and records FBOB_ERR_TIMEOUT.
__global__ void wait_timeout_selftest_kernel(int* status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait_bounded(&bar, 0, status, limit_ns);
  __syncthreads();
}

}  // namespace

cudaError_t launch_wait_timeout_selftest(int* status, long long limit_ns,
                                         cudaStream_t stream) {
  wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(status, (unsigned long long)limit_ns);
  return cudaGetLastError();
}

bool tc_supported(const Problem&) { return false; }

cudaError_t tc_forward(const Problem&, const void*, const void*, const void*,
                       void*, float*, const Workspace&, LaunchLog&) {
  return cudaErrorNotSupported;
}

cudaError_t tc_backward(const Problem&, const void*, const void*, const void*,
                        const void*, const float*, const void*, void*, void*,
                        void*, const Workspace&, LaunchLog&) {
  return cudaErrorNotSupported;
}

cudaError_t tc_bob(const Problem&, const void*, const void*, const void*,
                   const void*, const float*, const void*, const void*,
                   const void*, const void*, void*, void*, void*, void*,
                   const Workspace&, LaunchLog&) {
  return cudaErrorNotSupported;
}

}  // namespace fbob
