// selftest.cu -- a GPU check of the bounded barrier wait that every pipeline
// kernel relies on: one thread waits on an mbarrier that nothing will ever
// arrive on.  The wait must give up at its wall-clock limit, count a timeout
// in the status words and let the kernel exit normally, leaving the context
// usable.  No fault, trap or endless loop is involved.
#include <cuda_runtime.h>

#include "launch.h"
#include "ptx.cuh"
#include "schedule.h"

namespace flp {

__global__ void wait_timeout_kernel(uint64_t limit_ns, uint32_t *status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);  // one arrival expected; none will come
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait(&bar, 0, &abort_flag, limit_ns))
    atomicAdd(status + kStatTimeout, 1u);
}

cudaError_t launch_wait_timeout(uint64_t limit_ns, uint32_t *status, cudaStream_t stream) {
  wait_timeout_kernel<<<1, 32, 0, stream>>>(limit_ns, status);
  return cudaGetLastError();
}

}  // namespace flp
