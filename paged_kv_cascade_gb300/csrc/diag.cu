// Diagnostics: the failure path of the bounded waits, exercised without a
// fault.  One thread waits on an mbarrier that nothing arrives at, through
// the same bounded wait every kernel of the library uses; when the limit
// runs out the wait records PKC_ERR_TIMEOUT in the status word, raises the
// block's abort flag and returns false, and the kernel returns normally.
#include <cuda_runtime.h>

#include "pkc_device.cuh"
#include "pkc_internal.h"

namespace pkc {
namespace {

__global__ void wait_timeout_kernel(int32_t* status, int32_t* gave_up) {
  __shared__ uint64_t bar;
  __shared__ int abort;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // Phase 0 never completes: no thread arrives.
    const bool got = mbar_wait(smem_u32(&bar), 0, &abort, status);
    *gave_up = got ? 0 : 1;
  }
  __syncthreads();
  // Every other wait of the block now returns at once (abort is set).
  if (threadIdx.x == 1) {
    const bool got = mbar_wait(smem_u32(&bar), 0, &abort, status);
    if (got || !abort) *gave_up = 0;
  }
}

}  // namespace

int launch_wait_timeout(int32_t* status, void* stream) {
  // word 32 of the status block receives 1 when the wait gave up
  wait_timeout_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(status, status + 32);
  return (int)cudaGetLastError();
}

}  // namespace pkc
