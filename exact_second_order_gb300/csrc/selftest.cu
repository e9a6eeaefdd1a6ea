// Diagnostic kernel behind flashbob_check_wait_timeout: one thread waits on
// an mbarrier that nothing ever arrives on, through the same bounded wait the
// tensor-core kernels use.  After the wait limit it records error code 1 in
// the device error word and returns, so the host-side report
// (flashbob_last_device_error -> FLASHBOB_ERR_TIMEOUT) can be tested without
// a fault, a trap or a hang.
#include "internal.h"
#include "tc_common.cuh"

namespace flashbob {
namespace {

__global__ void wait_timeout_kernel(unsigned int* err) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);
    abort_flag = 0;
    tc::fence_barrier_init();
  }
  __syncthreads();
  // Phase 0 of a fresh barrier completes only after one arrival; none comes.
  if (threadIdx.x == 0) (void)tc::mbar_wait(&bar, 0, &abort_flag, err);
}

}  // namespace

cudaError_t launch_wait_timeout(cudaStream_t stream, unsigned int* err) {
  wait_timeout_kernel<<<1, 32, 0, stream>>>(err);
  return cudaGetLastError();
}

}  // namespace flashbob
