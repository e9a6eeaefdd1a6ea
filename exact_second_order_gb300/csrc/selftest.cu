// Diagnostic kernels.
//
// flashbob_check_wait_timeout: one thread waits on
// an mbarrier that nothing ever arrives on, through the same bounded wait the
// tensor-core kernels use.  After the wait limit it records error code 1 in
// the device error word and returns, so the host-side report
// (flashbob_last_device_error -> FLASHBOB_ERR_TIMEOUT) can be tested without
// a fault, a trap or a hang.
//
// flashbob_mma_cycles: one CTA issues a run of tcgen05.mma of one shape
// (M = 128, K = 16, bf16 operands, fp32 accumulator, N columns; A from shared
// memory or from tensor memory, B from shared memory, both K-major in the
// 128-byte swizzle) back to back from one thread and times the run with the
// SM clock, up to the completion of the last MMA.  The schedules of the BoB
// kernels are built around this per-instruction cost; the call lets it be
// re-measured on the device at hand.  The operands are whatever shared and
// tensor memory hold (the values do not matter for the timing).
#include "internal.h"
#include "tc_common.cuh"

namespace flashbob {

__device__ unsigned long long g_mma_cycles[2];

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

constexpr int kMmaRun = 4096;  // MMAs per timed run

template <bool TS>
__global__ void __launch_bounds__(128, 1) mma_cycles_kernel(int n, unsigned int* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ uint64_t bar;
  __shared__ uint32_t tslot;
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);
    abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == 0) tc::tmem_alloc(&tslot, 512);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tb = tslot;
  if (threadIdx.x == 32) {
    // A: 128 rows x 64 bf16 at offset 0; B: n rows x 64 bf16 at 16 KiB.
    const uint64_t dA = tc::smem_desc_sw128(tc::smem_u32(smem), 16, 1024);
    const uint64_t dB = tc::smem_desc_sw128(tc::smem_u32(smem + 16384), 16, 1024);
    const uint32_t id = tc::idesc_bf16(128, n, false);
    const unsigned long long t0 = clock64();
    for (int it = 0; it < kMmaRun; it += 4) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t o = 2 * kk;  // the next 16 columns: 32 bytes >> 4
        if (TS)
          tc::mma_ts(tb, tb + 256 + 8 * kk, dB + o, id, 1);
        else
          tc::mma_ss(tb, dA + o, dB + o, id, 1);
      }
    }
    const unsigned long long t1 = clock64();
    tc::mma_commit(&bar);
    const bool ok = tc::mbar_wait(&bar, 0, &abort_flag, err);
    const unsigned long long t2 = clock64();
    g_mma_cycles[0] = ok ? t2 - t0 : 0ull;
    g_mma_cycles[1] = t1 - t0;
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tb, 512);
  }
}

}  // namespace

cudaError_t mma_cycles(int n, bool a_in_tmem, cudaStream_t stream, unsigned int* err,
                       double* cycles_per_mma) {
  constexpr int smem = 49 * 1024;  // 48 KiB of operands + alignment
  const void* k = a_in_tmem ? reinterpret_cast<const void*>(mma_cycles_kernel<true>)
                            : reinterpret_cast<const void*>(mma_cycles_kernel<false>);
  cudaError_t e = tc_set_smem(k, smem);
  if (e != cudaSuccess) return e;
  if (a_in_tmem)
    mma_cycles_kernel<true><<<1, 128, smem, stream>>>(n, err);
  else
    mma_cycles_kernel<false><<<1, 128, smem, stream>>>(n, err);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  unsigned long long c[2] = {0, 0};
  e = cudaMemcpyFromSymbolAsync(c, g_mma_cycles, sizeof(c), 0, cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return e;
  *cycles_per_mma = static_cast<double>(c[0]) / kMmaRun;
  return cudaSuccess;
}

cudaError_t launch_wait_timeout(cudaStream_t stream, unsigned int* err) {
  wait_timeout_kernel<<<1, 32, 0, stream>>>(err);
  return cudaGetLastError();
}

}  // namespace flashbob
