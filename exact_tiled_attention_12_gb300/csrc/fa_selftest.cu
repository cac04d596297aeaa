// fa_selftest.cu — exercises the failure path every tensor-core kernel uses.
//
// Each pipeline wait in the kernels is bounded (sm103_ptx.cuh): after its
// time limit it records a fault code in the device fault word, raises the
// CTA's abort flag so the CTA's other waits give up too, and returns false so
// the kernel unwinds and exits.  Nothing in a correct run reaches that path,
// so this kernel builds the situation on purpose without faulting or hanging
// anything: one CTA waits on an mbarrier that nothing will ever arrive at.
// Warp 0's wait runs into the limit; warp 1 waits on a second such barrier
// and returns as soon as it sees warp 0's abort.  The CTA then exits normally
// and the host reads FA_ERR_TIMEOUT from fa_sync_status().
#include "fa_kernels.h"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

__global__ void __launch_bounds__(64) wait_timeout_kernel(unsigned int* fault) {
  __shared__ __align__(8) unsigned long long bars[2];
  __shared__ int abort_flag;
  const uint32_t b0 = smem_u32(&bars[0]);
  const uint32_t b1 = smem_u32(&bars[1]);
  if (threadIdx.x == 0) {
    mbar_init(b0, 1);
    mbar_init(b1, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const WaitCtx wc{&abort_flag, fault};
  const int warp = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) {
    // Phase 0 of a fresh barrier with one expected arrival never completes.
    if (warp == 0)
      mbar_wait(b0, 0, wc, 0x0F01u);
    else
      mbar_wait(b1, 0, wc, 0x0F02u);
  }
  __syncthreads();
}

}  // namespace

cudaError_t launch_wait_timeout_selftest(unsigned int* fault, cudaStream_t s) {
  wait_timeout_kernel<<<1, 64, 0, s>>>(fault);
  return cudaGetLastError();
}

}  // namespace fa
