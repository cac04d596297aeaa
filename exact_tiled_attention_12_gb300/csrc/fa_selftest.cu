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
//
// bounds_check_kernel does the same for the debug build's device-side
// checks: it evaluates them on fixed valid and invalid arguments and reports
// which passed, without ever using the invalid ones for an access.
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

// The debug build's device-side checks on fixed arguments, alternately valid
// and invalid; the invalid ones must fail (and the first one's code lands in
// the fault word).  Nothing here reads or writes memory with those
// arguments: each check is only evaluated and its result stored.
__global__ void __launch_bounds__(32) bounds_check_kernel(unsigned int* fault, int* results) {
  __shared__ int abort_flag;
  if (threadIdx.x == 0) abort_flag = 0;
  __syncwarp();
  if (threadIdx.x != 0) return;
  const WaitCtx wc{&abort_flag, fault};
  results[0] = dcheck(tma_x_ok(64, 64, 128), wc, kChkTmaX, 0xF1) ? 1 : 0;            // x on a 16-byte boundary
  results[1] = dcheck(tma_x_ok(4, 64, 128), wc, kChkTmaX, 0xF1) ? 1 : 0;             // 8-byte offset: invalid
  results[2] = dcheck(tma_rows_ok(896, 128, 1024), wc, kChkTmaRows, 0xF2) ? 1 : 0;   // last box of the rows
  results[3] = dcheck(tma_rows_ok(960, 128, 1024), wc, kChkTmaRows, 0xF2) ? 1 : 0;   // runs past the end
  results[4] = dcheck(tmem_ok(384, 128, 512), wc, kChkTmem, 0xF3) ? 1 : 0;           // last 128 columns
  results[5] = dcheck(tmem_ok(448, 128, 512), wc, kChkTmem, 0xF3) ? 1 : 0;           // past the allocation
  results[6] = dcheck(smem_ok(1024, 16384, 65536, 1024), wc, kChkSmem, 0xF4) ? 1 : 0;
  results[7] = dcheck(smem_ok(512, 16384, 65536, 1024), wc, kChkSmem, 0xF4) ? 1 : 0;  // not 1024-aligned
}

}  // namespace

cudaError_t launch_wait_timeout_selftest(unsigned int* fault, cudaStream_t s) {
  wait_timeout_kernel<<<1, 64, 0, s>>>(fault);
  return cudaGetLastError();
}

cudaError_t launch_bounds_check_selftest(unsigned int* fault, int* results, cudaStream_t s) {
  bounds_check_kernel<<<1, 32, 0, s>>>(fault, results);
  return cudaGetLastError();
}

}  // namespace fa
