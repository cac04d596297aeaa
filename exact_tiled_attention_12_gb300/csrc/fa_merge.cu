// fa_merge.cu — merge of partial attention results over disjoint key sets.
//
// "Flash Attention" tutorial, 2.Online Softmax §3.1 and §4.1: two blocks'
// softmax states merge exactly once they are brought to a common reference
// max; §七 names the uses (ring attention, streaming inference / prefix
// caching, distributed softmax).  A normalised partial result (O_k, LSE_k)
// is the state m = LSE_k, ℓ = 1, Õ = O_k, so for one query row
//   LSE = ln Σ_k e^{LSE_k},   O = Σ_k e^{LSE_k − LSE} O_k
// (taking the common reference m = max_k LSE_k inside the sum).  A part that
// saw no key of a row has LSE_k = −∞ and weight 0; a row no part saw gets
// O = 0 and LSE = −∞.
//
// One warp per row: lane k < n_parts holds part k's weight, and the lanes
// stride over the d columns (coalesced).  HBM-bound: it reads n_parts rows of
// O and LSE and writes one.
#include <cuda_fp16.h>

#include "fa_kernels.h"

namespace fa {
namespace {

constexpr unsigned kFullMask = 0xffffffffu;

// ELEM: 0 fp32, 1 bf16, 2 fp16.
template <int ELEM>
__device__ __forceinline__ float load_o(const void* p, long long i) {
  if constexpr (ELEM == 1)
    return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
  else if constexpr (ELEM == 2)
    return __half2float(static_cast<const __half*>(p)[i]);
  else
    return static_cast<const float*>(p)[i];
}

template <int ELEM>
__device__ __forceinline__ void store_o(void* p, long long i, float x) {
  if constexpr (ELEM == 1)
    static_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(x);
  else if constexpr (ELEM == 2)
    static_cast<__half*>(p)[i] = __float2half_rn(x);
  else
    static_cast<float*>(p)[i] = x;
}

template <int ELEM>
__global__ void __launch_bounds__(256) merge_kernel(const __grid_constant__ MergeArgs a) {
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= a.rows) return;   // warp-uniform
  const float mine = lane < a.n_parts ? a.lse_parts[lane][row] : -INFINITY;
  float m = mine;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFullMask, m, o));
  const long long base = row * (long long)a.d;
  __syncwarp();   // every lane has read its LSE part before anything is written
  if (m == -INFINITY) {   // warp-uniform after the reduction
    for (int c = lane; c < a.d; c += 32) store_o<ELEM>(a.o, base + c, 0.f);
    if (lane == 0) a.lse[row] = -INFINITY;
    return;
  }
  float e = lane < a.n_parts ? expf(mine - m) : 0.f;   // e^{LSE_k − m} ∈ [0, 1]
  float sum = e;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(kFullMask, sum, o);
  const float w = e / sum;                             // e^{LSE_k − LSE}
  // Every lane runs every column block, so the weight broadcasts are
  // warp-wide even when d is not a multiple of 32.
  for (int c0 = 0; c0 < a.d; c0 += 32) {
    const int c = c0 + lane;
    float acc = 0.f;
    for (int k = 0; k < a.n_parts; ++k) {
      const float wk = __shfl_sync(kFullMask, w, k);
      if (wk != 0.f && c < a.d) acc = fmaf(wk, load_o<ELEM>(a.o_parts[k], base + c), acc);
    }
    if (c < a.d) store_o<ELEM>(a.o, base + c, acc);
  }
  if (lane == 0) a.lse[row] = m + logf(sum);
}

}  // namespace

cudaError_t launch_merge(const MergeArgs& a, cudaStream_t s) {
  if (a.rows <= 0) return cudaSuccess;
  const unsigned blocks = (unsigned)((a.rows + 7) / 8);
  if (a.elem == 1)
    merge_kernel<1><<<blocks, 256, 0, s>>>(a);
  else if (a.elem == 2)
    merge_kernel<2><<<blocks, 256, 0, s>>>(a);
  else
    merge_kernel<0><<<blocks, 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace fa
