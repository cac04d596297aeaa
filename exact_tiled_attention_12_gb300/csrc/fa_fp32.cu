// fa_fp32.cu — float32 attention forward/backward with SIMT arithmetic.
//
// The float32 dtype of the library: the same online-softmax tiling as the
// tensor-core path ("Flash Attention" tutorial, 2.Online Softmax §4.2, with
// blocks of 32 keys), computed with fp32 FMAs so that results agree with an
// exact evaluation to ~1e-6.  No tensor cores: bf16 products cannot reach
// that accuracy.  Nq queries over Nk keys (any sizes ≥ 1), 1 ≤ d ≤ 128;
// causal masking as in the bf16 path (key j visible to query i iff
// j ≤ i + Nk − Nq, the queries being the last Nq positions).
//
// Each warp owns one output row (a query row in the forward and in the dQ
// pass, a key row in the dK/dV pass); lane j scores key/query j of the
// current 32-row block staged in shared memory, and each lane accumulates
// head dimensions lane, lane+32, lane+64, lane+96.
#include "fa_kernels.h"

namespace fa {
namespace {

constexpr int kRowsPerBlock = 8;    // warps per block = output rows per block
constexpr int kTile = 32;           // keys (or queries) per shared-memory block
constexpr int kMaxD = 128;
constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(kFull, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(kFull, x, o);
  return x;
}

// Stages rows [r0, r0 + 32) of a [N, d] matrix into shared memory with a
// padded stride of d + 1 floats (rows past N are zero).
__device__ __forceinline__ void stage_rows(float* dst, const float* src, int r0, int N, int d) {
  const int ld = d + 1;
  for (int idx = threadIdx.x; idx < kTile * d; idx += blockDim.x) {
    const int r = idx / d, c = idx - r * d;
    dst[r * ld + c] = (r0 + r < N) ? src[(size_t)(r0 + r) * d + c] : 0.f;
  }
}

// Forward.  grid = (ceil(Nq / 8), B·H); one warp per query row.
__global__ void __launch_bounds__(32 * kRowsPerBlock) fwd_f32_kernel(const float* __restrict__ q,
                                                                     const float* __restrict__ k,
                                                                     const float* __restrict__ v, float* __restrict__ o,
                                                                     float* __restrict__ lse, int Nq, int Nk, int d,
                                                                     float scale, int causal) {
  extern __shared__ float sm[];
  const int ld = d + 1;
  float* sK = sm;
  float* sV = sK + kTile * ld;
  float* sQ = sV + kTile * ld;   // kRowsPerBlock rows of d
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t head = blockIdx.y;
  const int i = blockIdx.x * kRowsPerBlock + warp;
  const bool live = i < Nq;
  const int off = Nk - Nq;                         // causal: query i sees keys ≤ i + off
  const float* qh = q + head * (size_t)Nq * d;
  const float* kh = k + head * (size_t)Nk * d;
  const float* vh = v + head * (size_t)Nk * d;
  for (int c = lane; c < d; c += 32) sQ[warp * d + c] = live ? qh[(size_t)i * d + c] : 0.f;
  const int last_row = min(Nq - 1, (int)blockIdx.x * kRowsPerBlock + kRowsPerBlock - 1);
  const int key_end = causal ? last_row + off + 1 : Nk;   // keys any row of this block can see
  float m = -INFINITY, ell = 0.f;
  float acc[kMaxD / 32] = {0.f, 0.f, 0.f, 0.f};
  for (int j0 = 0; j0 < key_end; j0 += kTile) {
    __syncthreads();
    stage_rows(sK, kh, j0, Nk, d);
    stage_rows(sV, vh, j0, Nk, d);
    __syncthreads();
    if (!live) continue;
    const int j = j0 + lane;
    const bool vis = j < Nk && (!causal || j <= i + off);
    float s = -INFINITY;
    if (vis) {
      float dot = 0.f;
      for (int c = 0; c < d; ++c) dot = fmaf(sQ[warp * d + c], sK[lane * ld + c], dot);
      s = dot * scale;
    }
    const float mt = warp_max(s);
    if (mt == -INFINITY) continue;            // nothing visible in this block (warp-uniform)
    const float m_new = fmaxf(m, mt);
    const float alpha = expf(m - m_new);      // 0 for the first visible block
    const float p = vis ? expf(s - m_new) : 0.f;
    ell = ell * alpha + warp_sum(p);
#pragma unroll
    for (int u = 0; u < kMaxD / 32; ++u) acc[u] *= alpha;
    for (int jj = 0; jj < kTile; ++jj) {
      const float pj = __shfl_sync(kFull, p, jj);
#pragma unroll
      for (int u = 0; u < kMaxD / 32; ++u) {
        const int c = lane + 32 * u;
        if (c < d) acc[u] = fmaf(pj, sV[jj * ld + c], acc[u]);
      }
    }
    m = m_new;
  }
  if (live) {
    const float inv = 1.f / ell;
#pragma unroll
    for (int u = 0; u < kMaxD / 32; ++u) {
      const int c = lane + 32 * u;
      if (c < d) o[(head * Nq + i) * (size_t)d + c] = acc[u] * inv;
    }
    if (lane == 0) lse[head * Nq + i] = m + logf(ell);
  }
}

// D_i = Σ_c dO_ic O_ic, one warp per row; also copies LSE_i next to it.
__global__ void __launch_bounds__(256) prep_f32_kernel(const float* __restrict__ o, const float* __restrict__ dO,
                                                       const float* __restrict__ lse, float* __restrict__ dvec,
                                                       float* __restrict__ lse_copy, long long rows, int d) {
  const long long row = (long long)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  float acc = 0.f;
  for (int c = lane; c < d; c += 32) acc = fmaf(o[row * d + c], dO[row * d + c], acc);
  acc = warp_sum(acc);
  if (lane == 0) {
    dvec[row] = acc;
    lse_copy[row] = lse[row];
  }
}

// dQ_i = scale · Σ_j P_ij (dP_ij - D_i) K_j with P and dP recomputed per block.
__global__ void __launch_bounds__(32 * kRowsPerBlock) dq_f32_kernel(
    const float* __restrict__ q, const float* __restrict__ k, const float* __restrict__ v,
    const float* __restrict__ dO, const float* __restrict__ lse, const float* __restrict__ dvec,
    float* __restrict__ dq, int Nq, int Nk, int d, float scale, int causal) {
  extern __shared__ float sm[];
  const int ld = d + 1;
  float* sK = sm;
  float* sV = sK + kTile * ld;
  float* sQ = sV + kTile * ld;
  float* sG = sQ + kRowsPerBlock * d;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t head = blockIdx.y;
  const int i = blockIdx.x * kRowsPerBlock + warp;
  const bool live = i < Nq;
  const int off = Nk - Nq;
  const size_t qbase = head * (size_t)Nq * d;
  const size_t kbase = head * (size_t)Nk * d;
  for (int c = lane; c < d; c += 32) {
    sQ[warp * d + c] = live ? q[qbase + (size_t)i * d + c] : 0.f;
    sG[warp * d + c] = live ? dO[qbase + (size_t)i * d + c] : 0.f;
  }
  const float Li = live ? lse[head * Nq + i] : 0.f;
  const float Di = live ? dvec[head * Nq + i] : 0.f;
  const int last_row = min(Nq - 1, (int)blockIdx.x * kRowsPerBlock + kRowsPerBlock - 1);
  const int key_end = causal ? last_row + off + 1 : Nk;
  float acc[kMaxD / 32] = {0.f, 0.f, 0.f, 0.f};
  for (int j0 = 0; j0 < key_end; j0 += kTile) {
    __syncthreads();
    stage_rows(sK, k + kbase, j0, Nk, d);
    stage_rows(sV, v + kbase, j0, Nk, d);
    __syncthreads();
    if (!live) continue;
    const int j = j0 + lane;
    const bool vis = j < Nk && (!causal || j <= i + off);
    float ds = 0.f;
    if (vis) {
      float s = 0.f, dp = 0.f;
      for (int c = 0; c < d; ++c) {
        s = fmaf(sQ[warp * d + c], sK[lane * ld + c], s);
        dp = fmaf(sG[warp * d + c], sV[lane * ld + c], dp);
      }
      const float p = expf(s * scale - Li);
      ds = p * (dp - Di);
    }
    for (int jj = 0; jj < kTile; ++jj) {
      const float dsj = __shfl_sync(kFull, ds, jj);
#pragma unroll
      for (int u = 0; u < kMaxD / 32; ++u) {
        const int c = lane + 32 * u;
        if (c < d) acc[u] = fmaf(dsj, sK[jj * ld + c], acc[u]);
      }
    }
  }
  if (live) {
#pragma unroll
    for (int u = 0; u < kMaxD / 32; ++u) {
      const int c = lane + 32 * u;
      if (c < d) dq[qbase + (size_t)i * d + c] = acc[u] * scale;
    }
  }
}

// dV_j = Σ_i P_ij dO_i and dK_j = scale · Σ_i dS_ij Q_i, one warp per key row j.
__global__ void __launch_bounds__(32 * kRowsPerBlock) dkv_f32_kernel(
    const float* __restrict__ q, const float* __restrict__ k, const float* __restrict__ v,
    const float* __restrict__ dO, const float* __restrict__ lse, const float* __restrict__ dvec,
    float* __restrict__ dk, float* __restrict__ dv, int Nq, int Nk, int d, float scale, int causal) {
  extern __shared__ float sm[];
  const int ld = d + 1;
  float* sQ = sm;
  float* sG = sQ + kTile * ld;
  float* sK = sG + kTile * ld;
  float* sV = sK + kRowsPerBlock * d;
  float* sL = sV + kRowsPerBlock * d;
  float* sD = sL + kTile;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t head = blockIdx.y;
  const int j = blockIdx.x * kRowsPerBlock + warp;
  const bool live = j < Nk;
  const int off = Nk - Nq;
  const size_t qbase = head * (size_t)Nq * d;
  const size_t kbase = head * (size_t)Nk * d;
  for (int c = lane; c < d; c += 32) {
    sK[warp * d + c] = live ? k[kbase + (size_t)j * d + c] : 0.f;
    sV[warp * d + c] = live ? v[kbase + (size_t)j * d + c] : 0.f;
  }
  // Under the causal mask only queries i ≥ j − off see key j.
  const int first_key = blockIdx.x * kRowsPerBlock;
  const int q_begin = causal ? (max(first_key - off, 0) / kTile) * kTile : 0;
  float acc_v[kMaxD / 32] = {0.f, 0.f, 0.f, 0.f};
  float acc_k[kMaxD / 32] = {0.f, 0.f, 0.f, 0.f};
  for (int i0 = q_begin; i0 < Nq; i0 += kTile) {
    __syncthreads();
    stage_rows(sQ, q + qbase, i0, Nq, d);
    stage_rows(sG, dO + qbase, i0, Nq, d);
    if (threadIdx.x < kTile) {
      const int ii = i0 + threadIdx.x;
      sL[threadIdx.x] = ii < Nq ? lse[head * Nq + ii] : 0.f;
      sD[threadIdx.x] = ii < Nq ? dvec[head * Nq + ii] : 0.f;
    }
    __syncthreads();
    if (!live) continue;
    const int i = i0 + lane;
    const bool vis = i < Nq && (!causal || j <= i + off);
    float p = 0.f, ds = 0.f;
    if (vis) {
      float s = 0.f, dp = 0.f;
      for (int c = 0; c < d; ++c) {
        s = fmaf(sQ[lane * ld + c], sK[warp * d + c], s);
        dp = fmaf(sG[lane * ld + c], sV[warp * d + c], dp);
      }
      p = expf(s * scale - sL[lane]);
      ds = p * (dp - sD[lane]);
    }
    for (int ii = 0; ii < kTile; ++ii) {
      const float pi = __shfl_sync(kFull, p, ii);
      const float dsi = __shfl_sync(kFull, ds, ii);
#pragma unroll
      for (int u = 0; u < kMaxD / 32; ++u) {
        const int c = lane + 32 * u;
        if (c < d) {
          acc_v[u] = fmaf(pi, sG[ii * ld + c], acc_v[u]);
          acc_k[u] = fmaf(dsi, sQ[ii * ld + c], acc_k[u]);
        }
      }
    }
  }
  if (live) {
#pragma unroll
    for (int u = 0; u < kMaxD / 32; ++u) {
      const int c = lane + 32 * u;
      if (c < d) {
        dv[kbase + (size_t)j * d + c] = acc_v[u];
        dk[kbase + (size_t)j * d + c] = acc_k[u] * scale;
      }
    }
  }
}

}  // namespace

cudaError_t launch_fwd_f32(const float* q, const float* k, const float* v, float* o, float* lse, int BH, int Nq,
                           int Nk, int d, float scale, int causal, cudaStream_t s) {
  const size_t smem = (size_t)(2 * kTile * (d + 1) + kRowsPerBlock * d) * sizeof(float);
  dim3 grid((unsigned)((Nq + kRowsPerBlock - 1) / kRowsPerBlock), (unsigned)BH);
  fwd_f32_kernel<<<grid, 32 * kRowsPerBlock, smem, s>>>(q, k, v, o, lse, Nq, Nk, d, scale, causal);
  return cudaGetLastError();
}

cudaError_t launch_bwd_prep_f32(const float* o, const float* dO, const float* lse, float* dvec, float* lse_copy,
                                long long rows, int d, cudaStream_t s) {
  const unsigned blocks = (unsigned)((rows + 7) / 8);
  prep_f32_kernel<<<blocks, 256, 0, s>>>(o, dO, lse, dvec, lse_copy, rows, d);
  return cudaGetLastError();
}

cudaError_t launch_bwd_f32(const float* q, const float* k, const float* v, const float* dO, const float* lse,
                           const float* dvec, float* dq, float* dk, float* dv, int BH, int Nq, int Nk, int d,
                           float scale, int causal, cudaStream_t s) {
  const dim3 grid_q((unsigned)((Nq + kRowsPerBlock - 1) / kRowsPerBlock), (unsigned)BH);
  const size_t smem_q = (size_t)(2 * kTile * (d + 1) + 2 * kRowsPerBlock * d) * sizeof(float);
  dq_f32_kernel<<<grid_q, 32 * kRowsPerBlock, smem_q, s>>>(q, k, v, dO, lse, dvec, dq, Nq, Nk, d, scale, causal);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const dim3 grid_k((unsigned)((Nk + kRowsPerBlock - 1) / kRowsPerBlock), (unsigned)BH);
  const size_t smem_kv = (size_t)(2 * kTile * (d + 1) + 2 * kRowsPerBlock * d + 2 * kTile) * sizeof(float);
  dkv_f32_kernel<<<grid_k, 32 * kRowsPerBlock, smem_kv, s>>>(q, k, v, dO, lse, dvec, dk, dv, Nq, Nk, d, scale,
                                                              causal);
  return cudaGetLastError();
}

}  // namespace fa
