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
// head dimensions lane, lane+32, lane+64, lane+96.  The next 32-row block is
// fetched into registers while the current one is used, so its global-load
// latency overlaps the arithmetic (these problems are small and latency
// bound: one load round trip per block instead of one per element).
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

constexpr int kThreadsF32 = 32 * kRowsPerBlock;
constexpr int kBlockRegs = kTile * kMaxD / kThreadsF32;   // floats of one 32-row block per thread

// Rows [r0, r0 + 32) of a row-major [N, d] matrix, held in registers: the
// block is 32·d contiguous floats and thread t holds elements t, t + 256, …
// (rows past N read as zero).
struct RowBlock {
  float x[kBlockRegs];
};

__device__ __forceinline__ void fetch_rows(RowBlock& b, const float* __restrict__ src, int r0, int N, int d) {
  const int n = min(N - r0, kTile) * d;
  const float* base = src + (size_t)r0 * d;
#pragma unroll
  for (int u = 0; u < kBlockRegs; ++u) {
    const int idx = (int)threadIdx.x + u * kThreadsF32;
    b.x[u] = idx < n ? base[idx] : 0.f;
  }
}

// Writes a fetched block into shared memory with a padded row stride of
// d + 1 floats (element idx goes to row idx / d, column idx % d; both are
// stepped, not divided, per element).
__device__ __forceinline__ void put_rows(float* dst, const RowBlock& b, int d) {
  const int ld = d + 1;
  const int step_r = kThreadsF32 / d, step_c = kThreadsF32 % d;
  int r = (int)threadIdx.x / d, c = (int)threadIdx.x % d;
#pragma unroll
  for (int u = 0; u < kBlockRegs; ++u) {
    if (r < kTile) dst[r * ld + c] = b.x[u];
    r += step_r;
    c += step_c;
    if (c >= d) {
      c -= d;
      ++r;
    }
  }
}

// Σ_c a[c]·b[c] over d terms with four independent partial sums.
__device__ __forceinline__ float dot_f32(const float* a, const float* b, int d) {
  float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
  int c = 0;
  for (; c + 4 <= d; c += 4) {
    s0 = fmaf(a[c], b[c], s0);
    s1 = fmaf(a[c + 1], b[c + 1], s1);
    s2 = fmaf(a[c + 2], b[c + 2], s2);
    s3 = fmaf(a[c + 3], b[c + 3], s3);
  }
  for (; c < d; ++c) s0 = fmaf(a[c], b[c], s0);
  return (s0 + s1) + (s2 + s3);
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
  RowBlock nk, nv;   // the next block of K and V, in flight
  fetch_rows(nk, kh, 0, Nk, d);
  fetch_rows(nv, vh, 0, Nk, d);
  for (int j0 = 0; j0 < key_end; j0 += kTile) {
    __syncthreads();   // every warp is done with the previous block
    put_rows(sK, nk, d);
    put_rows(sV, nv, d);
    __syncthreads();
    if (j0 + kTile < key_end) {
      fetch_rows(nk, kh, j0 + kTile, Nk, d);
      fetch_rows(nv, vh, j0 + kTile, Nk, d);
    }
    if (!live) continue;
    const int j = j0 + lane;
    const bool vis = j < Nk && (!causal || j <= i + off);
    float s = -INFINITY;
    if (vis) s = dot_f32(sQ + warp * d, sK + lane * ld, d) * scale;
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
  RowBlock nk, nv;   // the next block of K and V, in flight
  fetch_rows(nk, k + kbase, 0, Nk, d);
  fetch_rows(nv, v + kbase, 0, Nk, d);
  for (int j0 = 0; j0 < key_end; j0 += kTile) {
    __syncthreads();
    put_rows(sK, nk, d);
    put_rows(sV, nv, d);
    __syncthreads();
    if (j0 + kTile < key_end) {
      fetch_rows(nk, k + kbase, j0 + kTile, Nk, d);
      fetch_rows(nv, v + kbase, j0 + kTile, Nk, d);
    }
    if (!live) continue;
    const int j = j0 + lane;
    const bool vis = j < Nk && (!causal || j <= i + off);
    float ds = 0.f;
    if (vis) {
      const float s = dot_f32(sQ + warp * d, sK + lane * ld, d);
      const float dp = dot_f32(sG + warp * d, sV + lane * ld, d);
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
  RowBlock nq, ng;   // the next block of Q and dO, in flight
  float nl = 0.f, nd = 0.f;
  auto fetch = [&](int i0) {
    fetch_rows(nq, q + qbase, i0, Nq, d);
    fetch_rows(ng, dO + qbase, i0, Nq, d);
    if (threadIdx.x < kTile) {
      const int ii = i0 + (int)threadIdx.x;
      nl = ii < Nq ? lse[head * Nq + ii] : 0.f;
      nd = ii < Nq ? dvec[head * Nq + ii] : 0.f;
    }
  };
  if (q_begin < Nq) fetch(q_begin);
  for (int i0 = q_begin; i0 < Nq; i0 += kTile) {
    __syncthreads();
    put_rows(sQ, nq, d);
    put_rows(sG, ng, d);
    if (threadIdx.x < kTile) {
      sL[threadIdx.x] = nl;
      sD[threadIdx.x] = nd;
    }
    __syncthreads();
    if (i0 + kTile < Nq) fetch(i0 + kTile);
    if (!live) continue;
    const int i = i0 + lane;
    const bool vis = i < Nq && (!causal || j <= i + off);
    float p = 0.f, ds = 0.f;
    if (vis) {
      const float s = dot_f32(sQ + lane * ld, sK + warp * d, d);
      const float dp = dot_f32(sG + lane * ld, sV + warp * d, d);
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
