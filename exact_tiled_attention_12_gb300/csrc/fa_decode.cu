// fa_decode.cu — a decoding step: one query row per (batch, head) over Nk
// cached keys ("Flash Attention" tutorial, 2.Online Softmax §七: streaming
// inference extends a cached prefix one token at a time).
//
// One query costs 4·Nk·d FLOPs against 4·Nk·d bytes of K and V (16-bit), so
// the step is bound by HBM bandwidth; a 128-row tensor-core tile would spend
// 127 of its rows on nothing.  This kernel streams K and V with 16-byte loads
// on the CUDA cores instead:
//   * a CTA (8 warps) owns one key range of one head; a warp reads KPW
//     consecutive keys per load (G = 8, 16 or 32 lanes per key, 8 elements a
//     lane); a lane issues the next step's loads before this step's math;
//   * each lane group keeps its own online-softmax state (m, ℓ, Õ over its
//     8 head dims) — the update of 2.Online Softmax §4.1, over kUnroll keys
//     at a time with one rescale;
//   * the states merge exactly (§3.1/§4.1 with a common reference max):
//     across the groups of a warp by shuffles, across warps in shared memory;
//   * with one key range per head the CTA writes O and LSE; with several it
//     writes fp32 partials that decode_combine merges, one CTA per head.
#include "fa_decode.h"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

constexpr int kWarps = 8;
constexpr int kUnroll = 2;   // keys per lane per step; the next step's loads are issued before this step's math

template <int DR>
struct DecodeShape {
  static constexpr int kG = DR <= 64 ? 8 : (DR <= 128 ? 16 : 32);   // lanes per key
  static constexpr int kKpw = 32 / kG;                              // keys per warp load
};

template <bool F16>
__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = unpack2<F16>(w[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

// Folds state (mb, lb, accb) into (m, l, acc); both share the base-2 units.
__device__ __forceinline__ void merge_state(float& m, float& l, float (&acc)[8], float mb, float lb,
                                            const float (&accb)[8]) {
  const float M = fmaxf(m, mb);
  if (M == -INFINITY) return;   // neither has seen a key
  const float ca = ex2(m - M), cb = ex2(mb - M);
  l = l * ca + lb * cb;
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = acc[i] * ca + accb[i] * cb;
  m = M;
}

template <int DR, bool F16>
__global__ void __launch_bounds__(kWarps * 32, 4) decode_kernel(const __grid_constant__ DecodeArgs a) {
  using Sh = DecodeShape<DR>;
  constexpr int G = Sh::kG, KPW = Sh::kKpw;
  __shared__ float sm_m[kWarps], sm_l[kWarps];
  __shared__ __align__(16) float sm_acc[kWarps][DR];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane / G, gl = lane % G;
  const bool cols = gl * 8 < DR;   // d = 96: lanes 12-15 of a group hold no columns
  const int split = (int)blockIdx.x;
  const long long bh = blockIdx.y;
  const long long Nk = a.Nk;
  const long long kb = (long long)split * Nk / a.splits, ke = (long long)(split + 1) * Nk / a.splits;
  const uint16_t* kbase = static_cast<const uint16_t*>(a.k) + (size_t)bh * (size_t)Nk * DR + gl * 8;
  const uint16_t* vbase = static_cast<const uint16_t*>(a.v) + (size_t)bh * (size_t)Nk * DR + gl * 8;

  float qf[8];
  if (cols) {
    const uint4 qu = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.q) + (size_t)bh * DR + gl * 8);
    unpack8<F16>(qu, qf);
#pragma unroll
    for (int i = 0; i < 8; ++i) qf[i] *= a.scale_log2;   // scores in base-2 units
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) qf[i] = 0.f;
  }
  float m = -INFINITY, l = 0.f, acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;

  constexpr int kStep = kWarps * KPW * kUnroll;   // keys per CTA iteration
  // Loads of one step: kUnroll keys per lane group, 16 bytes of K and of V each.
  auto load = [&](long long base, uint4 (&ku)[kUnroll], uint4 (&vu)[kUnroll]) {
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const long long key = base + (long long)((u * kWarps + warp) * KPW + g);
      if (cols && key < ke) {
        ku[u] = __ldcs(reinterpret_cast<const uint4*>(kbase + key * DR));
        vu[u] = __ldcs(reinterpret_cast<const uint4*>(vbase + key * DR));
      } else {
        ku[u] = make_uint4(0u, 0u, 0u, 0u);
        vu[u] = ku[u];
      }
    }
  };
  uint4 ku[kUnroll], vu[kUnroll];
  load(kb, ku, vu);
  for (long long base = kb; base < ke; base += kStep) {
    // The next step's loads go out before this step's arithmetic, so a
    // lane always has loads in flight.
    uint4 kn[kUnroll], vn[kUnroll];
    load(base + kStep, kn, vn);
    float s[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const long long key = base + (long long)((u * kWarps + warp) * KPW + g);
      float kf[8];
      unpack8<F16>(ku[u], kf);
      float d0 = 0.f, d1 = 0.f;
#pragma unroll
      for (int i = 0; i < 8; i += 2) {
        d0 = fmaf(qf[i], kf[i], d0);
        d1 = fmaf(qf[i + 1], kf[i + 1], d1);
      }
      float dot = d0 + d1;
#pragma unroll
      for (int o = G / 2; o > 0; o >>= 1) dot += __shfl_xor_sync(kFull, dot, o);   // within the group
      s[u] = key < ke ? dot : -INFINITY;
    }
    float mx = m;
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) mx = fmaxf(mx, s[u]);
    // Reference for this step: the new max, or 0 while the group has seen no
    // key (so that no −∞ − (−∞) arises); the rescale of the old state is
    // exact either way.
    const float ref = mx == -INFINITY ? 0.f : mx;
    const float c = ex2(m - ref);
    l *= c;
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] *= c;
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const float p = ex2(s[u] - ref);
      l += p;
      float vf[8];
      unpack8<F16>(vu[u], vf);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = fmaf(p, vf[i], acc[i]);
    }
    m = mx;
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      ku[u] = kn[u];
      vu[u] = vn[u];
    }
  }

  // Groups of a warp, then warps.
#pragma unroll
  for (int o = G; o < 32; o <<= 1) {
    const float mb = __shfl_xor_sync(kFull, m, o), lb = __shfl_xor_sync(kFull, l, o);
    float accb[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) accb[i] = __shfl_xor_sync(kFull, acc[i], o);
    merge_state(m, l, acc, mb, lb, accb);
  }
  if (g == 0 && cols) {
#pragma unroll
    for (int i = 0; i < 8; ++i) sm_acc[warp][gl * 8 + i] = acc[i];
  }
  if (lane == 0) {
    sm_m[warp] = m;
    sm_l[warp] = l;
  }
  __syncthreads();
  if (warp != 0 || g != 0) return;
  float M = -INFINITY;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm_m[w]);
  float L = 0.f, out[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) out[i] = 0.f;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const float cw = sm_m[w] == -INFINITY ? 0.f : ex2(sm_m[w] - M);
    L += sm_l[w] * cw;
    if (cols) {
#pragma unroll
      for (int i = 0; i < 8; ++i) out[i] = fmaf(sm_acc[w][gl * 8 + i], cw, out[i]);
    }
  }
  // Every key range holds at least one key, so L > 0.
  const float inv = 1.0f / L;
  const float lse = (M + log2f(L)) * 0.69314718055994530942f;   // natural log of the scaled scores
  if (a.splits == 1) {
    if (cols) {
      uint4 pk;
      pk.x = pack2<F16>(out[0] * inv, out[1] * inv);
      pk.y = pack2<F16>(out[2] * inv, out[3] * inv);
      pk.z = pack2<F16>(out[4] * inv, out[5] * inv);
      pk.w = pack2<F16>(out[6] * inv, out[7] * inv);
      *reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.o) + (size_t)bh * DR + gl * 8) = pk;
    }
    if (gl == 0) a.lse[bh] = lse;
  } else {
    const size_t prow = (size_t)bh * (size_t)a.splits + (size_t)split;
    if (cols) {
      float4* dst = reinterpret_cast<float4*>(a.opart + prow * DR + gl * 8);
      dst[0] = make_float4(out[0] * inv, out[1] * inv, out[2] * inv, out[3] * inv);
      dst[1] = make_float4(out[4] * inv, out[5] * inv, out[6] * inv, out[7] * inv);
    }
    if (gl == 0) a.lpart[prow] = lse;
  }
}

// Merge of one head's key-range partials (2.Online Softmax §3.1/§4.1 in
// log-sum-exp form: LSE = ln Σ_k e^{LSE_k}, O = Σ_k e^{LSE_k − LSE} O_k).
// One CTA per head: every warp forms LSE (lanes over the ranges), warp w
// accumulates ranges w, w + 8, … over all head dims, shared memory sums the
// warps.  With few heads and many ranges this keeps the merge off the
// critical path.
template <int DR, bool F16>
__global__ void __launch_bounds__(kWarps * 32) decode_combine_kernel(const __grid_constant__ DecodeArgs a) {
  constexpr int V = (DR + 31) / 32;   // head dims per lane (the last lanes may hold fewer at d = 96)
  __shared__ __align__(16) float sm[kWarps][DR];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t bh = blockIdx.x;
  const int S = a.splits;
  const float* lp = a.lpart + bh * (size_t)S;
  const float* op = a.opart + bh * (size_t)S * DR;
  float mx = -INFINITY;
  for (int k = lane; k < S; k += 32) mx = fmaxf(mx, lp[k]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
  float sum = 0.f;
  for (int k = lane; k < S; k += 32) sum += expf(lp[k] - mx);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(kFull, sum, o);
  const float total = mx + logf(sum);
  float acc[V];
#pragma unroll
  for (int v = 0; v < V; ++v) acc[v] = 0.f;
  for (int k = warp; k < S; k += kWarps) {
    const float w = expf(lp[k] - total);
#pragma unroll
    for (int v = 0; v < V; ++v) {
      const int c = lane + 32 * v;
      if (c < DR) acc[v] = fmaf(w, op[(size_t)k * DR + c], acc[v]);
    }
  }
#pragma unroll
  for (int v = 0; v < V; ++v) {
    const int c = lane + 32 * v;
    if (c < DR) sm[warp][c] = acc[v];
  }
  __syncthreads();
  for (int c = threadIdx.x; c < DR; c += kWarps * 32) {
    float o = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) o += sm[w][c];
    static_cast<uint16_t*>(a.o)[bh * DR + c] = (uint16_t)(pack2<F16>(o, 0.f) & 0xFFFFu);
  }
  if (threadIdx.x == 0) a.lse[bh] = total;
}

template <int DR, bool F16>
cudaError_t launch_dr(const DecodeArgs& a, cudaStream_t s) {
  decode_kernel<DR, F16><<<dim3((unsigned)a.splits, (unsigned)a.BH), kWarps * 32, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || a.splits == 1) return e;
  decode_combine_kernel<DR, F16><<<(unsigned)a.BH, kWarps * 32, 0, s>>>(a);
  return cudaGetLastError();
}

template <bool F16>
cudaError_t dispatch(const DecodeArgs& a, cudaStream_t s) {
  switch (a.d) {
    case 64: return launch_dr<64, F16>(a, s);
    case 96: return launch_dr<96, F16>(a, s);
    case 128: return launch_dr<128, F16>(a, s);
    case 256: return launch_dr<256, F16>(a, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

int decode_splits(int heads, int num_sms, int Nk) {
  if (heads <= 0 || Nk <= 0) return 1;
  // About sixteen CTAs per SM (four resident at a time, so the last of
  // several waves is short), at least 256 keys per range, at most 128 ranges.
  const int sms = num_sms > 0 ? num_sms : 1;
  int s = (16 * sms + heads - 1) / heads;
  const int by_keys = Nk / 256 > 0 ? Nk / 256 : 1;
  if (s > by_keys) s = by_keys;
  if (s > 128) s = 128;
  return s < 1 ? 1 : s;
}

cudaError_t launch_fwd_decode(const DecodeArgs& a, cudaStream_t s) {
  if (a.BH <= 0 || a.BH > 65535 || a.splits < 1 || a.splits > a.Nk) return cudaErrorInvalidValue;
  if (a.splits > 1 && (a.opart == nullptr || a.lpart == nullptr)) return cudaErrorInvalidValue;
  return a.f16 ? dispatch<true>(a, s) : dispatch<false>(a, s);
}

}  // namespace fa
