// fa_bwd_bf16.cu — tiled attention backward on the sm_103a tensor cores.
//
// What it computes: "Flash Attention" tutorial, 4.附录A "反向传播的公式推导"
// 五-六 (and 3.Recomputation 四): with only O and LSE kept from the forward,
// each tile of P is rebuilt as exp(S - LSE); D = rowsum(dO ⊙ O) replaces
// rowsum(dP ⊙ P); then dV += Pᵀ dO, dP = dO Vᵀ, dS = P ⊙ (dP - D),
// dK += dSᵀ Q and dQ += dS K.  The scale of the scores multiplies dQ and dK
// (coreui.cn page "FlashAttention 反向传播", dQ = dS K / sqrt(d_k)).
//
// Loop order differs from the page's pseudocode (query tiles outermost): here
// a CTA owns one 128-row K/V tile and walks the query tiles, so dK and dV
// accumulate in tensor memory and only dQ is shared between CTAs (fp32
// reductions into a workspace accumulator).  The sums are the same.
//
// Everything is computed transposed relative to the page (rows = keys):
//   Sᵀ = K Qᵀ, dPᵀ = V dOᵀ   (tcgen05, M = 128 keys, N = BM queries)
//   Pᵀ = exp2(Sᵀ·scale·log2e - LSE2), dSᵀ = Pᵀ ⊙ (dPᵀ - D)   (one thread per key row)
//   dV += Pᵀ dO, dK += dSᵀ Q   (A = Pᵀ / dSᵀ from shared memory, M = 128 keys)
//   d = 128: dQᵀ = Kᵀ dSᵀ (M = 128 head dims, N = 64 queries)
//   d = 64:  dQ  = dS K   (M = 128 queries, N = 64 head dims)
//
// CTA: 14 warps.  Warps 0-7 compute Pᵀ/dSᵀ (warp w owns key rows 32(w%4).. and
// half w/4 of the query columns), warps 8-11 drain dQ from tensor memory into
// the fp32 accumulator with vector reductions, warp 12 issues TMA, warp 13
// issues the MMAs and owns tensor memory.
#include "fa_kernels.h"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

constexpr int kBN = 128;            // keys per CTA
constexpr int kThreads = 448;
constexpr int kComputeWarps = 8;
constexpr int kDrainWarp0 = 8;
constexpr int kTmaWarp = 12;
constexpr int kMmaWarp = 13;
constexpr int kBox = 16384;         // 128 rows × 128 bytes

template <int D>
struct BwdCfg {
  static constexpr int BM = D == 128 ? 64 : 128;  // queries per step
  static constexpr int NDP = D == 128 ? 2 : 1;    // dPᵀ buffers in tensor memory
  // shared memory
  static constexpr int kKV = kBN * D * 2;          // one K (or V) tile
  static constexpr int kQT = BM * D * 2;           // one Q (or dO) tile
  static constexpr int kQBox = BM * 128;           // one 64-column box of a Q tile
  static constexpr int kPT = kBN * BM * 2;         // one Pᵀ (or dSᵀ) tile
  static constexpr int kK = 0;
  static constexpr int kV = kK + kKV;
  static constexpr int kQ = kV + kKV;              // 2 stages
  static constexpr int kDO = kQ + 2 * kQT;         // 2 stages
  static constexpr int kP = kDO + 2 * kQT;         // 2 buffers
  static constexpr int kDS = kP + 2 * kPT;         // 2 buffers
  static constexpr int kLSE = kDS + 2 * kPT;       // 2 stages of BM floats
  static constexpr int kDV = kLSE + 2 * BM * 4;    // 2 stages of BM floats
  static constexpr int kBar = kDV + 2 * BM * 4;
  static constexpr int kBytes = kBar + 256;
  // tensor memory columns
  static constexpr uint32_t kColDV = 0;
  static constexpr uint32_t kColDK = D;
  static constexpr uint32_t col_s(int b) { return 2 * D + b * BM; }
  static constexpr uint32_t col_dp(int b) { return 2 * D + 2 * BM + (b % NDP) * BM; }
};

enum BwdBar : int {
  kKVFull = 0,
  kQFull = 1,       // +stage
  kQEmpty = 3,      // +stage
  kSFull = 5,       // +buffer
  kDPFull = 7,      // +buffer
  kTmUsed = 9,      // +buffer: compute threads have read Sᵀ and dPᵀ
  kPdsFull = 11,    // +buffer
  kPdsEmpty = 13,   // +buffer
  kDqFull = 15,     // +buffer
  kDqDrained = 17,  // +buffer
  kDKVFull = 19,
  kMmaDone = 20,
  kNumBars = 21,
};

__device__ __forceinline__ uint32_t site(int s) { return 0x0200u | (uint32_t)s; }

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1) fa_bwd_bf16_kernel(const __grid_constant__ BwdArgs a) {
  using C = BwdCfg<D>;
  constexpr int BM = C::BM;
  // Dynamic shared memory starts on a 1024-byte boundary (no static shared
  // memory is declared); 128-byte swizzled tiles need that alignment.
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t sbase = smem_u32(smem_raw);
  uint8_t* sgen = smem_raw;
  if (sbase & 1023u) {
    if (threadIdx.x == 0) atomicCAS(a.fault, 0u, site(0));
    return;
  }
  const uint32_t bars = sbase + C::kBar;
  auto bar = [&](int i) -> uint32_t { return bars + 8u * (uint32_t)i; };
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sgen + C::kBar + 8 * kNumBars);
  int* abort_flag = reinterpret_cast<int*>(sgen + C::kBar + 8 * kNumBars + 4);
  const WaitCtx wc{abort_flag, a.fault};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int N = a.N;
  const int bh = blockIdx.x;
  const int jt = blockIdx.y;                 // K/V tile; small jt = most work when causal
  const int kv0 = jt * kBN;
  const int row0 = bh * N;
  const int i0 = CAUSAL ? kv0 / BM : 0;      // first query tile with a visible query
  const int n = N / BM - i0;                 // query tiles visited

  if (threadIdx.x == 0) {
    mbar_init(bar(kKVFull), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(kQFull + s), 1);
      mbar_init(bar(kQEmpty + s), 1 + 32 * kComputeWarps);
      mbar_init(bar(kSFull + s), 1);
      mbar_init(bar(kDPFull + s), 1);
      mbar_init(bar(kTmUsed + s), 32 * kComputeWarps);
      mbar_init(bar(kPdsFull + s), 32 * kComputeWarps);
      mbar_init(bar(kPdsEmpty + s), 1);
      mbar_init(bar(kDqFull + s), 1);
      mbar_init(bar(kDqDrained + s), 128);
    }
    mbar_init(bar(kDKVFull), 1);
    mbar_init(bar(kMmaDone), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_holder), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp < kComputeWarps) {
    // ------------------------------------------------------------ Pᵀ, dSᵀ
    const int g = warp & 3;
    const int h = warp >> 2;                       // query-column half
    const int r = g * 32 + lane;                   // key row within the tile = TMEM lane
    const int kv = kv0 + r;
    const uint32_t lane_off = (uint32_t)(g * 32) << 16;
    constexpr int CW = BM / 2;                     // query columns per thread
    const float sl2 = a.scale_log2;
    bool ok = true;
    for (int i = 0; i < n; ++i) {
      const int b = i & 1;
      const uint32_t par = (uint32_t)((i >> 1) & 1);
      const int q0 = (i0 + i) * BM;
      ok = mbar_wait(bar(kSFull + b), par, wc, site(1)) && mbar_wait(bar(kDPFull + b), par, wc, site(2)) &&
           mbar_wait(bar(kQFull + b), par, wc, site(3)) &&
           (i < 2 || mbar_wait(bar(kPdsEmpty + b), (uint32_t)(((i >> 1) - 1) & 1), wc, site(4)));
      ok = __all_sync(kFull, ok);
      if (!ok) break;
      tc_fence_after();
      const float* lse2 = reinterpret_cast<const float*>(sgen + C::kLSE + b * BM * 4);
      const float* dvec = reinterpret_cast<const float*>(sgen + C::kDV + b * BM * 4);
      const bool masked = CAUSAL && q0 < kv0 + kBN;   // tile straddles the diagonal
      const uint32_t p_tile = sbase + C::kP + b * C::kPT;
      const uint32_t ds_tile = sbase + C::kDS + b * C::kPT;
#pragma unroll
      for (int ch = 0; ch < CW / 32; ++ch) {
        const int c0 = h * CW + ch * 32;           // first query column of this chunk
        uint32_t s[32], dp[32];
        tmem_ld_x32(tmem + lane_off + C::col_s(b) + (uint32_t)c0, s);
        tmem_ld_x32(tmem + lane_off + C::col_dp(b) + (uint32_t)c0, dp);
        uint32_t pk[16], dk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          float p0 = ex2(fmaf(u2f(s[e]), sl2, -lse2[c0 + e]));
          float p1 = ex2(fmaf(u2f(s[e + 1]), sl2, -lse2[c0 + e + 1]));
          if (masked) {
            // key kv is visible to query q iff kv ≤ q
            if (kv > q0 + c0 + e) p0 = 0.f;
            if (kv > q0 + c0 + e + 1) p1 = 0.f;
          }
          const float d0 = p0 * (u2f(dp[e]) - dvec[c0 + e]);
          const float d1 = p1 * (u2f(dp[e + 1]) - dvec[c0 + e + 1]);
          pk[e >> 1] = pack_bf16x2(p0, p1);
          dk[e >> 1] = pack_bf16x2(d0, d1);
        }
        // 32 query columns = 64 bytes = four 16-byte chunks of this key row,
        // placed with the 128-byte swizzle (chunk index XOR row % 8).
        const int box = c0 >> 6;
        const uint32_t row_addr = (uint32_t)(box * kBox + r * 128);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int chunk = ((c0 & 63) >> 3) + u;
          const uint32_t off = row_addr + (uint32_t)(((chunk ^ (r & 7)) & 7) * 16);
          st_shared_v4(p_tile + off, pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
          st_shared_v4(ds_tile + off, dk[4 * u], dk[4 * u + 1], dk[4 * u + 2], dk[4 * u + 3]);
        }
      }
      tc_fence_before();
      mbar_arrive(bar(kTmUsed + b));
      fence_proxy_async_smem();
      mbar_arrive(bar(kPdsFull + b));
      mbar_arrive(bar(kQEmpty + b));
    }
    // ------------------------------------------------------------ dK, dV epilogue
    if (ok) {
      ok = mbar_wait(bar(kDKVFull), 0, wc, site(5));
      ok = __all_sync(kFull, ok);
    }
    if (ok) {
      tc_fence_after();
      const uint32_t col = h == 0 ? C::kColDV : C::kColDK;
      const float mul = h == 0 ? 1.0f : a.scale;
      __nv_bfloat16* dst = (h == 0 ? a.dv : a.dk) + ((size_t)row0 + (size_t)kv) * D;
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t v[32];
        tmem_ld_x32(tmem + lane_off + col + 32 * cc, v);
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) pk[e] = pack_bf16x2(u2f(v[2 * e]) * mul, u2f(v[2 * e + 1]) * mul);
#pragma unroll
        for (int u = 0; u < 4; ++u)
          st_global_v4(dst + 32 * cc + 8 * u, pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
      }
    }
  } else if (warp < kTmaWarp) {
    // ------------------------------------------------------------ dQ drain
    const int g = warp - kDrainWarp0;
    const uint32_t lane_off = (uint32_t)(g * 32) << 16;
    for (int i = 0; i < n; ++i) {
      const int b = i & 1;
      bool ok = mbar_wait(bar(kDqFull + b), (uint32_t)((i >> 1) & 1), wc, site(6));
      ok = __all_sync(kFull, ok);
      if (!ok) break;
      tc_fence_after();
      uint32_t v[64];
      tmem_ld_x64(tmem + lane_off + C::col_s(b), v);
      tc_fence_before();
      mbar_arrive(bar(kDqDrained + b));
      const int q0 = (i0 + i) * BM;
      if constexpr (D == 128) {
        // lane = head dim, columns = 64 queries
        float* base = a.dqacc + ((size_t)row0 + (size_t)q0) * D + (size_t)(g * 32 + lane);
#pragma unroll
        for (int c = 0; c < 64; ++c) red_add_f32(base + (size_t)c * D, u2f(v[c]));
      } else {
        // lane = query row, columns = 64 head dims
        float* base = a.dqacc + ((size_t)row0 + (size_t)q0 + (size_t)(g * 32 + lane)) * D;
#pragma unroll
        for (int c = 0; c < 64; c += 4) red_add_v4_f32(base + c, u2f(v[c]), u2f(v[c + 1]), u2f(v[c + 2]), u2f(v[c + 3]));
      }
    }
  } else if (warp == kTmaWarp) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tmap(&a.tm_q);
      prefetch_tmap(&a.tm_k);
      prefetch_tmap(&a.tm_v);
      prefetch_tmap(&a.tm_do);
      mbar_arrive_expect_tx(bar(kKVFull), 2u * C::kKV);
      for (int bx = 0; bx < D / 64; ++bx) {
        tma_load_2d(sbase + C::kK + bx * kBox, &a.tm_k, bar(kKVFull), 64 * bx, row0 + kv0);
        tma_load_2d(sbase + C::kV + bx * kBox, &a.tm_v, bar(kKVFull), 64 * bx, row0 + kv0);
      }
      int issued[2] = {0, 0};
      for (int i = 0; i < n; ++i) {
        const int s = i & 1;
        if (i >= 2 && !mbar_wait(bar(kQEmpty + s), (uint32_t)(((i >> 1) - 1) & 1), wc, site(7))) break;
        const int q0 = (i0 + i) * BM;
        mbar_arrive_expect_tx(bar(kQFull + s), 2u * C::kQT + 2u * BM * 4);
        for (int bx = 0; bx < D / 64; ++bx) {
          tma_load_2d(sbase + C::kQ + s * C::kQT + bx * C::kQBox, &a.tm_q, bar(kQFull + s), 64 * bx, row0 + q0);
          tma_load_2d(sbase + C::kDO + s * C::kQT + bx * C::kQBox, &a.tm_do, bar(kQFull + s), 64 * bx,
                      row0 + q0);
        }
        bulk_load(sbase + C::kLSE + s * BM * 4, a.lse2 + row0 + q0, BM * 4, bar(kQFull + s));
        bulk_load(sbase + C::kDV + s * BM * 4, a.dvec + row0 + q0, BM * 4, bar(kQFull + s));
        ++issued[s];
      }
      mbar_wait_drain(bar(kKVFull), 0, wc, site(8));
      for (int s = 0; s < 2; ++s)
        if (issued[s] > 0) mbar_wait_drain(bar(kQFull + s), (uint32_t)((issued[s] - 1) & 1), wc, site(8));
    }
  } else {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16(128, BM, false, false);  // Sᵀ = K Qᵀ, dPᵀ = V dOᵀ
      constexpr uint32_t kIdKV = idesc_bf16(128, D, false, true);   // dV += Pᵀ dO, dK += dSᵀ Q
      // dQᵀ = Kᵀ dSᵀ (d = 128) or dQ = dS K (d = 64): both operands MN-major
      constexpr uint32_t kIdQ = idesc_bf16(128, 64, true, true);
      bool ok = mbar_wait(bar(kKVFull), 0, wc, site(9));
      auto issue_sdp = [&](int i) -> bool {
        const int b = i & 1;
        if (!mbar_wait(bar(kQFull + b), (uint32_t)((i >> 1) & 1), wc, site(10))) return false;
        if (i >= 2 && !mbar_wait(bar(kDqDrained + b), (uint32_t)(((i >> 1) - 1) & 1), wc, site(11))) return false;
        tc_fence_after();
        const uint32_t qb = sbase + C::kQ + b * C::kQT;
        const uint32_t ob = sbase + C::kDO + b * C::kQT;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t ok_ = (uint32_t)((ks >> 2) * kBox + (ks & 3) * 32);
          const uint32_t oq = (uint32_t)((ks >> 2) * C::kQBox + (ks & 3) * 32);
          mma_ss(tmem + C::col_s(b), sdesc_sw128(sbase + C::kK + ok_, 16, 1024), sdesc_sw128(qb + oq, 16, 1024),
                 kIdS, ks > 0 ? 1u : 0u);
        }
        tc_commit(bar(kSFull + b));
        // The dPᵀ buffer must have been read by the compute threads.
        if (C::NDP == 2) {
          if (i >= 2 && !mbar_wait(bar(kTmUsed + b), (uint32_t)(((i >> 1) - 1) & 1), wc, site(12))) return false;
        } else {
          if (i >= 1 && !mbar_wait(bar(kTmUsed + ((i - 1) & 1)), (uint32_t)(((i - 1) >> 1) & 1), wc, site(12)))
            return false;
        }
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t ok_ = (uint32_t)((ks >> 2) * kBox + (ks & 3) * 32);
          const uint32_t oq = (uint32_t)((ks >> 2) * C::kQBox + (ks & 3) * 32);
          mma_ss(tmem + C::col_dp(b), sdesc_sw128(sbase + C::kV + ok_, 16, 1024), sdesc_sw128(ob + oq, 16, 1024),
                 kIdS, ks > 0 ? 1u : 0u);
        }
        tc_commit(bar(kDPFull + b));
        return true;
      };
      if (ok && n > 0) ok = issue_sdp(0);
      if (ok && n > 1) ok = issue_sdp(1);
      for (int i = 0; ok && i < n; ++i) {
        const int b = i & 1;
        if (!mbar_wait(bar(kPdsFull + b), (uint32_t)((i >> 1) & 1), wc, site(13))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t pt = sbase + C::kP + b * C::kPT;
        const uint32_t dst = sbase + C::kDS + b * C::kPT;
        const uint32_t qb = sbase + C::kQ + b * C::kQT;
        const uint32_t ob = sbase + C::kDO + b * C::kQT;
        // dQ first, so that its drain overlaps the dV / dK products.
#pragma unroll
        for (int ks = 0; ks < kBN / 16; ++ks) {
          const uint32_t kst = (uint32_t)(ks * 2048);   // 16 key rows
          uint64_t da, db;
          if constexpr (D == 128) {
            da = sdesc_sw128(sbase + C::kK + kst, kBox, 1024);   // Kᵀ: M = head dims (two 64-wide blocks)
            db = sdesc_sw128(dst + kst, kBox, 1024);             // dSᵀ: N = 64 queries
          } else {
            da = sdesc_sw128(dst + kst, kBox, 1024);             // dS: M = 128 queries (two 64-wide blocks)
            db = sdesc_sw128(sbase + C::kK + kst, kBox, 1024);   // K: N = 64 head dims
          }
          mma_ss(tmem + C::col_s(b), da, db, kIdQ, ks > 0 ? 1u : 0u);
        }
        tc_commit(bar(kDqFull + b));
#pragma unroll
        for (int ks = 0; ks < BM / 16; ++ks) {
          const uint32_t oa = (uint32_t)((ks >> 2) * kBox + (ks & 3) * 32);   // Pᵀ / dSᵀ, K-major over queries
          const uint32_t ob2 = (uint32_t)(ks * 2048);                         // dO / Q, MN-major, 16 query rows
          mma_ss(tmem + C::kColDV, sdesc_sw128(pt + oa, 16, 1024), sdesc_sw128(ob + ob2, C::kQBox, 1024), kIdKV,
                 (i > 0 || ks > 0) ? 1u : 0u);
        }
#pragma unroll
        for (int ks = 0; ks < BM / 16; ++ks) {
          const uint32_t oa = (uint32_t)((ks >> 2) * kBox + (ks & 3) * 32);
          const uint32_t ob2 = (uint32_t)(ks * 2048);
          mma_ss(tmem + C::kColDK, sdesc_sw128(dst + oa, 16, 1024), sdesc_sw128(qb + ob2, C::kQBox, 1024), kIdKV,
                 (i > 0 || ks > 0) ? 1u : 0u);
        }
        tc_commit(bar(kQEmpty + b));
        tc_commit(bar(kPdsEmpty + b));
        if (i + 2 < n) ok = issue_sdp(i + 2);
      }
      if (ok) tc_commit(bar(kDKVFull));
      tc_commit(bar(kMmaDone));
      mbar_wait_drain(bar(kMmaDone), 0, wc, site(14));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool CAUSAL>
cudaError_t launch_impl(const BwdArgs& a, cudaStream_t s) {
  auto kern = fa_bwd_bf16_kernel<D, CAUSAL>;
  const size_t smem = BwdCfg<D>::kBytes;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)(a.B * a.H), (unsigned)(a.N / kBN));
  kern<<<grid, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ pre-pass and dQ finish

// One group of D/8 threads per row; each thread reads 8 bf16 of O and of dO
// (16 bytes each), so a warp covers 32·8 contiguous elements.
template <int D>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const __nv_bfloat16* __restrict__ o,
                                                       const __nv_bfloat16* __restrict__ dO,
                                                       const float* __restrict__ lse, float* __restrict__ dvec,
                                                       float* __restrict__ lse2, float* __restrict__ dqacc,
                                                       long long rows) {
  constexpr int G = D / 8;   // threads per row
  const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long row = tid / G;
  const int part = (int)(tid % G);
  float acc = 0.f;
  if (row < rows) {
    const uint4 ov = *reinterpret_cast<const uint4*>(o + row * D + part * 8);
    const uint4 gv = *reinterpret_cast<const uint4*>(dO + row * D + part * 8);
    const __nv_bfloat162* op = reinterpret_cast<const __nv_bfloat162*>(&ov);
    const __nv_bfloat162* gp = reinterpret_cast<const __nv_bfloat162*>(&gv);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 a2 = __bfloat1622float2(op[i]);
      const float2 b2 = __bfloat1622float2(gp[i]);
      acc = fmaf(a2.x, b2.x, acc);
      acc = fmaf(a2.y, b2.y, acc);
    }
    float4* z = reinterpret_cast<float4*>(dqacc + row * D + part * 8);
    z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int off = G / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(kFull, acc, off);
  if (row < rows && part == 0) {
    dvec[row] = acc;
    lse2[row] = lse[row] * 1.4426950408889634074f;
  }
}

__global__ void __launch_bounds__(256) dq_finish_kernel(const float* __restrict__ acc, __nv_bfloat16* __restrict__ dq,
                                                        long long n8, float scale) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n8) return;
  const float4 a0 = reinterpret_cast<const float4*>(acc)[2 * i];
  const float4 a1 = reinterpret_cast<const float4*>(acc)[2 * i + 1];
  uint4 out;
  out.x = pack_bf16x2(a0.x * scale, a0.y * scale);
  out.y = pack_bf16x2(a0.z * scale, a0.w * scale);
  out.z = pack_bf16x2(a1.x * scale, a1.y * scale);
  out.w = pack_bf16x2(a1.z * scale, a1.w * scale);
  reinterpret_cast<uint4*>(dq)[i] = out;
}

}  // namespace

int bwd_bf16_block_m(int d) { return d == 128 ? BwdCfg<128>::BM : BwdCfg<64>::BM; }

size_t bwd_bf16_smem_bytes(int d) {
  return d == 64 ? BwdCfg<64>::kBytes : BwdCfg<128>::kBytes;
}

cudaError_t launch_bwd_bf16(const BwdArgs& a, cudaStream_t s) {
  if (a.d == 128) return a.causal ? launch_impl<128, true>(a, s) : launch_impl<128, false>(a, s);
  if (a.d == 64) return a.causal ? launch_impl<64, true>(a, s) : launch_impl<64, false>(a, s);
  return cudaErrorInvalidValue;
}

cudaError_t launch_bwd_prep_bf16(const __nv_bfloat16* o, const __nv_bfloat16* dO, const float* lse, float* dvec,
                                 float* lse2, float* dqacc, long long rows, int d, cudaStream_t s) {
  const long long threads = rows * (d / 8);
  const unsigned blocks = (unsigned)((threads + 255) / 256);
  if (d == 128)
    bwd_prep_kernel<128><<<blocks, 256, 0, s>>>(o, dO, lse, dvec, lse2, dqacc, rows);
  else if (d == 64)
    bwd_prep_kernel<64><<<blocks, 256, 0, s>>>(o, dO, lse, dvec, lse2, dqacc, rows);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

cudaError_t launch_dq_finish_bf16(const float* dqacc, __nv_bfloat16* dq, long long elems, float scale,
                                  cudaStream_t s) {
  const long long n8 = elems / 8;
  const unsigned blocks = (unsigned)((n8 + 255) / 256);
  dq_finish_kernel<<<blocks, 256, 0, s>>>(dqacc, dq, n8, scale);
  return cudaGetLastError();
}

}  // namespace fa
