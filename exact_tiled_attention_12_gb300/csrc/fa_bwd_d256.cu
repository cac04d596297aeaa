// fa_bwd_d256.cu — tiled attention backward for head dimension 256 on the
// sm_103a tensor cores.
//
// What it computes is what fa_bwd_bf16.cu computes ("Flash Attention"
// tutorial, 4.附录A "反向传播的公式推导" 五-六 and 3.Recomputation 四: P
// rebuilt per tile as exp(S − LSE), D = rowsum(dO ⊙ O), dV = Pᵀ dO,
// dS = P ⊙ (dP − D), dK = scale·dSᵀ Q, dQ = scale·dS K with the scale of the
// coreui.cn page "FlashAttention 反向传播"); only the split of the work differs.
//
// At d = 256 the fp32 dK and dV accumulators of a 128-key tile would fill all
// 512 tensor-memory columns, so the work is split in two kernels, neither of
// which needs atomics:
//
//  * dkdv: a CTA owns 64 keys and walks the 128-row query tiles.  Rows of S,
//    dP (tensor memory lanes) are queries, so every product keeps M = 128:
//      S  = Q K_jᵀ, dP = dO V_jᵀ            (N = 64 keys, K = 256)
//      dVᵀ_h += dO_hᵀ P, dKᵀ_h += Q_hᵀ dS   (M = 128 head dims of half h, N = 64)
//    Tensor memory: S [0, 64), dP [64, 128), dVᵀ [128, 256), dKᵀ [256, 384).
//    P and dS go to shared memory ([query][key], 128-byte swizzle) as the B
//    operands.  Q and dO stream in boxes of 64 head dims × 128 rows, two
//    boxes (one half of the head dims) per barrier: a half is reloaded for
//    the next query tile as soon as the products that read it have completed.
//
//  * dq: a CTA owns 128 queries and walks 64-key tiles, recomputing S and dP:
//      S_b = Q K_jᵀ, dP_b = dO V_jᵀ into buffer b = j mod 2
//      dQ += dS K_j                        (A = dS from tensor memory, N = 256)
//    Tensor memory: S_b [64b, 64b + 64), dP_b [128 + 64b, ...), dQ [256, 512);
//    dS (16-bit) is written over the dP columns its thread read.  The MMA
//    order dQ_j, S_{j+1}, dP_{j+2} overlaps the elementwise work of tile
//    j + 1 with dP_{j+2}; K streams through a ring of two tiles (released
//    once dQ_j has read them, so K_{j+1} has had a whole step to load when
//    S_{j+1} wants it), V through one.  Each K or V tile lands on one barrier
//    and is released with one commit, not one per box: the MMA thread's waits
//    and commits sit on its issue path.  (On GB300, against dQ_j, dP_{j+2},
//    S_{j+2} with a wait and a commit per box: +1.8 % for the commits,
//    +1-2.5 % for the order, +3-4 % for the waits.)
//
// Both kernels: warps 0-7 do the elementwise work, thread (w, lane) owning
// query row 32(w mod 4) + lane and key columns 32⌊w/4⌋ .. +31 of a 64-key
// tile; warp 8 issues TMA, warp 9 the MMAs and owns tensor memory.  The
// pre-pass (fa_bwd_bf16.cu) supplies −LSE·log2 e and −D per query row.
#include "fa_kernels.h"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

constexpr int kD = 256;
constexpr int kBM = 128;          // queries per tile
constexpr int kBN = 64;           // keys per tile
constexpr int kThreads = 320;
constexpr int kTmaWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kQBox = 16384;      // 128 rows × 128 bytes (Q, dO)
constexpr int kKBox = 8192;       // 64 rows × 128 bytes (K, V)

// ------------------------------------------------------------------ shared helpers

// P = 2^(s·scale·log2e − LSE₂) for 32 key columns of one query row; columns
// with index > lim are masked to 0.
template <bool MASKED>
__device__ __forceinline__ void p_row32(const uint32_t (&s)[32], float sl2, float nlse, int lim, float (&p)[32]) {
#pragma unroll
  for (int k = 0; k < 32; ++k) {
    const float e = ex2(fmaf(u2f(s[k]), sl2, nlse));
    p[k] = (MASKED && k > lim) ? 0.f : e;
  }
}

// dS = P ⊙ (dP − D) for 32 columns (nd = −D), packed to the 16-bit type.
template <bool F16>
__device__ __forceinline__ void ds_row32(const float (&p)[32], const uint32_t (&dp)[32], float nd, uint32_t (&out)[16]) {
#pragma unroll
  for (int e = 0; e < 16; ++e)
    out[e] = pack2<F16>(p[2 * e] * (u2f(dp[2 * e]) + nd), p[2 * e + 1] * (u2f(dp[2 * e + 1]) + nd));
}

// Stores 32 packed 16-bit values (64 bytes) as chunks 4c .. 4c+3 of row r of
// a [rows][64] tile with 128-byte rows and the 128-byte swizzle.
__device__ __forceinline__ void st_row_sw128(uint32_t tile, int r, int c, const uint32_t (&v)[16]) {
  const uint32_t row = tile + (uint32_t)(r * 128);
#pragma unroll
  for (int u = 0; u < 4; ++u)
    st_shared_v4(row + (uint32_t)((((4 * c + u) ^ (r & 7)) & 7) * 16), v[4 * u], v[4 * u + 1], v[4 * u + 2],
                 v[4 * u + 3]);
}

// ================================================================== dK, dV

namespace kv {
constexpr int kK = 0;                         // 4 boxes of 64 keys
constexpr int kV = kK + 4 * kKBox;
constexpr int kQ = kV + 4 * kKBox;            // 4 boxes of 128 queries
constexpr int kDO = kQ + 4 * kQBox;
constexpr int kP = kDO + 4 * kQBox;           // [128 queries][64 keys] 16-bit
constexpr int kDS = kP + kQBox;
constexpr int kLSE = kDS + kQBox;             // 128 floats
constexpr int kDV = kLSE + kBM * 4;           // 128 floats
constexpr int kBar = kDV + kBM * 4;
constexpr int kBytes = kBar + 256;
static_assert(kBytes <= 232448, "shared memory exceeds the 227 KB a CTA may use");

enum Bar : int {
  kKVFull = 0,
  // Q and dO land and are released per half of the head dims (boxes 0-1,
  // boxes 2-3): the MMA thread's waits and commits sit on its issue path (one
  // per box measured 5 % slower on GB300).
  kQFull = 1,        // + half (half 0 also carries −LSE₂ and −D)
  kQEmpty = 3,       // + half
  kDOFull = 5,       // + half
  kDOEmpty = 7,      // + half
  kSFull = 9,
  kDPFull = 10,
  kPdsFull = 11,
  kDKVFull = 12,
  kMmaDone = 13,
  kNumBars = 14,
};
static_assert(8 * kNumBars + 8 <= 256, "barrier block too small");

constexpr uint32_t kColS = 0, kColDP = 64, kColDV = 128, kColDK = 256;

__device__ __forceinline__ uint32_t site(int s) { return 0x0400u | (uint32_t)s; }
}  // namespace kv

template <bool CAUSAL, bool RAGGED, bool F16>
__global__ void __launch_bounds__(kThreads, 1) fa_bwd_d256_dkdv_kernel(const __grid_constant__ BwdArgs a) {
  using namespace kv;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t sbase = smem_u32(smem_raw);
  uint8_t* sgen = smem_raw;
  if (sbase & 1023u) {
    if (threadIdx.x == 0) atomicCAS(a.fault, 0u, site(0));
    return;
  }
  const uint32_t bars = sbase + kBar;
  auto bar = [&](int i) -> uint32_t { return bars + 8u * (uint32_t)i; };
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sgen + kBar + 8 * kNumBars);
  int* abort_flag = reinterpret_cast<int*>(sgen + kBar + 8 * kNumBars + 4);
  const WaitCtx wc{abort_flag, a.fault};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int Nq = a.Nq, Nk = a.Nk;
  const int off = Nk - Nq;                   // causal: query i sees keys j ≤ i + off
  // Non-causal: head-major grid (key tile fastest); causal: batch·head
  // fastest so the tiles with the most query tiles (small jt) start first.
  const int jt = CAUSAL ? (int)blockIdx.y : (int)blockIdx.x;
  const int bh = CAUSAL ? (int)blockIdx.x : (int)blockIdx.y;
  const int kv0 = jt * kBN;
  const int n_tiles = (Nq + kBM - 1) / kBM;  // query tiles per head (the last may be ragged)
  const int wrow0 = bh * n_tiles * kBM;      // first workspace row of this head (whole tiles per head)
  // First query tile with a query that sees key kv0: q + off ≥ kv0.
  const int i0 = CAUSAL ? (kv0 > off ? (kv0 - off) / kBM : 0) : 0;
  const int n = n_tiles - i0;
  // A debug build checks each box's destination and coordinates first (K and V
  // boxes are 64 rows, Q and dO boxes 128) and, if a check fails, completes its
  // bytes on the barrier without copying; bulk copies likewise.
  auto load_rows = [&](uint32_t dst, const CUtensorMap* map, uint32_t bar_addr, int x, int pos, int nrows) {
    const bool kv_map = map == &a.tm_k || map == &a.tm_v;
    const uint32_t box = kv_map ? (uint32_t)kKBox : (uint32_t)kQBox;
    bool chk = dcheck(smem_ok(dst - sbase, box, (uint32_t)kBar, 1024), wc, kChkSmem, 48) &&
               dcheck(tma_x_ok(x, 64, kD), wc, kChkTmaX, 48);
    if constexpr (RAGGED)
      chk = chk && dcheck(tma_head_ok(pos, nrows, bh, a.B * a.H), wc, kChkTmaRows, 48);
    else
      chk = chk && dcheck(tma_rows_ok((long long)bh * nrows + pos, (int)(box / 128), (long long)a.B * a.H * nrows),
                          wc, kChkTmaRows, 48);
    if (!chk) {
      mbar_complete_tx(bar_addr, box);
      return;
    }
    if constexpr (RAGGED)
      tma_load_3d(dst, map, bar_addr, x, pos, bh);
    else
      tma_load_2d(dst, map, bar_addr, x, bh * nrows + pos);
  };
  auto load_bulk = [&](uint32_t dst, const float* src, uint32_t bytes, uint32_t bar_addr) {
    if (!dcheck(smem_ok(dst - sbase, bytes, (uint32_t)kBar, 16) && bulk_ok(reinterpret_cast<uint64_t>(src), dst, bytes),
                wc, kChkBulk, 48 + 1)) {
      mbar_complete_tx(bar_addr, bytes);
      return;
    }
    bulk_load(dst, src, bytes, bar_addr);
  };

  if (threadIdx.x == 0) {
    mbar_init(bar(kKVFull), 1);
    for (int h = 0; h < 2; ++h) {
      mbar_init(bar(kQFull + h), 1);
      mbar_init(bar(kQEmpty + h), 1);
      mbar_init(bar(kDOFull + h), 1);
      mbar_init(bar(kDOEmpty + h), 1);
    }
    mbar_init(bar(kSFull), 1);
    mbar_init(bar(kDPFull), 1);
    mbar_init(bar(kPdsFull), 256);
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

  if (warp < 8) {
    // ------------------------------------------------------------ P, dS
    const int c = warp >> 2;                   // key columns [32c, 32c + 32)
    const int g = warp & 3;
    const int r = g * 32 + lane;               // query row within the tile = TMEM lane
    const uint32_t lane_off = (uint32_t)(g * 32) << 16;
    const float sl2 = a.scale_log2;
    // Keys past Nk (the last tile of a ragged head) read as zero rows: mask
    // them (non-causal; the causal mask already hides them).
    const int dead_lim = Nk - kv0 - 32 * c - 1;
    const bool ragged_cta = RAGGED && !CAUSAL && kv0 + kBN > Nk;
    const float* lse_s = reinterpret_cast<const float*>(sgen + kLSE);
    const float* dv_s = reinterpret_cast<const float*>(sgen + kDV);
    bool ok = true;
    for (int i = 0; i < n; ++i) {
      const uint32_t par = (uint32_t)(i & 1);
      const int q0 = (i0 + i) * kBM;
      ok = mbar_wait(bar(kSFull), par, wc, site(1)) && mbar_wait(bar(kQFull), par, wc, site(2));
      ok = __all_sync(kFull, ok);
      if (!ok) break;
      tc_fence_after();
      const float nlse = lse_s[r], nd = dv_s[r];
      // key kv0 + 32c + k is visible to query q0 + r iff k ≤ r + q0 + off − kv0 − 32c
      const int delta = q0 + off - kv0;
      float p[32];
      {
        uint32_t s[32];
        if (dcheck(tmem_ok(kColS + 32u * c, 32, 512), wc, kChkTmem, 50))
          tmem_ld_x32(tmem + lane_off + kColS + 32u * (uint32_t)c, s);
        if (CAUSAL && delta < kBN - 1)
          p_row32<true>(s, sl2, nlse, r + delta - 32 * c, p);
        else if (ragged_cta)
          p_row32<true>(s, sl2, nlse, dead_lim, p);
        else
          p_row32<false>(s, sl2, nlse, 0, p);
      }
      ok = mbar_wait(bar(kDPFull), par, wc, site(3));
      ok = __all_sync(kFull, ok);
      if (!ok) break;
      tc_fence_after();
      uint32_t dp[32];
      if (dcheck(tmem_ok(kColDP + 32u * c, 32, 512), wc, kChkTmem, 51))
        tmem_ld_x32(tmem + lane_off + kColDP + 32u * (uint32_t)c, dp);
      uint32_t pk[16], dk[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) pk[e] = pack2<F16>(p[2 * e], p[2 * e + 1]);
      ds_row32<F16>(p, dp, nd, dk);
      if (dcheck(smem_ok(kP + r * 128, 128, kBar, 128) && smem_ok(kDS + r * 128, 128, kBar, 128), wc, kChkSmem, 52)) {
        st_row_sw128(sbase + kP, r, c, pk);
        st_row_sw128(sbase + kDS, r, c, dk);
      }
      tc_fence_before();
      fence_proxy_async_smem();
      mbar_arrive(bar(kPdsFull));
    }
    // ------------------------------------------------------------ epilogue
    // Warps 0-3 store dV, warps 4-7 dK (scaled): the accumulators hold the
    // transposes, lane = head dim 32g + lane of half h, column = key.
    if (ok) {
      ok = mbar_wait(bar(kDKVFull), 0, wc, site(4));
      ok = __all_sync(kFull, ok);
    }
    if (ok) {
      tc_fence_after();
      const float mul = c == 0 ? 1.0f : a.scale;
      uint16_t* dst = static_cast<uint16_t*>(c == 0 ? a.dv : a.dk) + ((size_t)bh * (size_t)Nk + (size_t)kv0) * kD;
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        uint32_t v[64];
        if (!dcheck(tmem_ok((c == 0 ? kColDV : kColDK) + 64u * h, 64, 512), wc, kChkTmem, 53)) continue;
        tmem_ld_x64(tmem + lane_off + (c == 0 ? kColDV : kColDK) + 64u * (uint32_t)h, v);   // warp-collective
        const int dim = 128 * h + r;
#pragma unroll
        for (int k = 0; k < 64; ++k) {
          const float x = n > 0 ? u2f(v[k]) * mul : 0.f;
          if (!RAGGED || kv0 + k < Nk) dst[(size_t)k * kD + dim] = (uint16_t)(pack2<F16>(x, 0.f) & 0xFFFFu);
        }
      }
    }
  } else if (warp == kTmaWarp) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tmap(&a.tm_q);
      prefetch_tmap(&a.tm_k);
      prefetch_tmap(&a.tm_v);
      prefetch_tmap(&a.tm_do);
      mbar_arrive_expect_tx(bar(kKVFull), 8u * kKBox);
      for (int bx = 0; bx < 4; ++bx) {
        load_rows(sbase + kK + bx * kKBox, &a.tm_k, bar(kKVFull), 64 * bx, kv0, Nk);
        load_rows(sbase + kV + bx * kKBox, &a.tm_v, bar(kKVFull), 64 * bx, kv0, Nk);
      }
      int issued_q[4] = {0, 0, 0, 0}, issued_do[4] = {0, 0, 0, 0};
      bool ok = true;
      for (int i = 0; ok && i < n; ++i) {
        const int q0 = (i0 + i) * kBM;
        // Q boxes free up first (dKᵀ is issued before dVᵀ), then dO boxes,
        // half by half of the head dims.
        for (int bx = 0; ok && bx < 4; ++bx) {
          if (i > 0 && (bx & 1) == 0 && !mbar_wait(bar(kQEmpty + (bx >> 1)), (uint32_t)((i - 1) & 1), wc, site(5))) {
            ok = false;
            break;
          }
          if ((bx & 1) == 0) mbar_arrive_expect_tx(bar(kQFull + (bx >> 1)), 2u * kQBox + (bx == 0 ? 2u * kBM * 4 : 0u));
          load_rows(sbase + kQ + bx * kQBox, &a.tm_q, bar(kQFull + (bx >> 1)), 64 * bx, q0, Nq);
          if (bx == 0) {
            load_bulk(sbase + kLSE, a.lse2 + wrow0 + q0, kBM * 4, bar(kQFull));
            load_bulk(sbase + kDV, a.dvec + wrow0 + q0, kBM * 4, bar(kQFull));
          }
          ++issued_q[bx];
        }
        for (int bx = 0; ok && bx < 4; ++bx) {
          if (i > 0 && (bx & 1) == 0 && !mbar_wait(bar(kDOEmpty + (bx >> 1)), (uint32_t)((i - 1) & 1), wc, site(6))) {
            ok = false;
            break;
          }
          if ((bx & 1) == 0) mbar_arrive_expect_tx(bar(kDOFull + (bx >> 1)), 2u * kQBox);
          load_rows(sbase + kDO + bx * kQBox, &a.tm_do, bar(kDOFull + (bx >> 1)), 64 * bx, q0, Nq);
          ++issued_do[bx];
        }
      }
      // Never leave the CTA with copies in flight.
      mbar_wait_drain(bar(kKVFull), 0, wc, site(7));
      for (int bx = 0; bx < 4; bx += 2) {
        if (issued_q[bx] > 0) mbar_wait_drain(bar(kQFull + (bx >> 1)), (uint32_t)((issued_q[bx] - 1) & 1), wc, site(7));
        if (issued_do[bx] > 0) mbar_wait_drain(bar(kDOFull + (bx >> 1)), (uint32_t)((issued_do[bx] - 1) & 1), wc, site(7));
      }
    }
  } else {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_f16kind(128, kBN, false, false, F16);  // S = Q Kᵀ, dP = dO Vᵀ
      constexpr uint32_t kIdT = idesc_f16kind(128, kBN, true, true, F16);    // dVᵀ += dOᵀ P, dKᵀ += Qᵀ dS
      // S (A = Q) or dP (A = dO) of query tile i, box by box as the boxes land.
      auto issue_sd = [&](int i, uint32_t col, uint32_t a_tile, uint32_t b_tile, int full) -> bool {
        const uint64_t ad = sdesc_sw128(a_tile, 16, 1024), bd = sdesc_sw128(b_tile, 16, 1024);
        const uint32_t dcol = tmem + col;
        const bool chk = dcheck(tmem_ok(col, kBN, 512), wc, kChkTmem, 54) &&
                         dcheck(smem_ok(a_tile - sbase, 4 * kQBox, kBar, 1024) &&
                                    smem_ok(b_tile - sbase, 4 * kKBox, kBar, 1024), wc, kChkSmem, 54);
        for (int bx = 0; bx < 4; ++bx) {
          if ((bx & 1) == 0) {
            if (!mbar_wait(bar(full + (bx >> 1)), (uint32_t)(i & 1), wc, site(8))) return false;
            tc_fence_after();
          }
#pragma unroll
          for (int k = 0; k < 4; ++k)
            if (chk) mma_ss(dcol, sdesc_add(ad, bx * kQBox + 32u * k), sdesc_add(bd, bx * kKBox + 32u * k), kIdS,
                   (bx > 0 || k > 0) ? 1u : 0u);
        }
        return true;
      };
      // dKᵀ / dVᵀ operands: Q, dO read MN-major (A), dS, P read MN-major (B).
      const uint64_t q_mn = sdesc_sw128(sbase + kQ, kQBox, 1024), do_mn = sdesc_sw128(sbase + kDO, kQBox, 1024);
      const uint64_t ds_mn = sdesc_sw128(sbase + kDS, kQBox, 1024), p_mn = sdesc_sw128(sbase + kP, kQBox, 1024);
      bool ok = mbar_wait(bar(kKVFull), 0, wc, site(9));
      if (ok && n > 0) {
        ok = issue_sd(0, kColS, sbase + kQ, sbase + kK, kQFull);
        if (ok) {
          tc_commit(bar(kSFull));
          ok = issue_sd(0, kColDP, sbase + kDO, sbase + kV, kDOFull);
          if (ok) tc_commit(bar(kDPFull));
        }
      }
      for (int i = 0; ok && i < n; ++i) {
        if (!mbar_wait(bar(kPdsFull), (uint32_t)(i & 1), wc, site(10))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const bool chk = dcheck(tmem_ok(kColDK, 2 * kBN, 512) && tmem_ok(kColDV, 2 * kBN, 512), wc, kChkTmem, 55);
        // dKᵀ_h += Q_hᵀ dS, then dVᵀ_h += dO_hᵀ P: A MN-major over the two
        // boxes of half h, B = dS / P [query][key] MN-major; K-steps of 16 queries.
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
          for (int ks = 0; ks < kBM / 16; ++ks)
            if (chk) mma_ss(tmem + kColDK + 64u * h, sdesc_add(q_mn, 2 * h * kQBox + ks * 2048), sdesc_add(ds_mn, ks * 2048),
                   kIdT, (i > 0 || ks > 0) ? 1u : 0u);
          tc_commit(bar(kQEmpty + h));
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
          for (int ks = 0; ks < kBM / 16; ++ks)
            if (chk) mma_ss(tmem + kColDV + 64u * h, sdesc_add(do_mn, 2 * h * kQBox + ks * 2048), sdesc_add(p_mn, ks * 2048),
                   kIdT, (i > 0 || ks > 0) ? 1u : 0u);
          tc_commit(bar(kDOEmpty + h));
        }
        // The next tile's S and dP overwrite the columns the compute warps
        // have read; its P / dS stores wait for S, i.e. for these products.
        if (i + 1 < n) {
          ok = issue_sd(i + 1, kColS, sbase + kQ, sbase + kK, kQFull);
          if (!ok) break;
          tc_commit(bar(kSFull));
          ok = issue_sd(i + 1, kColDP, sbase + kDO, sbase + kV, kDOFull);
          if (!ok) break;
          tc_commit(bar(kDPFull));
        }
      }
      if (ok) tc_commit(bar(kDKVFull));
      tc_commit(bar(kMmaDone));
      mbar_wait_drain(bar(kMmaDone), 0, wc, site(11));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ================================================================== dQ

namespace dq {
constexpr int kKSlots = 8;                    // K ring, in boxes (two tiles)
constexpr int kQ = 0;                         // 4 boxes of 128 queries
constexpr int kDO = kQ + 4 * kQBox;
constexpr int kK = kDO + 4 * kQBox;           // kKSlots boxes of 64 keys
constexpr int kV = kK + kKSlots * kKBox;      // 4 boxes
constexpr int kLSE = kV + 4 * kKBox;
constexpr int kDV = kLSE + kBM * 4;
constexpr int kBar = kDV + kBM * 4;
constexpr int kBytes = kBar + 512;
static_assert(kBytes <= 232448, "shared memory exceeds the 227 KB a CTA may use");

enum Bar : int {
  kQFull = 0,                    // Q, dO, −LSE₂, −D
  kKFull = 1,                    // + tile of the ring (2): its four boxes land together
  kKEmpty = kKFull + 2,          // + tile of the ring (2): its four boxes are released together
  kVFull = kKEmpty + 2,          // the V tile
  kVEmpty = kVFull + 1,          // the V tile, released once dP has read all four boxes
  kSFull = kVEmpty + 1,          // + buffer (2)
  kDPFull = kSFull + 2,          // + buffer
  kDsFull = kDPFull + 2,         // + buffer
  kDqFull = kDsFull + 2,
  kMmaDone,
  kNumBars,
};
static_assert(8 * kNumBars + 8 <= 512, "barrier block too small");

constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 256;

__device__ __forceinline__ uint32_t site(int s) { return 0x0500u | (uint32_t)s; }
}  // namespace dq

template <bool CAUSAL, bool RAGGED, bool F16>
__global__ void __launch_bounds__(kThreads, 1) fa_bwd_d256_dq_kernel(const __grid_constant__ BwdArgs a) {
  using namespace dq;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t sbase = smem_u32(smem_raw);
  uint8_t* sgen = smem_raw;
  if (sbase & 1023u) {
    if (threadIdx.x == 0) atomicCAS(a.fault, 0u, site(0));
    return;
  }
  const uint32_t bars = sbase + kBar;
  auto bar = [&](int i) -> uint32_t { return bars + 8u * (uint32_t)i; };
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sgen + kBar + 8 * kNumBars);
  int* abort_flag = reinterpret_cast<int*>(sgen + kBar + 8 * kNumBars + 4);
  const WaitCtx wc{abort_flag, a.fault};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int Nq = a.Nq, Nk = a.Nk;
  const int off = Nk - Nq;
  const int tiles = (Nq + kBM - 1) / kBM;
  // Causal: batch·head fastest, the longest query tiles (the last ones) first.
  const int bh = CAUSAL ? (int)blockIdx.x : (int)blockIdx.y;
  const int it = CAUSAL ? tiles - 1 - (int)blockIdx.y : (int)blockIdx.x;
  const int q0 = it * kBM;
  const int wrow0 = bh * tiles * kBM;
  const int row0 = bh * Nq;
  // Key tiles visited: under the causal mask up to the last key the tile's
  // last real query sees.
  const int last_key = (q0 + kBM - 1 < Nq ? q0 + kBM - 1 : Nq - 1) + off;
  const int n_all = (Nk + kBN - 1) / kBN;
  const int n = CAUSAL ? last_key / kBN + 1 : n_all;
  // A debug build checks each box's destination and coordinates first (K and V
  // boxes are 64 rows, Q and dO boxes 128) and, if a check fails, completes its
  // bytes on the barrier without copying; bulk copies likewise.
  auto load_rows = [&](uint32_t dst, const CUtensorMap* map, uint32_t bar_addr, int x, int pos, int nrows) {
    const bool kv_map = map == &a.tm_k || map == &a.tm_v;
    const uint32_t box = kv_map ? (uint32_t)kKBox : (uint32_t)kQBox;
    bool chk = dcheck(smem_ok(dst - sbase, box, (uint32_t)kBar, 1024), wc, kChkSmem, 56) &&
               dcheck(tma_x_ok(x, 64, kD), wc, kChkTmaX, 56);
    if constexpr (RAGGED)
      chk = chk && dcheck(tma_head_ok(pos, nrows, bh, a.B * a.H), wc, kChkTmaRows, 56);
    else
      chk = chk && dcheck(tma_rows_ok((long long)bh * nrows + pos, (int)(box / 128), (long long)a.B * a.H * nrows),
                          wc, kChkTmaRows, 56);
    if (!chk) {
      mbar_complete_tx(bar_addr, box);
      return;
    }
    if constexpr (RAGGED)
      tma_load_3d(dst, map, bar_addr, x, pos, bh);
    else
      tma_load_2d(dst, map, bar_addr, x, bh * nrows + pos);
  };
  auto load_bulk = [&](uint32_t dst, const float* src, uint32_t bytes, uint32_t bar_addr) {
    if (!dcheck(smem_ok(dst - sbase, bytes, (uint32_t)kBar, 16) && bulk_ok(reinterpret_cast<uint64_t>(src), dst, bytes),
                wc, kChkBulk, 56 + 1)) {
      mbar_complete_tx(bar_addr, bytes);
      return;
    }
    bulk_load(dst, src, bytes, bar_addr);
  };

  if (threadIdx.x == 0) {
    mbar_init(bar(kQFull), 1);
    for (int t = 0; t < 2; ++t) mbar_init(bar(kKFull + t), 1);
    for (int t = 0; t < 2; ++t) mbar_init(bar(kKEmpty + t), 1);
    mbar_init(bar(kVFull), 1);
    mbar_init(bar(kVEmpty), 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(kSFull + b), 1);
      mbar_init(bar(kDPFull + b), 1);
      mbar_init(bar(kDsFull + b), 256);
    }
    mbar_init(bar(kDqFull), 1);
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

  if (warp < 8) {
    // ------------------------------------------------------------ dS
    const int c = warp >> 2;                   // key columns [32c, 32c + 32)
    const int g = warp & 3;
    const int r = g * 32 + lane;               // query row within the tile = TMEM lane
    const uint32_t lane_off = (uint32_t)(g * 32) << 16;
    const float sl2 = a.scale_log2;
    bool ok = mbar_wait(bar(kQFull), 0, wc, site(1));
    ok = __all_sync(kFull, ok);
    const float nlse = ok ? reinterpret_cast<const float*>(sgen + kLSE)[r] : 0.f;
    const float nd = ok ? reinterpret_cast<const float*>(sgen + kDV)[r] : 0.f;
    for (int j = 0; ok && j < n; ++j) {
      const int b = j & 1;
      const uint32_t par = (uint32_t)((j >> 1) & 1);
      ok = mbar_wait(bar(kSFull + b), par, wc, site(2));
      ok = __all_sync(kFull, ok);
      if (!ok) break;
      tc_fence_after();
      const int kv0 = j * kBN;
      const int delta = q0 + off - kv0;       // key kv0 + 32c + k visible iff k ≤ r + delta − 32c
      float p[32];
      {
        uint32_t s[32];
        if (dcheck(tmem_ok(kColS + 64u * b + 32u * c, 32, 512), wc, kChkTmem, 58))
          tmem_ld_x32(tmem + lane_off + kColS + 64u * (uint32_t)b + 32u * (uint32_t)c, s);
        if (CAUSAL && delta < kBN - 1)
          p_row32<true>(s, sl2, nlse, r + delta - 32 * c, p);
        else if (RAGGED && !CAUSAL && kv0 + kBN > Nk)
          p_row32<true>(s, sl2, nlse, Nk - kv0 - 32 * c - 1, p);
        else
          p_row32<false>(s, sl2, nlse, 0, p);
      }
      ok = mbar_wait(bar(kDPFull + b), par, wc, site(3));
      ok = __all_sync(kFull, ok);
      if (!ok) break;
      tc_fence_after();
      const uint32_t dp_col = kColDP + 64u * (uint32_t)b + 32u * (uint32_t)c;
      uint32_t dp[32];
      const bool chk = dcheck(tmem_ok(dp_col, 32, 512), wc, kChkTmem, 59);
      if (chk) tmem_ld_x32(tmem + lane_off + dp_col, dp);
      uint32_t ds[16];
      ds_row32<F16>(p, dp, nd, ds);
      // dS over the first 16 of the 32 dP columns this thread has just read.
      if (chk) tmem_st_x16(tmem + lane_off + dp_col, ds);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(kDsFull + b));
    }
    // ------------------------------------------------------------ epilogue
    if (ok) {
      ok = mbar_wait(bar(kDqFull), 0, wc, site(4));
      ok = __all_sync(kFull, ok);
    }
    if (ok) {
      tc_fence_after();
      const int q = q0 + r;
      const bool live = !RAGGED || q < Nq;
      uint16_t* drow = static_cast<uint16_t*>(a.dq) + ((size_t)row0 + (size_t)q) * kD + 128 * c;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t v[32];
        if (!dcheck(tmem_ok(kColDQ + 128u * c + 32u * cc, 32, 512), wc, kChkTmem, 60)) continue;
        tmem_ld_x32(tmem + lane_off + kColDQ + 128u * (uint32_t)c + 32u * (uint32_t)cc, v);   // warp-collective
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) pk[e] = pack2<F16>(u2f(v[2 * e]) * a.scale, u2f(v[2 * e + 1]) * a.scale);
        if (live) {
#pragma unroll
          for (int u = 0; u < 4; ++u)
            st_global_v4(drow + 32 * cc + 8 * u, pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
        }
      }
    }
  } else if (warp == kTmaWarp) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tmap(&a.tm_q);
      prefetch_tmap(&a.tm_k);
      prefetch_tmap(&a.tm_v);
      prefetch_tmap(&a.tm_do);
      mbar_arrive_expect_tx(bar(kQFull), 8u * kQBox + 2u * kBM * 4);
      for (int bx = 0; bx < 4; ++bx) {
        load_rows(sbase + kQ + bx * kQBox, &a.tm_q, bar(kQFull), 64 * bx, q0, Nq);
        load_rows(sbase + kDO + bx * kQBox, &a.tm_do, bar(kQFull), 64 * bx, q0, Nq);
      }
      load_bulk(sbase + kLSE, a.lse2 + wrow0 + q0, kBM * 4, bar(kQFull));
      load_bulk(sbase + kDV, a.dvec + wrow0 + q0, kBM * 4, bar(kQFull));
      int k_boxes = 0, v_loads[4] = {0, 0, 0, 0};
      auto load_k = [&](int j) -> bool {
        for (int bx = 0; bx < 4; ++bx) {
          const int gi = 4 * j + bx, slot = gi % kKSlots, round = gi / kKSlots;
          if (round > 0 && bx == 0 && !mbar_wait(bar(kKEmpty + (j & 1)), (uint32_t)((round - 1) & 1), wc, site(5))) return false;
          if (bx == 0) mbar_arrive_expect_tx(bar(kKFull + (j & 1)), 4u * kKBox);
          load_rows(sbase + kK + slot * kKBox, &a.tm_k, bar(kKFull + (j & 1)), 64 * bx, j * kBN, Nk);
          ++k_boxes;
        }
        return true;
      };
      auto load_v = [&](int j) -> bool {
        for (int bx = 0; bx < 4; ++bx) {
          if (j > 0 && bx == 0 && !mbar_wait(bar(kVEmpty), (uint32_t)((j - 1) & 1), wc, site(6))) return false;
          if (bx == 0) mbar_arrive_expect_tx(bar(kVFull), 4u * kKBox);
          load_rows(sbase + kV + bx * kKBox, &a.tm_v, bar(kVFull), 64 * bx, j * kBN, Nk);
          ++v_loads[bx];
        }
        return true;
      };
      // K_0, V_0, K_1, V_1, then V_j before K_j: V_j waits for dP_{j-1},
      // K_j for dQ_{j-2}; the MMA order is dQ_{j-2}, S_{j-1}, dP_j.
      bool ok = load_k(0) && load_v(0);
      if (ok && n > 1) ok = load_k(1) && load_v(1);
      for (int j = 2; ok && j < n; ++j) ok = load_v(j) && load_k(j);
      mbar_wait_drain(bar(kQFull), 0, wc, site(7));
      const int k_tiles = k_boxes / 4;
      for (int t = 0; t < 2 && t < k_tiles; ++t) {
        const int last = t + (k_tiles - 1 - t) / 2 * 2;
        mbar_wait_drain(bar(kKFull + t), (uint32_t)((last / 2) & 1), wc, site(7));
      }
      if (v_loads[0] > 0) mbar_wait_drain(bar(kVFull), (uint32_t)((v_loads[0] - 1) & 1), wc, site(7));
    }
  } else {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_f16kind(128, kBN, false, false, F16);   // S = Q Kᵀ, dP = dO Vᵀ
      constexpr uint32_t kIdQ = idesc_f16kind(128, kD, false, true, F16);     // dQ += dS K, N = 256 over the four K boxes
      const uint64_t q_k = sdesc_sw128(sbase + kQ, 16, 1024), do_k = sdesc_sw128(sbase + kDO, 16, 1024);
      const uint64_t k_k = sdesc_sw128(sbase + kK, 16, 1024), v_k = sdesc_sw128(sbase + kV, 16, 1024);
      const uint64_t k_mn = sdesc_sw128(sbase + kK, kKBox, 1024);
      auto issue_s = [&](int j) -> bool {
        const uint32_t col = tmem + kColS + 64u * (uint32_t)(j & 1);
        const bool chk = dcheck(tmem_ok(kColS + 64u * (j & 1), kBN, 512), wc, kChkTmem, 61);
        for (int bx = 0; bx < 4; ++bx) {
          const int gi = 4 * j + bx, slot = gi % kKSlots;
          if (bx == 0) {
            if (!mbar_wait(bar(kKFull + (j & 1)), (uint32_t)((gi / kKSlots) & 1), wc, site(8))) return false;
            tc_fence_after();
          }
#pragma unroll
          for (int k = 0; k < 4; ++k)
            if (chk) mma_ss(col, sdesc_add(q_k, bx * kQBox + 32u * k), sdesc_add(k_k, slot * kKBox + 32u * k), kIdS,
                   (bx > 0 || k > 0) ? 1u : 0u);
        }
        tc_commit(bar(kSFull + (j & 1)));
        return true;
      };
      auto issue_dp = [&](int j) -> bool {
        const uint32_t col = tmem + kColDP + 64u * (uint32_t)(j & 1);
        const bool chk = dcheck(tmem_ok(kColDP + 64u * (j & 1), kBN, 512), wc, kChkTmem, 62);
        for (int bx = 0; bx < 4; ++bx) {
          if (bx == 0) {
            if (!mbar_wait(bar(kVFull), (uint32_t)(j & 1), wc, site(9))) return false;
            tc_fence_after();
          }
#pragma unroll
          for (int k = 0; k < 4; ++k)
            if (chk) mma_ss(col, sdesc_add(do_k, bx * kQBox + 32u * k), sdesc_add(v_k, bx * kKBox + 32u * k), kIdS,
                   (bx > 0 || k > 0) ? 1u : 0u);
        }
        tc_commit(bar(kVEmpty));
        tc_commit(bar(kDPFull + (j & 1)));
        return true;
      };
      // dQ += dS_j K_j: A = dS from tensor memory (keys 0-31 in the first 16
      // columns written by warps 0-3, keys 32-63 in those written by warps
      // 4-7), B = K_j MN-major, N = 256 over its four boxes, which sit in
      // consecutive ring slots 4(j mod 2) .. +3.
      auto issue_dq = [&](int j) {
        const uint32_t ds_col = tmem + kColDP + 64u * (uint32_t)(j & 1);
        const uint32_t slot0 = (uint32_t)((4 * j) % kKSlots);
        const bool chk = dcheck(tmem_ok(kColDQ, kD, 512) && tmem_ok(kColDP + 64u * (j & 1), kBN, 512), wc, kChkTmem,
                                63) &&
                         dcheck(smem_ok(kK + slot0 * kKBox, 4 * kKBox, kBar, 1024), wc, kChkSmem, 63);
#pragma unroll
        for (int ks = 0; ks < kBN / 16; ++ks)
          if (chk) mma_ts(tmem + kColDQ, ds_col + (uint32_t)(ks < 2 ? 8 * ks : 32 + 8 * (ks - 2)),
                 sdesc_add(k_mn, slot0 * kKBox + ks * 2048), kIdQ, (j > 0 || ks > 0) ? 1u : 0u);
        tc_commit(bar(kKEmpty + (j & 1)));
      };
      bool ok = mbar_wait(bar(kQFull), 0, wc, site(10));
      if (ok && n > 0) ok = issue_s(0) && issue_dp(0);
      if (ok && n > 1) ok = issue_dp(1);
      for (int j = 0; ok && j < n; ++j) {
        if (!mbar_wait(bar(kDsFull + (j & 1)), (uint32_t)((j >> 1) & 1), wc, site(11))) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_dq(j);
        if (j + 1 < n) ok = issue_s(j + 1);
        if (ok && j + 2 < n) ok = issue_dp(j + 2);
      }
      if (ok) tc_commit(bar(kDqFull));
      tc_commit(bar(kMmaDone));
      mbar_wait_drain(bar(kMmaDone), 0, wc, site(12));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <bool CAUSAL, bool RAGGED, bool F16>
cudaError_t launch_impl(const BwdArgs& a, cudaStream_t s) {
  auto k1 = fa_bwd_d256_dkdv_kernel<CAUSAL, RAGGED, F16>;
  auto k2 = fa_bwd_d256_dq_kernel<CAUSAL, RAGGED, F16>;
  cudaError_t e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, kv::kBytes);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, dq::kBytes);
  if (e != cudaSuccess) return e;
  const unsigned heads = (unsigned)(a.B * a.H);
  const unsigned kt = (unsigned)((a.Nk + kBN - 1) / kBN), qt = (unsigned)((a.Nq + kBM - 1) / kBM);
  k1<<<CAUSAL ? dim3(heads, kt) : dim3(kt, heads), kThreads, kv::kBytes, s>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  k2<<<CAUSAL ? dim3(heads, qt) : dim3(qt, heads), kThreads, dq::kBytes, s>>>(a);
  return cudaGetLastError();
}

template <bool F16>
cudaError_t dispatch(const BwdArgs& a, bool ragged, cudaStream_t s) {
  if (ragged) return a.causal ? launch_impl<true, true, F16>(a, s) : launch_impl<false, true, F16>(a, s);
  return a.causal ? launch_impl<true, false, F16>(a, s) : launch_impl<false, false, F16>(a, s);
}

}  // namespace

cudaError_t launch_bwd_d256(const BwdArgs& a, cudaStream_t s) {
  if (a.d != kD || a.dq == nullptr) return cudaErrorInvalidValue;
  const bool ragged = a.Nq % kBM != 0 || a.Nk % kBM != 0;
  return a.f16 ? dispatch<true>(a, ragged, s) : dispatch<false>(a, ragged, s);
}

}  // namespace fa
