// fa_fwd_bf16.cu — tiled attention forward on the sm_103a tensor cores.
//
// What it computes: "Flash Attention" tutorial, 2.Online Softmax §4.2 — one
// pass over K/V tiles with the running (m, ℓ) of §3.1 and the unnormalised
// output Õ of §4.1, divided by ℓ once at the end; the saved statistic is
// LSE = m + ln ℓ (3.Recomputation 三).  Scores never leave the SM.
//
// CTA = two 128-row query tiles of one (batch, head), 10 warps:
//   warps 0-3  softmax for query tile 0 (one thread per query row)
//   warps 4-7  softmax for query tile 1
//   warp  8    TMA producer: Q once, then K_j / V_j through a 2-stage ring
//   warp  9    MMA issuer (one thread) and tensor-memory owner
// Tensor memory (512 columns × 128 lanes × 32 bit):
//   S_t  = cols [128 t, 128 t + 128)   fp32 scores of tile t (S = Q_t K_jᵀ)
//   P_t  = cols [128 t, 128 t + 64)    bf16x2 probabilities, written over S_t
//   O_t  = cols [256 + d t, 256 + d t + d)   fp32 unnormalised output
// Per K/V tile the MMA thread issues, for each query tile, O_t += P_t V_j (A
// from tensor memory) and then S_t = Q_t K_{j+1}ᵀ, so the softmax of one
// tile overlaps the products of the other.  That order matters: issuing each
// tile's products from its own thread (two issuers, the tensor pipe then
// interleaving them) measured 7-14 % slower on GB300.
//
// Rescaling is lazy: the reference max m only moves when a row's new max
// exceeds it by more than 8 (base 2), so P ≤ 2^8 and ℓ and Õ keep sharing one
// reference — the merge of §3.1/§4.1 with a stale but common reference is
// still exact.  When it moves, the softmax thread rescales its row of O_t in
// tensor memory; the commit that signalled S_t also guarantees the previous
// O_t += P_t V product has finished.
#include <cmath>

#include "fa_kernels.h"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

constexpr int kBM = 128;           // query rows per tile
constexpr int kBN = 128;           // keys per K/V tile
constexpr int kThreads = 320;
constexpr int kTmaWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kBoxBytes = 128 * 128;   // one TMA box: 128 rows × 128 bytes
// Exponential pairs per FMA-pipe exponential (0 = all on MUFU).  Measured on
// GB300: moving 1/8, 1/4 or 1/2 of them to the FMA pipe slows the softmax
// (it is issue-bound, not MUFU-bound), so all stay on MUFU.
constexpr int kPolyEvery = 0;

// K and V ring depths.  Measured on GB300 (clock64 trace): the loads arrive
// well before the MMA thread needs them, and deeper rings (three to six
// stages at d = 64, a third V stage at d = 128) were no faster or slower.
template <int D>
struct FwdStages {
  static constexpr int kK = 2;
  static constexpr int kV = 2;
};

// Shared-memory layout (offsets from a 1024-byte aligned base).
template <int D>
struct FwdLayout {
  static constexpr int kKS = FwdStages<D>::kK;
  static constexpr int kVS = FwdStages<D>::kV;
  static constexpr int kTile = kBM * D * 2;       // bytes of one 128 × D bf16 tile
  static constexpr int kQ = 0;                    // Q tile t at kQ + t·kTile
  static constexpr int kK = kQ + 2 * kTile;       // K stage s at kK + s·kTile
  static constexpr int kV = kK + kKS * kTile;     // V stage s at kV + s·kTile
  static constexpr int kBar = kV + kVS * kTile;
  static constexpr int kBytes = kBar + 512;
};

// Barrier slots (8 bytes each) inside the barrier block.
template <int KS, int VS>
struct FwdBars {
  static constexpr int kQFull = 0;
  static constexpr int kKFull = 1;               // +stage
  static constexpr int kKEmpty = kKFull + KS;    // +stage
  static constexpr int kVFull = kKEmpty + KS;    // +stage
  static constexpr int kVEmpty = kVFull + VS;    // +stage
  static constexpr int kSFull = kVEmpty + VS;    // +tile
  static constexpr int kPFull = kSFull + 2;      // +tile
  static constexpr int kOFull = kPFull + 2;      // +tile
  static constexpr int kMmaDone = kOFull + 2;
  static constexpr int kNumBars = kMmaDone + 1;
  static_assert(8 * kNumBars + 8 <= 512, "barrier block too small");
};

// Fault codes recorded when a wait runs out of time (kernel id 1 in the high byte).
__device__ __forceinline__ uint32_t site(int s) { return 0x0100u | (uint32_t)s; }

// P = 2^(s·scale·log2e − m) for one 128-column row of S, rounded to bf16 and
// stored over the row's first 64 tensor-memory columns; returns Σ P in fp32.
// The scale-and-subtract and the sum run as packed f32x2 operations; with
// POLY_EVERY > 0, one pair of exponentials in POLY_EVERY runs on the FMA pipe
// (exp2_fma_x2), the others on MUFU.
template <int POLY_EVERY, bool F16>
__device__ __forceinline__ float exp_tile_to_p(const uint32_t (&s)[128], float sl2, float m_ref, uint32_t p_addr) {
  const uint64_t sl2x2 = f2_pack(sl2, sl2);
  const uint64_t negx2 = f2_pack(-m_ref, -m_ref);
  uint64_t lsum0 = f2_pack(0.f, 0.f), lsum1 = lsum0;
#pragma unroll
  for (int cc = 0; cc < 4; ++cc) {
    uint32_t p[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint64_t x = f2_fma(f2_pack(u2f(s[32 * cc + 2 * i]), u2f(s[32 * cc + 2 * i + 1])), sl2x2, negx2);
      float x0, x1, e0, e1;
      f2_unpack(x, x0, x1);
      if (POLY_EVERY > 0 && i % (POLY_EVERY > 0 ? POLY_EVERY : 1) == POLY_EVERY - 1) {
        exp2_fma_x2(x0, x1, e0, e1);
      } else {
        e0 = ex2(x0);
        e1 = ex2(x1);
      }
      if (i & 1)
        lsum1 = f2_add(lsum1, f2_pack(e0, e1));
      else
        lsum0 = f2_add(lsum0, f2_pack(e0, e1));
      p[i] = pack2<F16>(e0, e1);
    }
    tmem_st_x16(p_addr + 16 * cc, p);
  }
  float la, lb, lc, ld;
  f2_unpack(lsum0, la, lb);
  f2_unpack(lsum1, lc, ld);
  return (la + lb) + (lc + ld);
}

// RAGGED (Nq or Nk not a multiple of 128): 3-D per-head tensor maps whose
// rows past the end read as zero, masking of the missing keys and
// row-predicated stores.  Otherwise 2-D maps over the row views and none of
// that code.
// F16: fp16 inputs and outputs (else bf16); P is rounded to the same type.
// DR: the head dimension (64, 96 or 128).  Tiles are laid out D = 64 or 128
// columns wide; with DR = 96 the tensor maps read columns 96..127 as zeros,
// the products run over the 96 real columns only (6 K-steps of 16 for S, an
// N = 96 product for O) and 96 columns are stored.
template <int DR, bool CAUSAL, bool RAGGED, bool F16>
__global__ void __launch_bounds__(kThreads, 1) fa_fwd_bf16_kernel(const __grid_constant__ FwdArgs a) {
  constexpr int D = DR <= 64 ? 64 : 128;
  using L = FwdLayout<D>;
  constexpr int KS = L::kKS, VS = L::kVS;
  using Bar = FwdBars<KS, VS>;
  constexpr int kQFull = Bar::kQFull, kKFull = Bar::kKFull, kKEmpty = Bar::kKEmpty, kVFull = Bar::kVFull,
                kVEmpty = Bar::kVEmpty, kSFull = Bar::kSFull, kPFull = Bar::kPFull, kOFull = Bar::kOFull,
                kMmaDone = Bar::kMmaDone, kNumBars = Bar::kNumBars;
  // Dynamic shared memory starts on a 1024-byte boundary (no static shared
  // memory is declared); 128-byte swizzled tiles need that alignment.
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t sbase = smem_u32(smem_raw);
  uint8_t* sgen = smem_raw;
  if (sbase & 1023u) {
    if (threadIdx.x == 0) atomicCAS(a.fault, 0u, site(0));
    return;
  }
  const uint32_t bars = sbase + L::kBar;
  auto bar = [&](int i) -> uint32_t { return bars + 8u * (uint32_t)i; };
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sgen + L::kBar + 8 * kNumBars);
  int* abort_flag = reinterpret_cast<int*>(sgen + L::kBar + 8 * kNumBars + 4);
  const WaitCtx wc{abort_flag, a.fault};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int Nq = a.Nq, Nk = a.Nk;
  const int off = Nk - Nq;                               // causal: query i sees keys j ≤ i + off
  const int pairs = (Nq + 2 * kBM - 1) / (2 * kBM);      // two-tile units per head
  // Work of this CTA (1-D grid).  Causal without a split: batch·head fastest
  // with the heaviest pairs first across the whole grid (longest tiles
  // scheduled first).  Otherwise head-major (pair fastest), so a wave touches
  // few heads' K/V and they stay in L2; units [n_full, units) are split into
  // `splits` CTAs over equal ranges of the K/V tiles they see, each writing a
  // partial result (normalised O and LSE of its keys) that fwd_combine
  // merges: the last partial wave of a long problem, or every unit of a
  // problem with few queries (which streams K/V far more than it computes).
  const int n_kv_all = (Nk + kBN - 1) / kBN;
  int bh, pair, kv_begin = 0, n_kv = n_kv_all, part_slot = -1;
  const int idx = (int)blockIdx.x;
  if (CAUSAL && a.splits <= 1) {
    bh = idx % (a.B * a.H);
    pair = pairs - 1 - idx / (a.B * a.H);
  } else if (idx < a.n_full) {
    bh = idx / pairs;
    pair = idx % pairs;
  } else {
    part_slot = idx - a.n_full;                            // = split unit · splits + part
    const int unit = a.n_full + part_slot / a.splits;
    const int part = part_slot % a.splits;
    bh = unit / pairs;
    pair = unit % pairs;
    // K/V tiles the unit's queries see: all of them without the mask; with
    // it, up to the last key of the unit's last query.
    int n_vis = n_kv_all;
    if (CAUSAL) {
      const int last_q = pair * 2 * kBM + 2 * kBM - 1 < Nq ? pair * 2 * kBM + 2 * kBM - 1 : Nq - 1;
      n_vis = (last_q + off) / kBN + 1;
    }
    kv_begin = part * n_vis / a.splits;
    n_kv = (part + 1) * n_vis / a.splits - kv_begin;
  }
  const int q0 = pair * 2 * kBM;
  const int row0 = bh * Nq;                                // first row of this head in the [B·H·Nq, d] view
  // Keys of the head's last K/V tile that exist (128 unless Nk is ragged).
  // Non-causal rows must not see the zero-filled keys past Nk; causal rows
  // never do, since those keys lie beyond every real query's last key.
  const int kv_tail = Nk - (n_kv_all - 1) * kBN;
  const bool ragged_last = RAGGED && !CAUSAL && kv_tail < kBN && kv_begin + n_kv == n_kv_all;
  // Loads rows [pos, pos + 128) of this head from a map over heads of `n` rows.
  // A debug build checks the destination and the coordinates first and, if a
  // check fails, completes the box's bytes on the barrier without copying.
  auto load_rows = [&](uint32_t dst, const CUtensorMap* map, uint32_t bar_addr, int x, int pos, int n) {
    bool chk = dcheck(smem_ok(dst - sbase, kBoxBytes, (uint32_t)L::kBar, 1024), wc, kChkSmem, 1) &&
               dcheck(tma_x_ok(x, 64, D), wc, kChkTmaX, 1);
    if constexpr (RAGGED)
      chk = chk && dcheck(tma_head_ok(pos, n, bh, a.B * a.H), wc, kChkTmaRows, 1);
    else
      chk = chk && dcheck(tma_rows_ok((long long)bh * n + pos, kBM, (long long)a.B * a.H * n), wc, kChkTmaRows, 1);
    if (!chk) {
      mbar_complete_tx(bar_addr, kBoxBytes);
      return;
    }
    if constexpr (RAGGED)
      tma_load_3d(dst, map, bar_addr, x, pos, bh);
    else
      tma_load_2d(dst, map, bar_addr, x, bh * n + pos);
  };

  // Number of K/V tiles each query tile visits (0 if the tile is past Nq),
  // and under the causal mask the first tile that masks some of its scores:
  // tile j holds keys 128j + c, visible to row qt + r iff
  // c ≤ r + (qt + off − 128j); the last row that exists sees up to
  // min(qt + 127, Nq − 1) + off ≤ Nk − 1.
  int n_t[2], first_masked[2];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int qt = q0 + t * kBM;
    const int last_key = (qt + kBM - 1 < Nq ? qt + kBM - 1 : Nq - 1) + off;
    // K/V tiles this query tile visits within [kv_begin, kv_begin + n_kv),
    // and the first of them (relative to kv_begin) that masks a score.
    int vis = CAUSAL ? last_key / kBN + 1 - kv_begin : n_kv;
    vis = vis < 0 ? 0 : (vis > n_kv ? n_kv : vis);
    n_t[t] = qt >= Nq ? 0 : vis;
    first_masked[t] = (qt + off + 1) / kBN - kv_begin;
  }
  const int J = n_t[0] > n_t[1] ? n_t[0] : n_t[1];

  if (threadIdx.x == 0) {
    mbar_init(bar(kQFull), 1);
    for (int s = 0; s < KS; ++s) {
      mbar_init(bar(kKFull + s), 1);
      mbar_init(bar(kKEmpty + s), 1);
    }
    for (int s = 0; s < VS; ++s) {
      mbar_init(bar(kVFull + s), 1);
      mbar_init(bar(kVEmpty + s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(kSFull + t), 1);
      mbar_init(bar(kPFull + t), 128);
      mbar_init(bar(kOFull + t), 1);
    }
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
  auto s_col = [](int t) -> uint32_t { return (uint32_t)(128 * t); };
  auto o_col = [](int t) -> uint32_t { return (uint32_t)(256 + D * t); };

  if (warp < 8) {
    // ------------------------------------------------------------ softmax
    const int t = warp >> 2;
    const int r = (warp & 3) * 32 + lane;                // row within the tile = TMEM lane
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const int nt = n_t[t];
    const int fm = first_masked[t];
    const int qt = q0 + t * kBM;
    const float sl2 = a.scale_log2;
    float m_ref = -INFINITY;   // reference max of the row, base-2 scaled units
    float ell = 0.f;
    bool ok = true;
    for (int j = 0; j < nt; ++j) {
      ok = mbar_wait(bar(kSFull + t), (uint32_t)(j & 1), wc, site(1));
      ok = __all_sync(kFull, ok);
      if (!ok) break;
      tc_fence_after();
      uint32_t s[128];
      if (dcheck(tmem_ok(s_col(t), 128, 512), wc, kChkTmem, 2)) tmem_ld_x128(tmem + lane_off + s_col(t), s);
      if (CAUSAL && j >= fm) {
        // A tile crossing the diagonal: key 128j + c is visible to query
        // qt + r iff c ≤ r + qt + off − 128j (c ≤ r for square problems).
        const int lim = r + qt + off - (kv_begin + j) * kBN;
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c > lim) s[c] = f2u(-INFINITY);
      }
      if (ragged_last && j == nt - 1) {
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c >= kv_tail) s[c] = f2u(-INFINITY);
      }
      // Row max: four independent chains of 3-input maxima.
      float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
      for (int c = 0; c < 128; c += 8) {
        mx0 = max3(mx0, u2f(s[c]), u2f(s[c + 1]));
        mx1 = max3(mx1, u2f(s[c + 2]), u2f(s[c + 3]));
        mx2 = max3(mx2, u2f(s[c + 4]), u2f(s[c + 5]));
        mx3 = max3(mx3, u2f(s[c + 6]), u2f(s[c + 7]));
      }
      const float mx = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * sl2;
      const bool move = mx > m_ref + 8.0f;                 // always true on the first tile
      const float m_new = move ? mx : m_ref;
      const float alpha = ex2(m_ref - m_new);              // 0 on the first tile, 1 if the reference stays
      if (j > 0 && __any_sync(kFull, move)) {
        // O_t += P_t V_{j-1} has completed (it was issued before S_t = Q_t K_jᵀ,
        // whose commit we just waited on) and the next product into O_t waits
        // for P_full, so this row of O_t is ours to rescale.
#pragma unroll
        for (int cc = 0; cc < DR / 32; ++cc) {
          if (!dcheck(tmem_ok(o_col(t) + 32 * cc, 32, 512), wc, kChkTmem, 3)) continue;
          uint32_t o[32];
          tmem_ld_x32(tmem + lane_off + o_col(t) + 32 * cc, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = f2u(u2f(o[i]) * alpha);
          tmem_st_x32(tmem + lane_off + o_col(t) + 32 * cc, o);
        }
      }
      ell *= alpha;
      m_ref = m_new;
      // Masked tiles take every exponential on MUFU, so masked scores give
      // exactly 0.
      const uint32_t p_addr = tmem + lane_off + s_col(t);
      if (!dcheck(tmem_ok(s_col(t), kBN / 2, 512), wc, kChkTmem, 4)) {
      } else if ((CAUSAL && j >= fm) || (ragged_last && j == nt - 1))
        ell += exp_tile_to_p<0, F16>(s, sl2, m_ref, p_addr);
      else
        ell += exp_tile_to_p<kPolyEvery, F16>(s, sl2, m_ref, p_addr);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(kPFull + t));
    }
    if (ok && nt > 0) {
      ok = mbar_wait(bar(kOFull + t), 0, wc, site(2));
      ok = __all_sync(kFull, ok);
      if (ok) {
        tc_fence_after();
        const int q = q0 + t * kBM + r;
        const float inv = 1.0f / ell;
        // LSE in natural log of the scaled scores: (m + log2 ℓ) · ln 2.
        const float lse = (m_ref + log2f(ell)) * 0.69314718055994530942f;
        if (part_slot < 0) {
          // tcgen05.ld is warp-collective: every lane loads, and only rows
          // below Nq (the last tile of a ragged head) are stored.
          const bool live = !RAGGED || q < Nq;
          uint16_t* orow = static_cast<uint16_t*>(a.o) + ((size_t)row0 + (size_t)q) * DR;
#pragma unroll
          for (int cc = 0; cc < DR / 32; ++cc) {
            if (!dcheck(tmem_ok(o_col(t) + 32 * cc, 32, 512), wc, kChkTmem, 5)) continue;
            uint32_t o[32];
            tmem_ld_x32(tmem + lane_off + o_col(t) + 32 * cc, o);
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) pk[i] = pack2<F16>(u2f(o[2 * i]) * inv, u2f(o[2 * i + 1]) * inv);
            if (live) {
#pragma unroll
              for (int v4 = 0; v4 < 4; ++v4)
                st_global_v4(orow + 32 * cc + 8 * v4, pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
            }
          }
          if (live) a.lse[(size_t)row0 + (size_t)q] = lse;
        } else {
          // Partial over this CTA's keys: normalised O and LSE in fp32, one
          // row per query of the unit that exists (a slot holds part_rows
          // rows: 256, or the query count of a problem with few queries).
          const int urow = t * kBM + r;
          const bool live = urow < a.part_rows && q < Nq;
          const size_t prow = (size_t)part_slot * (size_t)a.part_rows + (size_t)urow;
          float* orow = a.opart + prow * DR;
#pragma unroll
          for (int cc = 0; cc < DR / 32; ++cc) {
            if (!dcheck(tmem_ok(o_col(t) + 32 * cc, 32, 512), wc, kChkTmem, 6)) continue;
            uint32_t o[32];
            tmem_ld_x32(tmem + lane_off + o_col(t) + 32 * cc, o);   // warp-collective: every lane loads
            if (!live) continue;
#pragma unroll
            for (int v4 = 0; v4 < 8; ++v4)
              st_global_v4(orow + 32 * cc + 4 * v4, f2u(u2f(o[4 * v4]) * inv), f2u(u2f(o[4 * v4 + 1]) * inv),
                           f2u(u2f(o[4 * v4 + 2]) * inv), f2u(u2f(o[4 * v4 + 3]) * inv));
          }
          if (live) a.lpart[prow] = lse;
        }
      }
    }
  } else if (warp == kTmaWarp) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tmap(&a.tm_q);
      prefetch_tmap(&a.tm_k);
      prefetch_tmap(&a.tm_v);
      int issued_k[KS] = {}, issued_v[VS] = {};
      const uint32_t tile = (uint32_t)L::kTile;
      const uint32_t qbytes = (n_t[0] > 0 ? tile : 0u) + (n_t[1] > 0 ? tile : 0u);
      const bool have_q = qbytes > 0;
      if (have_q) {
        mbar_arrive_expect_tx(bar(kQFull), qbytes);
        for (int t = 0; t < 2; ++t)
          if (n_t[t] > 0)
            for (int b = 0; b < D / 64; ++b)
              load_rows(sbase + L::kQ + t * L::kTile + b * kBoxBytes, &a.tm_q, bar(kQFull), 64 * b, q0 + t * kBM, Nq);
      }
      // Tile j goes to K stage j % KS and V stage j % VS; its n-th use of a
      // stage (n = j / stages) completes phase n of that stage's barriers, so a
      // reuse waits for the release of use n − 1 (parity (n − 1) & 1).
      for (int j = 0; j < J; ++j) {
        const int sk = j % KS, sv = j % VS;
        if (j >= KS && !mbar_wait(bar(kKEmpty + sk), (uint32_t)((j / KS - 1) & 1), wc, site(3))) break;
        mbar_arrive_expect_tx(bar(kKFull + sk), tile);
        for (int b = 0; b < D / 64; ++b)
          load_rows(sbase + L::kK + sk * L::kTile + b * kBoxBytes, &a.tm_k, bar(kKFull + sk), 64 * b,
                    (kv_begin + j) * kBN, Nk);
        ++issued_k[sk];
        if (j >= VS && !mbar_wait(bar(kVEmpty + sv), (uint32_t)((j / VS - 1) & 1), wc, site(4))) break;
        mbar_arrive_expect_tx(bar(kVFull + sv), tile);
        for (int b = 0; b < D / 64; ++b)
          load_rows(sbase + L::kV + sv * L::kTile + b * kBoxBytes, &a.tm_v, bar(kVFull + sv), 64 * b,
                    (kv_begin + j) * kBN, Nk);
        ++issued_v[sv];
      }
      // Never leave the CTA with copies in flight: wait for the last load of
      // every stage (already complete in the normal case).
      if (have_q) mbar_wait_drain(bar(kQFull), 0, wc, site(5));
      for (int s = 0; s < KS; ++s)
        if (issued_k[s] > 0) mbar_wait_drain(bar(kKFull + s), (uint32_t)((issued_k[s] - 1) & 1), wc, site(5));
      for (int s = 0; s < VS; ++s)
        if (issued_v[s] > 0) mbar_wait_drain(bar(kVFull + s), (uint32_t)((issued_v[s] - 1) & 1), wc, site(5));
    }
  } else {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_f16kind(128, kBN, false, false, F16);   // S = Q Kᵀ, both K-major
      constexpr uint32_t kIdO = idesc_f16kind(128, DR, false, true, F16);     // O += P V, V is MN-major
      bool ok = J == 0 || mbar_wait(bar(kQFull), 0, wc, site(6));
      int k_ready = -1;
      auto issue_s = [&](int t, int j) -> bool {
        if (k_ready < j) {
          if (!mbar_wait(bar(kKFull + j % KS), (uint32_t)((j / KS) & 1), wc, site(7))) return false;
          k_ready = j;
        }
        tc_fence_after();
        const uint64_t qd = sdesc_sw128(sbase + L::kQ + t * L::kTile, 16, 1024);
        const uint64_t kd = sdesc_sw128(sbase + L::kK + (j % KS) * L::kTile, 16, 1024);
        const uint32_t dcol = tmem + s_col(t);
        const bool chk = dcheck(tmem_ok(s_col(t), kBN, 512), wc, kChkTmem, 7) &&
                         dcheck(smem_ok(L::kQ + t * L::kTile, L::kTile, L::kBar, 1024), wc, kChkSmem, 7) &&
                         dcheck(smem_ok(L::kK + (j % KS) * L::kTile, L::kTile, L::kBar, 1024), wc, kChkSmem, 7);
#pragma unroll
        for (int ks = 0; ks < DR / 16; ++ks) {
          if (!chk) break;
          const uint32_t off = (uint32_t)((ks >> 2) * kBoxBytes + (ks & 3) * 32);
          mma_ss(dcol, sdesc_add(qd, off), sdesc_add(kd, off), kIdS, ks > 0 ? 1u : 0u);
        }
        tc_commit(bar(kSFull + t));
        return true;
      };
      if (ok && J > 0) {
        for (int t = 0; t < 2 && ok; ++t)
          if (n_t[t] > 0) ok = issue_s(t, 0);
        if (ok) tc_commit(bar(kKEmpty + 0));
      }
      for (int j = 0; ok && j < J; ++j) {
        if (!mbar_wait(bar(kVFull + j % VS), (uint32_t)((j / VS) & 1), wc, site(8))) {
          ok = false;
          break;
        }
        const uint64_t vd = sdesc_sw128(sbase + L::kV + (j % VS) * L::kTile, kBoxBytes, 1024);
        for (int t = 0; t < 2 && ok; ++t) {
          if (j >= n_t[t]) continue;
          if (!mbar_wait(bar(kPFull + t), (uint32_t)(j & 1), wc, site(9))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t ocol = tmem + o_col(t), pcol = tmem + s_col(t);
          const bool chk = dcheck(tmem_ok(o_col(t), DR, 512), wc, kChkTmem, 8) &&
                           dcheck(tmem_ok(s_col(t), kBN / 2, 512), wc, kChkTmem, 8) &&
                           dcheck(smem_ok(L::kV + (j % VS) * L::kTile, L::kTile, L::kBar, 1024), wc, kChkSmem, 8);
#pragma unroll
          for (int ks = 0; ks < kBN / 16; ++ks)
            if (chk)
              mma_ts(ocol, pcol + (uint32_t)(8 * ks), sdesc_add(vd, (uint32_t)(ks * 2048)), kIdO,
                     (j > 0 || ks > 0) ? 1u : 0u);
          if (j == n_t[t] - 1) tc_commit(bar(kOFull + t));
          if (j + 1 < n_t[t]) ok = issue_s(t, j + 1);
        }
        if (!ok) break;
        tc_commit(bar(kVEmpty + j % VS));
        if (j + 1 < J) tc_commit(bar(kKEmpty + (j + 1) % KS));
      }
      // Every product must be finished before tensor memory is released.
      tc_commit(bar(kMmaDone));
      mbar_wait_drain(bar(kMmaDone), 0, wc, site(10));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Persistent form of the forward for problems without the mask whose units
// see few K/V tiles (every unit sees all of them; no split): one CTA per SM
// walks the units u = blockIdx.x, blockIdx.x + gridDim.x, ...  The K/V ring,
// the score and P barriers count on across units; the next unit's Q load
// starts as soon as the current unit's last scores are computed (QEmpty),
// its first scores while the softmax warps still write the current unit's
// O, and its first P V product once they have read O out of tensor memory
// (OEmpty).  So a unit's start-up and drain overlap its neighbours' work
// instead of leaving the SM idle between one-unit CTAs.
template <int DR, bool RAGGED, bool F16>
__global__ void __launch_bounds__(kThreads, 1) fa_fwd_bf16_persist_kernel(const __grid_constant__ FwdArgs a) {
  constexpr int D = DR <= 64 ? 64 : 128;
  using L = FwdLayout<D>;
  constexpr int KS = L::kKS, VS = L::kVS;
  using Bar = FwdBars<KS, VS>;
  constexpr int kQFull = Bar::kQFull, kKFull = Bar::kKFull, kKEmpty = Bar::kKEmpty, kVFull = Bar::kVFull,
                kVEmpty = Bar::kVEmpty, kSFull = Bar::kSFull, kPFull = Bar::kPFull, kOFull = Bar::kOFull,
                kMmaDone = Bar::kMmaDone;
  constexpr int kQEmpty = Bar::kNumBars;        // the unit's scores are done: Q may be reloaded
  constexpr int kOEmpty = Bar::kNumBars + 1;    // +tile: O_t has been read out
  constexpr int kNumBars = Bar::kNumBars + 3;
  static_assert(8 * kNumBars + 8 <= 512, "barrier block too small");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t sbase = smem_u32(smem_raw);
  uint8_t* sgen = smem_raw;
  if (sbase & 1023u) {
    if (threadIdx.x == 0) atomicCAS(a.fault, 0u, site(0));
    return;
  }
  const uint32_t bars = sbase + L::kBar;
  auto bar = [&](int i) -> uint32_t { return bars + 8u * (uint32_t)i; };
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sgen + L::kBar + 8 * kNumBars);
  int* abort_flag = reinterpret_cast<int*>(sgen + L::kBar + 8 * kNumBars + 4);
  const WaitCtx wc{abort_flag, a.fault};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int Nq = a.Nq, Nk = a.Nk;
  const int pairs = (Nq + 2 * kBM - 1) / (2 * kBM);      // two-tile units per head
  const int units = a.B * a.H * pairs;
  const int n_kv = (Nk + kBN - 1) / kBN;                 // every unit visits every K/V tile
  const int kv_tail = Nk - (n_kv - 1) * kBN;
  const bool ragged_last = RAGGED && kv_tail < kBN;      // the last tile holds keys past Nk
  // Query tiles of a unit that exist: tile 1 of a head's last pair may not.
  auto tiles_of = [&](int u, int t) -> int { return (u % pairs) * 2 * kBM + t * kBM < Nq ? n_kv : 0; };
  auto load_rows = [&](uint32_t dst, const CUtensorMap* map, uint32_t bar_addr, int x, int pos, int n, int bh) {
    bool chk = dcheck(smem_ok(dst - sbase, kBoxBytes, (uint32_t)L::kBar, 1024), wc, kChkSmem, 11) &&
               dcheck(tma_x_ok(x, 64, D), wc, kChkTmaX, 11);
    if constexpr (RAGGED)
      chk = chk && dcheck(tma_head_ok(pos, n, bh, a.B * a.H), wc, kChkTmaRows, 11);
    else
      chk = chk && dcheck(tma_rows_ok((long long)bh * n + pos, kBM, (long long)a.B * a.H * n), wc, kChkTmaRows, 11);
    if (!chk) {
      mbar_complete_tx(bar_addr, kBoxBytes);
      return;
    }
    if constexpr (RAGGED)
      tma_load_3d(dst, map, bar_addr, x, pos, bh);
    else
      tma_load_2d(dst, map, bar_addr, x, bh * n + pos);
  };

  if (threadIdx.x == 0) {
    mbar_init(bar(kQFull), 1);
    mbar_init(bar(kQEmpty), 1);
    for (int s = 0; s < KS; ++s) {
      mbar_init(bar(kKFull + s), 1);
      mbar_init(bar(kKEmpty + s), 1);
    }
    for (int s = 0; s < VS; ++s) {
      mbar_init(bar(kVFull + s), 1);
      mbar_init(bar(kVEmpty + s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(kSFull + t), 1);
      mbar_init(bar(kPFull + t), 128);
      mbar_init(bar(kOFull + t), 1);
      mbar_init(bar(kOEmpty + t), 128);
    }
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
  auto s_col = [](int t) -> uint32_t { return (uint32_t)(128 * t); };
  auto o_col = [](int t) -> uint32_t { return (uint32_t)(256 + D * t); };

  if (warp < 8) {
    // ------------------------------------------------------------ softmax
    const int t = warp >> 2;
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const float sl2 = a.scale_log2;
    int n_s = 0;      // scores of tile t consumed so far (SFull phases)
    int n_o = 0;      // units of tile t finished so far (OFull / OEmpty phases)
    bool ok = true;
    for (int u = (int)blockIdx.x; ok && u < units; u += (int)gridDim.x) {
      const int nt = tiles_of(u, t);
      if (nt == 0) continue;
      const int bh = u / pairs;
      const int qt = (u % pairs) * 2 * kBM + t * kBM;
      float m_ref = -INFINITY;
      float ell = 0.f;
      for (int j = 0; j < nt; ++j, ++n_s) {
        ok = mbar_wait(bar(kSFull + t), (uint32_t)(n_s & 1), wc, site(12));
        ok = __all_sync(kFull, ok);
        if (!ok) break;
        tc_fence_after();
        uint32_t s[128];
        if (dcheck(tmem_ok(s_col(t), 128, 512), wc, kChkTmem, 12)) tmem_ld_x128(tmem + lane_off + s_col(t), s);
        if (ragged_last && j == nt - 1) {
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c >= kv_tail) s[c] = f2u(-INFINITY);
        }
        float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
        for (int c = 0; c < 128; c += 8) {
          mx0 = max3(mx0, u2f(s[c]), u2f(s[c + 1]));
          mx1 = max3(mx1, u2f(s[c + 2]), u2f(s[c + 3]));
          mx2 = max3(mx2, u2f(s[c + 4]), u2f(s[c + 5]));
          mx3 = max3(mx3, u2f(s[c + 6]), u2f(s[c + 7]));
        }
        const float mx = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * sl2;
        const bool move = mx > m_ref + 8.0f;
        const float m_new = move ? mx : m_ref;
        const float alpha = ex2(m_ref - m_new);
        if (j > 0 && __any_sync(kFull, move)) {
          // The previous P V into O_t has completed (it was issued before
          // these scores) and the next one waits for P_full: O_t is ours.
#pragma unroll
          for (int cc = 0; cc < DR / 32; ++cc) {
            if (!dcheck(tmem_ok(o_col(t) + 32 * cc, 32, 512), wc, kChkTmem, 13)) continue;
            uint32_t o[32];
            tmem_ld_x32(tmem + lane_off + o_col(t) + 32 * cc, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = f2u(u2f(o[i]) * alpha);
            tmem_st_x32(tmem + lane_off + o_col(t) + 32 * cc, o);
          }
        }
        ell *= alpha;
        m_ref = m_new;
        const uint32_t p_addr = tmem + lane_off + s_col(t);
        if (!dcheck(tmem_ok(s_col(t), kBN / 2, 512), wc, kChkTmem, 14)) {
        } else if (ragged_last && j == nt - 1)
          ell += exp_tile_to_p<0, F16>(s, sl2, m_ref, p_addr);
        else
          ell += exp_tile_to_p<kPolyEvery, F16>(s, sl2, m_ref, p_addr);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(kPFull + t));
      }
      if (!ok) break;
      // Epilogue of this unit's tile: O = Õ / ℓ and LSE; O_t is released to
      // the next unit's first P V as soon as it has been read.
      ok = mbar_wait(bar(kOFull + t), (uint32_t)(n_o & 1), wc, site(13));
      ok = __all_sync(kFull, ok);
      if (!ok) break;
      tc_fence_after();
      const int q = qt + r;
      const float inv = 1.0f / ell;
      const float lse = (m_ref + log2f(ell)) * 0.69314718055994530942f;
      const bool live = !RAGGED || q < Nq;
      uint16_t* orow = static_cast<uint16_t*>(a.o) + ((size_t)bh * (size_t)Nq + (size_t)q) * DR;
#pragma unroll
      for (int cc = 0; cc < DR / 32; ++cc) {
        if (!dcheck(tmem_ok(o_col(t) + 32 * cc, 32, 512), wc, kChkTmem, 15)) continue;
        uint32_t o[32];
        tmem_ld_x32(tmem + lane_off + o_col(t) + 32 * cc, o);   // warp-collective: every lane loads
        if (cc == DR / 32 - 1) {
          tc_fence_before();
          mbar_arrive(bar(kOEmpty + t));
        }
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) pk[i] = pack2<F16>(u2f(o[2 * i]) * inv, u2f(o[2 * i + 1]) * inv);
        if (live) {
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4)
            st_global_v4(orow + 32 * cc + 8 * v4, pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
        }
      }
      if (live) a.lse[(size_t)bh * (size_t)Nq + (size_t)q] = lse;
      ++n_o;
    }
  } else if (warp == kTmaWarp) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tmap(&a.tm_q);
      prefetch_tmap(&a.tm_k);
      prefetch_tmap(&a.tm_v);
      const uint32_t tile = (uint32_t)L::kTile;
      int g = 0;                      // K/V tiles issued so far, over all units
      int n_q = 0;                    // Q loads issued
      int issued_k[KS] = {}, issued_v[VS] = {};
      bool ok = true;
      for (int u = (int)blockIdx.x; ok && u < units; u += (int)gridDim.x) {
        const int bh = u / pairs;
        const int q0 = (u % pairs) * 2 * kBM;
        const int nt1 = tiles_of(u, 1);
        for (int j = 0; j < n_kv; ++j, ++g) {
          // Tile g goes to K stage g % KS (its use g / KS) and V stage g % VS.
          const int sk = g % KS, sv = g % VS;
          if (g >= KS && !mbar_wait(bar(kKEmpty + sk), (uint32_t)((g / KS - 1) & 1), wc, site(14))) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar(kKFull + sk), tile);
          for (int b = 0; b < D / 64; ++b)
            load_rows(sbase + L::kK + sk * L::kTile + b * kBoxBytes, &a.tm_k, bar(kKFull + sk), 64 * b, j * kBN, Nk,
                      bh);
          ++issued_k[sk];
          if (j == 0) {
            // Q of this unit once the previous unit's scores have all been computed.
            if (n_q > 0 && !mbar_wait(bar(kQEmpty), (uint32_t)((n_q - 1) & 1), wc, site(15))) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(bar(kQFull), (nt1 > 0 ? 2u : 1u) * tile);
            for (int t = 0; t < (nt1 > 0 ? 2 : 1); ++t)
              for (int b = 0; b < D / 64; ++b)
                load_rows(sbase + L::kQ + t * L::kTile + b * kBoxBytes, &a.tm_q, bar(kQFull), 64 * b, q0 + t * kBM,
                          Nq, bh);
            ++n_q;
          }
          if (g >= VS && !mbar_wait(bar(kVEmpty + sv), (uint32_t)((g / VS - 1) & 1), wc, site(16))) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar(kVFull + sv), tile);
          for (int b = 0; b < D / 64; ++b)
            load_rows(sbase + L::kV + sv * L::kTile + b * kBoxBytes, &a.tm_v, bar(kVFull + sv), 64 * b, j * kBN, Nk,
                      bh);
          ++issued_v[sv];
        }
      }
      // Never leave the CTA with copies in flight: wait for the last load of
      // every barrier (already complete in the normal case).
      if (n_q > 0) mbar_wait_drain(bar(kQFull), (uint32_t)((n_q - 1) & 1), wc, site(17));
      for (int s = 0; s < KS; ++s)
        if (issued_k[s] > 0) mbar_wait_drain(bar(kKFull + s), (uint32_t)((issued_k[s] - 1) & 1), wc, site(17));
      for (int s = 0; s < VS; ++s)
        if (issued_v[s] > 0) mbar_wait_drain(bar(kVFull + s), (uint32_t)((issued_v[s] - 1) & 1), wc, site(17));
    }
  } else {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_f16kind(128, kBN, false, false, F16);
      constexpr uint32_t kIdO = idesc_f16kind(128, DR, false, true, F16);
      int g = 0;                  // K/V tiles consumed so far, over all units
      int n_q = 0;                // units started (QFull / QEmpty phases)
      int n_p[2] = {0, 0};        // P of tile t consumed (PFull phases)
      int n_o[2] = {0, 0};        // units of tile t finished (OFull / OEmpty phases)
      int k_ready = -1;           // last K tile (global index) seen complete
      bool ok = true;
      auto issue_s = [&](int t, int gk) -> bool {
        if (k_ready < gk) {
          if (!mbar_wait(bar(kKFull + gk % KS), (uint32_t)((gk / KS) & 1), wc, site(18))) return false;
          k_ready = gk;
        }
        tc_fence_after();
        const uint64_t qd = sdesc_sw128(sbase + L::kQ + t * L::kTile, 16, 1024);
        const uint64_t kd = sdesc_sw128(sbase + L::kK + (gk % KS) * L::kTile, 16, 1024);
        const bool chk = dcheck(tmem_ok(s_col(t), kBN, 512), wc, kChkTmem, 16) &&
                         dcheck(smem_ok(L::kQ + t * L::kTile, L::kTile, L::kBar, 1024), wc, kChkSmem, 16) &&
                         dcheck(smem_ok(L::kK + (gk % KS) * L::kTile, L::kTile, L::kBar, 1024), wc, kChkSmem, 16);
#pragma unroll
        for (int ks = 0; ks < DR / 16; ++ks) {
          if (!chk) break;
          const uint32_t off = (uint32_t)((ks >> 2) * kBoxBytes + (ks & 3) * 32);
          mma_ss(tmem + s_col(t), sdesc_add(qd, off), sdesc_add(kd, off), kIdS, ks > 0 ? 1u : 0u);
        }
        tc_commit(bar(kSFull + t));
        return true;
      };
      for (int u = (int)blockIdx.x; ok && u < units; u += (int)gridDim.x, g += n_kv, ++n_q) {
        const int nt[2] = {tiles_of(u, 0), tiles_of(u, 1)};
        const int t_last = nt[1] > 0 ? 1 : 0;        // the tile whose last scores finish the unit's use of Q
        if (!mbar_wait(bar(kQFull), (uint32_t)(n_q & 1), wc, site(19))) {
          ok = false;
          break;
        }
        for (int t = 0; t < 2 && ok; ++t)
          if (nt[t] > 0) ok = issue_s(t, g);
        if (!ok) break;
        if (n_kv == 1) tc_commit(bar(kQEmpty));
        tc_commit(bar(kKEmpty + g % KS));
        for (int j = 0; ok && j < n_kv; ++j) {
          const int gj = g + j;
          if (!mbar_wait(bar(kVFull + gj % VS), (uint32_t)((gj / VS) & 1), wc, site(20))) {
            ok = false;
            break;
          }
          const uint64_t vd = sdesc_sw128(sbase + L::kV + (gj % VS) * L::kTile, kBoxBytes, 1024);
          for (int t = 0; t < 2 && ok; ++t) {
            if (nt[t] == 0) continue;
            if (!mbar_wait(bar(kPFull + t), (uint32_t)(n_p[t] & 1), wc, site(21))) {
              ok = false;
              break;
            }
            ++n_p[t];
            // The first product into O_t overwrites it: the previous unit's
            // epilogue must have read it out.
            if (j == 0 && n_o[t] > 0 && !mbar_wait(bar(kOEmpty + t), (uint32_t)((n_o[t] - 1) & 1), wc, site(22))) {
              ok = false;
              break;
            }
            tc_fence_after();
            const bool chk = dcheck(tmem_ok(o_col(t), DR, 512), wc, kChkTmem, 17) &&
                             dcheck(tmem_ok(s_col(t), kBN / 2, 512), wc, kChkTmem, 17) &&
                             dcheck(smem_ok(L::kV + (gj % VS) * L::kTile, L::kTile, L::kBar, 1024), wc, kChkSmem, 17);
#pragma unroll
            for (int ks = 0; ks < kBN / 16; ++ks)
              if (chk)
                mma_ts(tmem + o_col(t), tmem + s_col(t) + (uint32_t)(8 * ks), sdesc_add(vd, (uint32_t)(ks * 2048)),
                       kIdO, (j > 0 || ks > 0) ? 1u : 0u);
            if (j == n_kv - 1) tc_commit(bar(kOFull + t));
            if (j + 1 < n_kv) {
              ok = issue_s(t, gj + 1);
              if (ok && t == t_last && j + 2 == n_kv) tc_commit(bar(kQEmpty));
            }
          }
          if (!ok) break;
          tc_commit(bar(kVEmpty + gj % VS));
          if (j + 1 < n_kv) tc_commit(bar(kKEmpty + (gj + 1) % KS));
        }
        for (int t = 0; t < 2; ++t)
          if (nt[t] > 0) ++n_o[t];
      }
      // Every product must be finished before tensor memory is released.
      tc_commit(bar(kMmaDone));
      mbar_wait_drain(bar(kMmaDone), 0, wc, site(23));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int DR, bool RAGGED, bool F16>
cudaError_t launch_persist(const FwdArgs& a, cudaStream_t s) {
  auto kern = fa_fwd_bf16_persist_kernel<DR, RAGGED, F16>;
  const size_t smem = FwdLayout<(DR <= 64 ? 64 : 128)>::kBytes;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)a.persist_ctas, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

template <int DR, bool CAUSAL, bool RAGGED, bool F16>
cudaError_t launch_impl(const FwdArgs& a, cudaStream_t s) {
  auto kern = fa_fwd_bf16_kernel<DR, CAUSAL, RAGGED, F16>;
  const size_t smem = FwdLayout<(DR <= 64 ? 64 : 128)>::kBytes;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const long long units = (long long)fwd_units(a.B, a.H, a.Nq, DR);
  const long long ctas = a.splits > 1 ? a.n_full + (units - a.n_full) * a.splits : units;
  kern<<<(unsigned)ctas, kThreads, smem, s>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess || a.splits <= 1 || a.n_full >= units) return e;
  return launch_fwd_combine(a, (int)(units - a.n_full), 2 * kBM, s);
}

// Merge of the split partials, "Flash Attention" tutorial, 2.Online Softmax
// §3.1/§4.1 and §七 (the merge is log-sum-exp): for one query row with
// partials (O_k, L_k) over disjoint key ranges, L = ln Σ_k e^{L_k} and
// O = Σ_k e^{L_k − L} O_k.  One warp per row; lanes over the head dims.
// A work unit covers `unit_rows` query rows of one head (256 for the
// two-tile kernel, 128 at d = 256); partial row p of unit slot u·splits + k
// is opart row (u·splits + k)·part_rows + p, for the part_rows ≤ unit_rows
// rows a slot holds.
template <int DR, bool F16>
__global__ void __launch_bounds__(256) fwd_combine_kernel(const float* __restrict__ opart,
                                                          const float* __restrict__ lpart, uint16_t* __restrict__ o,
                                                          float* __restrict__ lse, int Nq, int n_full, int splits,
                                                          int tail, int unit_rows, int part_rows) {
  constexpr int V = DR / 32;   // consecutive head dims per lane
  const int row = (int)(blockIdx.x * 8 + (threadIdx.x >> 5));
  const int lane = threadIdx.x & 31;
  if (row >= tail * part_rows) return;
  const int u = row / part_rows, rr = row % part_rows;
  const int per_head = (Nq + unit_rows - 1) / unit_rows;
  const int unit = n_full + u;
  const int q = (unit % per_head) * unit_rows + rr;
  if (q >= Nq) return;
  const size_t orow = (size_t)(unit / per_head) * Nq + (size_t)q;
  float mx = -INFINITY;
  for (int k = 0; k < splits; ++k) mx = fmaxf(mx, lpart[(size_t)(u * splits + k) * part_rows + rr]);
  float sum = 0.f;
  for (int k = 0; k < splits; ++k) sum += expf(lpart[(size_t)(u * splits + k) * part_rows + rr] - mx);
  const float total = mx + logf(sum);
  float acc[V];
#pragma unroll
  for (int v = 0; v < V; ++v) acc[v] = 0.f;
  for (int k = 0; k < splits; ++k) {
    const size_t pr = (size_t)(u * splits + k) * part_rows + rr;
    const float w = expf(lpart[pr] - total);
    const float* src = opart + pr * DR + lane * V;
#pragma unroll
    for (int v = 0; v < V; ++v) acc[v] = fmaf(w, src[v], acc[v]);
  }
  uint16_t* dst = o + orow * DR + lane * V;
  if constexpr (V % 2 == 0) {
#pragma unroll
    for (int v = 0; v < V; v += 2) reinterpret_cast<uint32_t*>(dst)[v / 2] = pack2<F16>(acc[v], acc[v + 1]);
  } else {   // an odd count per lane (DR = 96): 16-bit stores
#pragma unroll
    for (int v = 0; v < V; ++v) dst[v] = (uint16_t)(pack2<F16>(acc[v], 0.f) & 0xFFFFu);
  }
  if (lane == 0) lse[orow] = total;
}

template <int DR, bool F16>
cudaError_t combine_impl(const FwdArgs& a, int tail, int unit_rows, cudaStream_t s) {
  const int rows = tail * a.part_rows;
  fwd_combine_kernel<DR, F16><<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(
      a.opart, a.lpart, static_cast<uint16_t*>(a.o), a.lse, a.Nq, a.n_full, a.splits, tail, unit_rows, a.part_rows);
  return cudaGetLastError();
}

template <bool F16>
cudaError_t combine_dispatch(const FwdArgs& a, int tail, int unit_rows, cudaStream_t s) {
  switch (a.d) {
    case 64: return combine_impl<64, F16>(a, tail, unit_rows, s);
    case 96: return combine_impl<96, F16>(a, tail, unit_rows, s);
    case 128: return combine_impl<128, F16>(a, tail, unit_rows, s);
    case 256: return combine_impl<256, F16>(a, tail, unit_rows, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

int fwd_unit_rows(int d) { return d == 256 ? kBM : 2 * kBM; }

int fwd_units(int B, int H, int Nq, int d) {
  const int rows = fwd_unit_rows(d);
  return B * H * ((Nq + rows - 1) / rows);
}

cudaError_t launch_fwd_combine(const FwdArgs& a, int tail, int unit_rows, cudaStream_t s) {
  return a.f16 ? combine_dispatch<true>(a, tail, unit_rows, s) : combine_dispatch<false>(a, tail, unit_rows, s);
}

void fwd_split_plan(int units, int num_sms, int n_kv, int* n_full, int* splits) {
  *n_full = units;
  *splits = 1;
  if (num_sms <= 0 || units <= 0) return;
  const int tail = units % num_sms;
  if (tail == 0) return;
  int s = num_sms / tail;         // CTAs per tail unit that still fit in one wave
  // Up to 4 parts for the last wave of a multi-wave grid; when every unit
  // fits in one partial wave (few heads, long K/V: decoding), up to 16, so
  // that the K/V reads spread over more SMs.
  const int cap = units < num_sms ? 16 : 4;
  if (s > cap) s = cap;
  // Each part must keep at least 8 K/V tiles: shorter parts cost more in
  // per-CTA start-up, fp32 partial writes and the merge than they save
  // (measured on GB300 with 8 tiles per unit split in two).
  while (s > 1 && n_kv / s < 8) --s;
  if (s < 2) return;
  *splits = s;
  *n_full = units - tail;
}

int fwd_split_short(int units, int num_sms, int n_kv) {
  // Parts of at least 8 K/V tiles (shorter ones cost more in start-up than
  // they spread) and at most 16; among those, the count whose grid fills its
  // last wave best, with fewer than two waves weighed down (the CTAs of one
  // wave finish at different times too); ties (within 1 %) go to fewer parts.
  if (num_sms <= 0 || units <= 0) return 1;
  int best = 1;
  double best_score = -1.0;
  for (int s = 1; s <= 16 && n_kv / s >= 8; ++s) {
    const double waves = (double)units * s / num_sms;
    double score = waves / std::ceil(waves);
    if (waves < 2.0) score *= waves / 2.0;
    if (score > best_score * 1.01) {
      best_score = score;
      best = s;
    }
  }
  return best;
}

size_t fwd_bf16_smem_bytes(int d) {
  return d <= 64 ? FwdLayout<64>::kBytes : FwdLayout<128>::kBytes;
}

template <bool F16>
static cudaError_t dispatch_fwd(const FwdArgs& a, bool ragged, cudaStream_t s) {
  if (a.persist_ctas > 0 && !a.causal && a.splits <= 1) {
    switch (a.d) {
      case 128: return ragged ? launch_persist<128, true, F16>(a, s) : launch_persist<128, false, F16>(a, s);
      case 96: return ragged ? launch_persist<96, true, F16>(a, s) : launch_persist<96, false, F16>(a, s);
      case 64: return ragged ? launch_persist<64, true, F16>(a, s) : launch_persist<64, false, F16>(a, s);
    }
    return cudaErrorInvalidValue;
  }
  if (a.d == 128) {
    if (ragged) return a.causal ? launch_impl<128, true, true, F16>(a, s) : launch_impl<128, false, true, F16>(a, s);
    return a.causal ? launch_impl<128, true, false, F16>(a, s) : launch_impl<128, false, false, F16>(a, s);
  }
  if (a.d == 96) {
    if (ragged) return a.causal ? launch_impl<96, true, true, F16>(a, s) : launch_impl<96, false, true, F16>(a, s);
    return a.causal ? launch_impl<96, true, false, F16>(a, s) : launch_impl<96, false, false, F16>(a, s);
  }
  if (a.d == 64) {
    if (ragged) return a.causal ? launch_impl<64, true, true, F16>(a, s) : launch_impl<64, false, true, F16>(a, s);
    return a.causal ? launch_impl<64, true, false, F16>(a, s) : launch_impl<64, false, false, F16>(a, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_fwd_bf16(const FwdArgs& a, cudaStream_t s) {
  if (a.d == 256) return launch_fwd_d256(a, s);
  const bool ragged = a.Nq % kBM != 0 || a.Nk % kBN != 0;
  if (a.f16) return dispatch_fwd<true>(a, ragged, s);
  return dispatch_fwd<false>(a, ragged, s);
}

}  // namespace fa
