// fa_fwd_d256.cu — tiled attention forward for head dimension 256 on the
// sm_103a tensor cores.
//
// What it computes is what fa_fwd_bf16.cu computes ("Flash Attention"
// tutorial, 2.Online Softmax §4.2: one pass over K/V tiles with the running
// (m, ℓ) and the unnormalised Õ, divided by ℓ at the end; LSE = m + ln ℓ as
// in 3.Recomputation 三); only the tiling differs.
//
// At d = 256 the fp32 output accumulator of one 128-row query tile fills half
// of the 512 tensor-memory columns, so a CTA owns ONE query tile and spends
// the other half on two score buffers:
//   S_b = cols [128 b, 128 b + 128)  (b = j mod 2); P_j (16-bit) over its first 64
//   O   = cols [256, 512)
// The MMA thread issues S_0, S_1, PV_0, S_2, PV_1, ...: the scores of tile
// j + 1 are computed while the softmax works on tile j, and S_{j+2} reuses
// the buffer of P_j right after PV_j has been issued (products run in issue
// order).
//
// Shared memory (226 KB): Q resident (four boxes of 64 head dims × 128 rows,
// 16 KB each), K through a ring of six such boxes (a box is released as soon
// as the four K-steps that read it have completed, so the next tile's K
// streams in box by box), V in one 64 KB slot.
//
// Warps 0-7 run the softmax: thread (w, lane) owns row 32(w mod 4) + lane and
// key columns 64⌊w/4⌋ .. +63 of each tile.  The two threads of a row swap
// their partial maxima through shared memory every tile, so both hold the
// same reference max; they keep separate partial sums ℓ (added once at the
// end) and each rescales and stores its own half of the output columns.
// Warp 8 issues TMA, warp 9 the MMAs and owns tensor memory.
#include "fa_kernels.h"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

constexpr int kD = 256;
constexpr int kBM = 128;          // query rows per CTA
constexpr int kBN = 128;          // keys per K/V tile
constexpr int kThreads = 320;
constexpr int kTmaWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kBox = 16384;       // one TMA box: 128 rows × 128 bytes
constexpr int kKSlots = 6;        // K ring, in boxes

// Shared-memory layout (offsets from a 1024-byte aligned base).
constexpr int kQ = 0;                               // 4 boxes
constexpr int kK = kQ + 4 * kBox;                   // kKSlots boxes
constexpr int kV = kK + kKSlots * kBox;             // 4 boxes
constexpr int kXch = kV + 4 * kBox;                 // fp32 [2 parities][2 halves][128 rows]
constexpr int kBar = kXch + 2 * 2 * kBM * 4;
constexpr int kSmemBytes = kBar + 256;

enum Bar : int {
  kQFull = 0,
  kKFull = 1,                     // + ring slot
  kKEmpty = kKFull + kKSlots,     // + ring slot
  kVFull = kKEmpty + kKSlots,
  kVEmpty,
  kSFull,                         // + score buffer (2)
  kPFull = kSFull + 2,            // + score buffer (2)
  kPVDone = kPFull + 2,           // one phase per O += P_j V_j
  kOFull,                         // the last O += P V has completed
  kMmaDone,
  kNumBars,
};
static_assert(8 * kNumBars + 8 <= 256, "barrier block too small");
static_assert(kSmemBytes <= 232448, "shared memory exceeds the 227 KB a CTA may use");

// Fault codes recorded when a wait runs out of time (kernel id 3 in the high byte).
__device__ __forceinline__ uint32_t site(int s) { return 0x0300u | (uint32_t)s; }

// P = 2^(s·scale·log2e − m) for 64 columns of one row, rounded to the 16-bit
// type and stored at `p_addr` (32 tensor-memory columns); returns Σ P in fp32.
template <bool F16>
__device__ __forceinline__ float exp_half_to_p(const uint32_t (&s)[64], float sl2, float m_ref, uint32_t p_addr) {
  const uint64_t sl2x2 = f2_pack(sl2, sl2);
  const uint64_t negx2 = f2_pack(-m_ref, -m_ref);
  uint64_t lsum0 = f2_pack(0.f, 0.f), lsum1 = lsum0;
#pragma unroll
  for (int cc = 0; cc < 2; ++cc) {
    uint32_t p[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint64_t x = f2_fma(f2_pack(u2f(s[32 * cc + 2 * i]), u2f(s[32 * cc + 2 * i + 1])), sl2x2, negx2);
      float x0, x1;
      f2_unpack(x, x0, x1);
      const float e0 = ex2(x0), e1 = ex2(x1);
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
// row-predicated stores.  F16: fp16 inputs and outputs (else bf16).
template <bool CAUSAL, bool RAGGED, bool F16>
__global__ void __launch_bounds__(kThreads, 1) fa_fwd_d256_kernel(const __grid_constant__ FwdArgs a) {
  // Dynamic shared memory starts on a 1024-byte boundary (no static shared
  // memory is declared); 128-byte swizzled tiles need that alignment.
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
  const int off = Nk - Nq;                       // causal: query i sees keys j ≤ i + off
  const int tiles = (Nq + kBM - 1) / kBM;        // query tiles (work units) per head
  // Work of this CTA (1-D grid), as in the two-tile kernel: causal grids put
  // batch·head fastest and the heaviest tiles first; non-causal grids are
  // head-major, and the units of the last partial wave are split into
  // `splits` CTAs over equal K/V sub-ranges that write fp32 partials.
  const int n_kv_all = (Nk + kBN - 1) / kBN;
  int bh, tile, kv_begin = 0, n_kv = n_kv_all, part_slot = -1;
  const int idx = (int)blockIdx.x;
  if (CAUSAL) {
    bh = idx % (a.B * a.H);
    tile = tiles - 1 - idx / (a.B * a.H);
  } else if (idx < a.n_full) {
    bh = idx / tiles;
    tile = idx % tiles;
  } else {
    part_slot = idx - a.n_full;
    const int unit = a.n_full + part_slot / a.splits;
    const int part = part_slot % a.splits;
    bh = unit / tiles;
    tile = unit % tiles;
    kv_begin = part * n_kv / a.splits;
    n_kv = (part + 1) * n_kv / a.splits - kv_begin;
  }
  const int q0 = tile * kBM;
  const int row0 = bh * Nq;
  const int kv_tail = Nk - (n_kv_all - 1) * kBN;   // keys of the head's last tile that exist
  const bool ragged_last = RAGGED && !CAUSAL && kv_tail < kBN && kv_begin + n_kv == n_kv_all;
  // A debug build checks each box's destination and coordinates first and, if
  // a check fails, completes its bytes on the barrier without copying.
  auto load_rows = [&](uint32_t dst, const CUtensorMap* map, uint32_t bar_addr, int x, int pos, int n) {
    bool chk = dcheck(smem_ok(dst - sbase, kBox, (uint32_t)kBar, 1024), wc, kChkSmem, 32) &&
               dcheck(tma_x_ok(x, 64, kD), wc, kChkTmaX, 32);
    if constexpr (RAGGED)
      chk = chk && dcheck(tma_head_ok(pos, n, bh, a.B * a.H), wc, kChkTmaRows, 32);
    else
      chk = chk && dcheck(tma_rows_ok((long long)bh * n + pos, kBM, (long long)a.B * a.H * n), wc, kChkTmaRows, 32);
    if (!chk) {
      mbar_complete_tx(bar_addr, kBox);
      return;
    }
    if constexpr (RAGGED)
      tma_load_3d(dst, map, bar_addr, x, pos, bh);
    else
      tma_load_2d(dst, map, bar_addr, x, bh * n + pos);
  };
  // K/V tiles visited and, under the causal mask, the first one that masks
  // some score (tile j holds keys 128j + c, visible to row q0 + r iff
  // c ≤ r + q0 + off − 128j).
  const int last_key = (q0 + kBM - 1 < Nq ? q0 + kBM - 1 : Nq - 1) + off;
  const int J = CAUSAL ? last_key / kBN + 1 : n_kv;
  const int fm = (q0 + off + 1) / kBN;

  if (threadIdx.x == 0) {
    mbar_init(bar(kQFull), 1);
    for (int s = 0; s < kKSlots; ++s) {
      mbar_init(bar(kKFull + s), 1);
      mbar_init(bar(kKEmpty + s), 1);
    }
    mbar_init(bar(kVFull), 1);
    mbar_init(bar(kVEmpty), 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(kSFull + b), 1);
      mbar_init(bar(kPFull + b), 256);
    }
    mbar_init(bar(kPVDone), 1);
    mbar_init(bar(kOFull), 1);
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
    // ------------------------------------------------------------ softmax
    const int c = warp >> 2;                     // key columns [64c, 64c + 64), output columns [128c, 128c + 128)
    const int g = warp & 3;
    const int r = g * 32 + lane;                 // row within the tile = TMEM lane
    const uint32_t lane_off = (uint32_t)(g * 32) << 16;
    float* xch = reinterpret_cast<float*>(sgen + kXch);   // [parity][half][row]
    const float sl2 = a.scale_log2;
    float m_ref = -INFINITY;   // reference max of the row, base-2 scaled units (same in both halves)
    float ell = 0.f;           // this half's partial sum
    bool ok = true;
    // Never leave the loop except right after the pair barrier, so that both
    // warps of a lane quarter always meet at the same barriers.
    for (int j = 0; j < J; ++j) {
      const int b = j & 1;
      bool okj = ok && mbar_wait(bar(kSFull + b), (uint32_t)((j >> 1) & 1), wc, site(1));
      okj = __all_sync(kFull, okj);
      uint32_t s[64];
      float mxh = -INFINITY;
      if (okj) {
        tc_fence_after();
        if (dcheck(tmem_ok(128u * b + 64u * c, 64, 512), wc, kChkTmem, 33))
          tmem_ld_x64(tmem + lane_off + 128u * (uint32_t)b + 64u * (uint32_t)c, s);
        if (CAUSAL && j >= fm) {
          const int lim = r + q0 + off - j * kBN - 64 * c;
#pragma unroll
          for (int cc = 0; cc < 64; ++cc)
            if (cc > lim) s[cc] = f2u(-INFINITY);
        }
        if (ragged_last && j == J - 1) {
          const int lim = kv_tail - 64 * c;
#pragma unroll
          for (int cc = 0; cc < 64; ++cc)
            if (cc >= lim) s[cc] = f2u(-INFINITY);
        }
        float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
        for (int cc = 0; cc < 64; cc += 8) {
          mx0 = max3(mx0, u2f(s[cc]), u2f(s[cc + 1]));
          mx1 = max3(mx1, u2f(s[cc + 2]), u2f(s[cc + 3]));
          mx2 = max3(mx2, u2f(s[cc + 4]), u2f(s[cc + 5]));
          mx3 = max3(mx3, u2f(s[cc + 6]), u2f(s[cc + 7]));
        }
        mxh = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * sl2;
      }
      // Both halves of the row have read their scores (so P may now be
      // written over them) and published their partial maxima.
      xch[(b * 2 + c) * kBM + r] = mxh;
      ok = named_bar_and(1 + g, 64, okj);
      if (!ok) break;
      const float mx = fmaxf(mxh, xch[(b * 2 + (1 - c)) * kBM + r]);
      const bool move = mx > m_ref + 8.0f;             // always true on the first tile
      const float m_new = move ? mx : m_ref;
      const float alpha = ex2(m_ref - m_new);          // 0 on the first tile, 1 if the reference stays
      if (j > 0 && __any_sync(kFull, move)) {
        // O += P_{j-1} V_{j-1} was issued after this tile's scores: wait for
        // it before rescaling this half of O.  (The scores of tile j were
        // issued after O += P_{j-2} V_{j-2}, so the barrier is at most one
        // phase behind the one awaited.)
        bool okw = mbar_wait(bar(kPVDone), (uint32_t)((j - 1) & 1), wc, site(2));
        okw = __all_sync(kFull, okw);
        if (okw) {
          tc_fence_after();
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            uint32_t o[32];
            const uint32_t col = 256u + 128u * (uint32_t)c + 32u * (uint32_t)cc;
            if (!dcheck(tmem_ok(col, 32, 512), wc, kChkTmem, 34)) continue;
            tmem_ld_x32(tmem + lane_off + col, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = f2u(u2f(o[i]) * alpha);
            tmem_st_x32(tmem + lane_off + col, o);
          }
        } else {
          ok = false;   // the next pair barrier takes both warps out of the loop
          continue;
        }
      }
      ell *= alpha;
      m_ref = m_new;
      if (dcheck(tmem_ok(128u * b + 32u * c, 32, 512), wc, kChkTmem, 35))
        ell += exp_half_to_p<F16>(s, sl2, m_ref, tmem + lane_off + 128u * (uint32_t)b + 32u * (uint32_t)c);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(kPFull + b));
    }
    // ℓ of the row = the two partial sums (same reference max), swapped
    // through the parity buffer the last tile did not use.
    const int pb = J & 1;
    xch[(pb * 2 + c) * kBM + r] = ell;
    ok = named_bar_and(1 + g, 64, ok);
    if (ok) {
      const float ell_all = ell + xch[(pb * 2 + (1 - c)) * kBM + r];
      bool okw = mbar_wait(bar(kOFull), 0, wc, site(3));
      okw = __all_sync(kFull, okw);
      if (okw) {
        tc_fence_after();
        const int q = q0 + r;
        const float inv = 1.0f / ell_all;
        const float lse = (m_ref + log2f(ell_all)) * 0.69314718055994530942f;
        if (part_slot < 0) {
          // tcgen05.ld is warp-collective: every lane loads, and only rows
          // below Nq are stored.
          const bool live = !RAGGED || q < Nq;
          uint16_t* orow = static_cast<uint16_t*>(a.o) + ((size_t)row0 + (size_t)q) * kD + 128 * c;
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            uint32_t o[32];
            if (!dcheck(tmem_ok(256u + 128u * c + 32u * cc, 32, 512), wc, kChkTmem, 36)) continue;
            tmem_ld_x32(tmem + lane_off + 256u + 128u * (uint32_t)c + 32u * (uint32_t)cc, o);
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) pk[i] = pack2<F16>(u2f(o[2 * i]) * inv, u2f(o[2 * i + 1]) * inv);
            if (live) {
#pragma unroll
              for (int v4 = 0; v4 < 4; ++v4)
                st_global_v4(orow + 32 * cc + 8 * v4, pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
            }
          }
          if (live && c == 0) a.lse[(size_t)row0 + (size_t)q] = lse;
        } else {
          // Partial over this CTA's keys: normalised O and LSE in fp32.
          const bool live_part = r < a.part_rows && q < Nq;
          const size_t prow = (size_t)part_slot * (size_t)a.part_rows + (size_t)r;
          float* orow = a.opart + prow * kD + 128 * c;
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            uint32_t o[32];
            if (!dcheck(tmem_ok(256u + 128u * c + 32u * cc, 32, 512), wc, kChkTmem, 36)) continue;
            tmem_ld_x32(tmem + lane_off + 256u + 128u * (uint32_t)c + 32u * (uint32_t)cc, o);   // warp-collective
            if (!live_part) continue;
#pragma unroll
            for (int v4 = 0; v4 < 8; ++v4)
              st_global_v4(orow + 32 * cc + 4 * v4, f2u(u2f(o[4 * v4]) * inv), f2u(u2f(o[4 * v4 + 1]) * inv),
                           f2u(u2f(o[4 * v4 + 2]) * inv), f2u(u2f(o[4 * v4 + 3]) * inv));
          }
          if (c == 0 && live_part) a.lpart[prow] = lse;
        }
      }
    }
  } else if (warp == kTmaWarp) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tmap(&a.tm_q);
      prefetch_tmap(&a.tm_k);
      prefetch_tmap(&a.tm_v);
      mbar_arrive_expect_tx(bar(kQFull), 4u * kBox);
      for (int bx = 0; bx < 4; ++bx) load_rows(sbase + kQ + bx * kBox, &a.tm_q, bar(kQFull), 64 * bx, q0, Nq);
      int k_boxes = 0, v_tiles = 0;
      // K box 4j + bx goes to ring slot (4j + bx) mod 6 once the box six
      // places earlier has been read.
      auto load_k = [&](int j) -> bool {
        for (int bx = 0; bx < 4; ++bx) {
          const int gi = 4 * j + bx, slot = gi % kKSlots, round = gi / kKSlots;
          if (round > 0 && !mbar_wait(bar(kKEmpty + slot), (uint32_t)((round - 1) & 1), wc, site(4))) return false;
          mbar_arrive_expect_tx(bar(kKFull + slot), kBox);
          load_rows(sbase + kK + slot * kBox, &a.tm_k, bar(kKFull + slot), 64 * bx, (kv_begin + j) * kBN, Nk);
          ++k_boxes;
        }
        return true;
      };
      auto load_v = [&](int j) -> bool {
        if (j > 0 && !mbar_wait(bar(kVEmpty), (uint32_t)((j - 1) & 1), wc, site(5))) return false;
        mbar_arrive_expect_tx(bar(kVFull), 4u * kBox);
        for (int bx = 0; bx < 4; ++bx)
          load_rows(sbase + kV + bx * kBox, &a.tm_v, bar(kVFull), 64 * bx, (kv_begin + j) * kBN, Nk);
        ++v_tiles;
        return true;
      };
      // K runs one tile ahead of V (K_0, K_1, V_0, K_2, V_1, ...), matching
      // the MMA order S_0, S_1, PV_0, S_2, PV_1: each load waits only for a
      // product that is issued before the one that needs the load.
      bool ok = load_k(0);
      if (ok && J > 1) ok = load_k(1);
      if (ok) ok = load_v(0);
      for (int j = 2; ok && j <= J; ++j) {
        if (j < J) ok = load_k(j);
        if (ok) ok = load_v(j - 1);
      }
      // Never leave the CTA with copies in flight: wait for the last load of
      // every slot (already complete in the normal case).
      mbar_wait_drain(bar(kQFull), 0, wc, site(6));
      for (int s = 0; s < kKSlots; ++s) {
        if (s >= k_boxes) continue;
        const int last = s + (k_boxes - 1 - s) / kKSlots * kKSlots;   // last ring index that used slot s
        mbar_wait_drain(bar(kKFull + s), (uint32_t)((last / kKSlots) & 1), wc, site(6));
      }
      if (v_tiles > 0) mbar_wait_drain(bar(kVFull), (uint32_t)((v_tiles - 1) & 1), wc, site(6));
    }
  } else {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_f16kind(128, kBN, false, false, F16);   // S = Q Kᵀ, both K-major
      constexpr uint32_t kIdO = idesc_f16kind(128, kD, false, true, F16);     // O += P V, V is MN-major
      bool ok = mbar_wait(bar(kQFull), 0, wc, site(7));
      // S_j into buffer j mod 2, K box by box from the ring.
      auto issue_s = [&](int j) -> bool {
        const uint32_t col = 128u * (uint32_t)(j & 1);
        for (int bx = 0; bx < 4; ++bx) {
          const int gi = 4 * j + bx, slot = gi % kKSlots;
          if (!mbar_wait(bar(kKFull + slot), (uint32_t)((gi / kKSlots) & 1), wc, site(8))) return false;
          tc_fence_after();
          const uint32_t qa = sbase + kQ + bx * kBox, kb = sbase + kK + slot * kBox;
          const bool chk = dcheck(tmem_ok(col, kBN, 512), wc, kChkTmem, 37) &&
                           dcheck(smem_ok(qa - sbase, kBox, kBar, 1024) && smem_ok(kb - sbase, kBox, kBar, 1024), wc,
                                  kChkSmem, 37);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            if (chk) mma_ss(tmem + col, sdesc_sw128(qa + 32u * k, 16, 1024), sdesc_sw128(kb + 32u * k, 16, 1024), kIdS,
                   (bx > 0 || k > 0) ? 1u : 0u);
          tc_commit(bar(kKEmpty + slot));
        }
        tc_commit(bar(kSFull + (j & 1)));
        return true;
      };
      if (ok) ok = issue_s(0);
      if (ok && J > 1) ok = issue_s(1);
      for (int j = 0; ok && j < J; ++j) {
        if (!mbar_wait(bar(kPFull + (j & 1)), (uint32_t)((j >> 1) & 1), wc, site(9)) ||
            !mbar_wait(bar(kVFull), (uint32_t)(j & 1), wc, site(10))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t pcol = 128u * (uint32_t)(j & 1);
        const bool chk = dcheck(tmem_ok(256u, kD, 512) && tmem_ok(pcol, kBN / 2, 512), wc, kChkTmem, 38) &&
                         dcheck(smem_ok(kV, 4 * kBox, kBar, 1024), wc, kChkSmem, 38);
#pragma unroll
        for (int ks = 0; ks < kBN / 16; ++ks)
          if (chk) mma_ts(tmem + 256u, tmem + pcol + (uint32_t)(8 * ks), sdesc_sw128(sbase + kV + (uint32_t)(ks * 2048), kBox, 1024),
                 kIdO, (j > 0 || ks > 0) ? 1u : 0u);
        tc_commit(bar(kVEmpty));
        tc_commit(bar(kPVDone));
        if (j == J - 1) tc_commit(bar(kOFull));
        if (j + 2 < J) ok = issue_s(j + 2);
      }
      // Every product must be finished before tensor memory is released.
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

template <bool CAUSAL, bool RAGGED, bool F16>
cudaError_t launch_impl(const FwdArgs& a, cudaStream_t s) {
  auto kern = fa_fwd_d256_kernel<CAUSAL, RAGGED, F16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  const long long units = (long long)fwd_units(a.B, a.H, a.Nq, kD);
  const long long ctas = CAUSAL ? units : a.n_full + (units - a.n_full) * a.splits;
  kern<<<(unsigned)ctas, kThreads, kSmemBytes, s>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess || CAUSAL || a.splits <= 1 || a.n_full >= units) return e;
  return launch_fwd_combine(a, (int)(units - a.n_full), kBM, s);
}

template <bool F16>
cudaError_t dispatch(const FwdArgs& a, bool ragged, cudaStream_t s) {
  if (ragged) return a.causal ? launch_impl<true, true, F16>(a, s) : launch_impl<false, true, F16>(a, s);
  return a.causal ? launch_impl<true, false, F16>(a, s) : launch_impl<false, false, F16>(a, s);
}

}  // namespace

cudaError_t launch_fwd_d256(const FwdArgs& a, cudaStream_t s) {
  if (a.d != kD) return cudaErrorInvalidValue;
  const bool ragged = a.Nq % kBM != 0 || a.Nk % kBN != 0;
  return a.f16 ? dispatch<true>(a, ragged, s) : dispatch<false>(a, ragged, s);
}

}  // namespace fa
