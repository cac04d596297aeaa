// fa_bwd_bf16.cu — tiled attention backward on the sm_103a tensor cores.
//
// What it computes: "Flash Attention" tutorial, 4.附录A "反向传播的公式推导"
// 五-六 (and 3.Recomputation 四): with only O and LSE kept from the forward,
// each tile of P is rebuilt as exp(S - LSE); D = rowsum(dO ⊙ O) replaces
// rowsum(dP ⊙ P); then dV += Pᵀ dO, dP = dO Vᵀ, dS = P ⊙ (dP - D),
// dK += dSᵀ Q and dQ += dS K.  The scale of the scores multiplies dQ and dK
// (coreui.cn page "FlashAttention 反向传播", dQ = dS K / sqrt(d_k)).
//
// Loop order differs from the page's pseudocode (query tiles outermost): a CTA
// owns one 128-row K/V tile and walks the 128-row query tiles, so dK and dV
// accumulate in tensor memory and only dQ is shared between CTAs (fp32
// vector reductions into a workspace accumulator).  The sums are the same.
//
// Per query tile (rows = keys for the first four, rows = queries for dQ):
//   Sᵀ  = K Qᵀ        tcgen05, A = K (smem), B = Q (smem), both K-major
//   dPᵀ = V dOᵀ       same with V and dO
//   Pᵀ  = exp2(Sᵀ·scale·log2e − LSE₂), dSᵀ = Pᵀ ⊙ (dPᵀ − D)   one thread per key row
//   dV += Pᵀ dO       A = Pᵀ from tensor memory (written over Sᵀ), B = dO (MN-major)
//   dK += dSᵀ Q       A = dSᵀ (smem, K-major over queries), B = Q (MN-major)
//   dQ                d = 128: dQᵀ = Kᵀ dSᵀ (M = head dims, N = queries);
//                     d = 64:  dQ = dS K (M = queries, N = head dims);
//                     both read the dSᵀ tile and K MN-major from smem
// Every product is M = 128 with N ≥ 64 (N = 128 except dV, dK, dQ at d = 64).
//
// Tensor memory (512 columns), d = 128: dV [0, 128), dK [128, 256), Sᵀ/Pᵀ
// [256, 384), dPᵀ/dQᵀ [384, 512).  dQᵀ reuses the dPᵀ columns once the
// compute warps have read dPᵀ; the next dPᵀ waits until dQᵀ has been
// drained, and the next Sᵀ goes over Pᵀ right after dV.  d = 64: dV [0, 64),
// dK [64, 128), two Sᵀ/Pᵀ buffers [128, 256) and [384, 512) used by
// alternate tiles, dPᵀ [256, 384).  Tile i's dQ goes into the last 64
// columns of its Sᵀ buffer (Pᵀ holds the first 64), so the next dPᵀ is
// issued right after dQ and dK, and Sᵀ of tile i + 2 is issued into that
// buffer once dV has read Pᵀ and dQ has been drained: the compute warps
// find each tile's scores ready (measured on GB300: +5.9 % at d = 64).
//
// CTA: 16 warps.  Warps 0-7 compute Pᵀ/dSᵀ (warp w owns key rows 32(w%4)..+31
// and query columns 64(w/4)..+63); warps 8-11 drain each tile's dQ from
// tensor memory into the fp32 accumulator with global reductions, so those
// run while the compute warps work on the next tile; warp 12 issues TMA,
// warp 13 issues the MMAs and owns tensor memory; at d = 128 warp 14 issues
// dK += dSᵀ Q once warp 13 has issued the next Sᵀ — the products keep their
// order in the pipe, and the main issuing thread, which sets the pace
// (clock64 traces on GB300), has 8 fewer products a step (+1.4 %).  The grid
// is head-major (K/V tile fastest).
#include "fa_kernels.h"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

constexpr int kBN = 128;            // keys per CTA
constexpr int kBM = 128;            // queries per step
constexpr int kThreads = 512;       // four warpgroups
constexpr int kComputeWarps = 8;    // warpgroups 0, 1: Pᵀ and dSᵀ
constexpr int kRedWarp = 8;         // warpgroup 2: dQ reductions
constexpr int kRedWarps = 4;
constexpr int kTmaWarp = 12;        // warpgroup 3: TMA, MMA, dK MMA (warp 15 idle)
constexpr int kMmaWarp = 13;
constexpr int kDkWarp = 14;
// Registers per thread of each warpgroup (setmaxnreg).  The CTA's pool is
// fixed at launch: kThreads × (65536 / kThreads) = 65536; the four
// warpgroups' shares must fit in it or an increase would wait forever.
constexpr int kRegsCompute = 176;
constexpr int kRegsRed = 80;
constexpr int kRegsMisc = 80;
constexpr int kEndBarrier = 15;     // named barrier of the CTA's last step (1..4: Pᵀ pair barriers)
static_assert(128 * (2 * kRegsCompute + kRegsRed + kRegsMisc) <= 65536, "warpgroup register shares exceed the pool");
constexpr int kBox = 16384;         // one TMA box: 128 rows × 128 bytes
// Exponential pairs per FMA-pipe exponential (0 = all on MUFU); measured on
// GB300 the split makes no difference here, so all stay on MUFU.
constexpr int kPolyEvery = 0;

template <int D>
struct BwdCfg {
  // Stages of the Q / dO / LSE / D ring: d = 64 issues each Sᵀ two tiles
  // ahead (a second Sᵀ buffer), so its ring holds three tiles.
  static constexpr int kQS = D == 64 ? 3 : 2;
  // shared memory (offsets from a 1024-byte aligned base)
  static constexpr int kTile = 128 * D * 2;        // one 128 × D bf16 tile (D/64 boxes)
  static constexpr int kK = 0;
  static constexpr int kV = kK + kTile;
  static constexpr int kQ = kV + kTile;            // kQS stages
  static constexpr int kDO = kQ + kQS * kTile;     // kQS stages
  static constexpr int kDS = kDO + kQS * kTile;    // dSᵀ [128 keys][128 queries] bf16: 2 boxes
  static constexpr int kLSE = kDS + 2 * kBox;      // kQS stages of 128 floats
  static constexpr int kDV = kLSE + kQS * kBM * 4; // kQS stages of 128 floats
  static constexpr int kBar = kDV + kQS * kBM * 4;
  static constexpr int kBytes = kBar + 256;
  // tensor memory columns
  static constexpr uint32_t kColDV = 0;
  static constexpr uint32_t kColDK = D;
  static constexpr uint32_t kColS = 2 * D;
  static constexpr uint32_t kColDP = 2 * D + 128;
  // d = 64: a second Sᵀ buffer in the 128 columns the 64-wide accumulators leave free.
  static constexpr uint32_t kColS2 = 2 * D + 256;
};

// Barrier slots (8 bytes each) inside the barrier block.
template <int QS>
struct BwdBars {
  static constexpr int kKVFull = 0;
  static constexpr int kQFull = 1;             // +stage
  static constexpr int kQEmpty = 1 + QS;       // +stage
  static constexpr int kSFull = 1 + 2 * QS;
  static constexpr int kDPFull = kSFull + 1;
  static constexpr int kPdsFull = kSFull + 2;
  static constexpr int kDqFull = kSFull + 3;
  static constexpr int kDqDrained = kSFull + 4;
  static constexpr int kDKVFull = kSFull + 5;
  static constexpr int kMmaDone = kSFull + 6;
  static constexpr int kSIssued = kSFull + 7;    // warp 13 has issued step i's products before dK
  static constexpr int kDkDone = kSFull + 8;     // dK of step i done: dSᵀ may be overwritten
  static constexpr int kMmaDone2 = kSFull + 9;   // every product of the dK warp has finished
  static constexpr int kSFull2 = kSFull + 10;    // the second Sᵀ buffer (d = 64)
  static constexpr int kNumBars = kSFull + 11;
  static_assert(8 * kNumBars + 8 <= 256, "barrier block too small");
};

__device__ __forceinline__ uint32_t site(int s) { return 0x0200u | (uint32_t)s; }

// Pᵀ for 32 query columns of one key row: p = 2^(s·scale·log2e − LSE₂) as
// packed pairs, from Sᵀ (32 TMEM words) and −LSE₂ (16 pairs).  With MASKED,
// columns whose query precedes the key (column index < `row_minus_col0`) are
// zero.  With POLY_EVERY > 0 one pair in POLY_EVERY takes its exponentials on
// the FMA pipe.
template <bool MASKED, int POLY_EVERY>
__device__ __forceinline__ void p_chunk(const uint32_t (&s)[32], uint64_t sl2x2, const uint64_t* nlse,
                                        int row_minus_col0, uint64_t* p) {
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    const uint64_t x = f2_fma(f2_pack(u2f(s[2 * e]), u2f(s[2 * e + 1])), sl2x2, nlse[e]);
    float x0, x1, e0, e1;
    f2_unpack(x, x0, x1);
    if (POLY_EVERY > 0 && e % (POLY_EVERY > 0 ? POLY_EVERY : 1) == POLY_EVERY - 1) {
      exp2_fma_x2(x0, x1, e0, e1);
    } else {
      e0 = ex2(x0);
      e1 = ex2(x1);
    }
    if (MASKED) {
      // key kv is visible to query q iff kv ≤ q
      e0 = row_minus_col0 > 2 * e ? 0.f : e0;
      e1 = row_minus_col0 > 2 * e + 1 ? 0.f : e1;
    }
    p[e] = f2_pack(e0, e1);
  }
}

// Barrier among the two compute warps that share a TMEM lane quarter, with an
// AND over their `ok` flags so both take the same branch.
__device__ __forceinline__ bool pair_sync_and(int id, bool ok) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.b32 p, %1, 0;\n bar.red.and.pred q, %2, 64, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)ok), "r"(id)
      : "memory");
  return r != 0;
}

// RAGGED (Nq or Nk not a multiple of 128): 3-D per-head tensor maps whose
// rows past the end read as zero, masking of the keys past Nk and
// row-predicated dK/dV stores.  Otherwise 2-D maps over the row views and
// none of that.
// F16: fp16 inputs and outputs (else bf16); Pᵀ and dSᵀ are rounded to the same type.
// DR: the head dimension (64, 96 or 128).  Tiles are laid out D = 64 or 128
// columns wide; with DR = 96 the tensor maps read columns 96..127 as zeros,
// the products run over the 96 real columns (6 K-steps for Sᵀ and dPᵀ,
// N = 96 for dV and dK; dQᵀ keeps M = 128 with zero rows past 96) and only
// 96 columns are reduced or stored.
template <int DR, bool CAUSAL, bool RAGGED, bool F16>
__global__ void __launch_bounds__(kThreads, 1) fa_bwd_bf16_kernel(const __grid_constant__ BwdArgs a) {
  constexpr int D = DR <= 64 ? 64 : 128;
  using C = BwdCfg<D>;
  constexpr int QS = C::kQS;
  // dK from its own warp where it measured faster (the 128-column layout:
  // d = 96, 128); at d = 64 the extra hand-over costs more than it saves.
  constexpr bool kDkSplit = D == 128;
  // Two Sᵀ buffers where tensor memory has room for them (d = 64): step i
  // uses buffer i mod 2, and the MMA thread issues Sᵀ of tile i + 2 as soon
  // as dV of tile i has read its Pᵀ, so the compute warps find the next
  // tile's scores ready when they finish a tile.
  constexpr bool kSDouble = D == 64;
  static_assert(kSDouble != kDkSplit, "the 64-column layout issues dK inline, the 128-column one from warp 14");
  static_assert(!kSDouble || C::kColS2 + 128 <= 512, "second score buffer outside tensor memory");
  using Bar = BwdBars<QS>;
  constexpr int kKVFull = Bar::kKVFull, kQFull = Bar::kQFull, kQEmpty = Bar::kQEmpty, kSFull = Bar::kSFull,
                kDPFull = Bar::kDPFull, kPdsFull = Bar::kPdsFull, kDqFull = Bar::kDqFull,
                kDqDrained = Bar::kDqDrained, kDKVFull = Bar::kDKVFull, kMmaDone = Bar::kMmaDone,
                kNumBars = Bar::kNumBars, kSIssued = Bar::kSIssued, kDkDone = Bar::kDkDone, kMmaDone2 = Bar::kMmaDone2,
                kSFull2 = Bar::kSFull2;
  // Sᵀ buffer of step i: its tensor-memory columns, its barrier and the parity of its use.
  auto s_cols = [](int i) -> uint32_t { return (kSDouble && (i & 1)) ? C::kColS2 : C::kColS; };
  auto s_bar_id = [](int i) -> int { return (kSDouble && (i & 1)) ? kSFull2 : kSFull; };
  auto s_parity = [](int i) -> uint32_t { return kSDouble ? (uint32_t)((i >> 1) & 1) : (uint32_t)(i & 1); };
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
  const int Nq = a.Nq, Nk = a.Nk;
  const int off = Nk - Nq;                   // causal: query i sees keys j ≤ i + off
  // Non-causal: head-major grid (K/V tile fastest), so a wave touches few
  // heads' Q, dO and dQ accumulator and they stay in L2.  Causal: batch·head
  // fastest, so the heaviest tiles (small jt) of every head go first.
  const int jt = CAUSAL ? (int)blockIdx.y : (int)blockIdx.x;
  const int bh = CAUSAL ? (int)blockIdx.x : (int)blockIdx.y;
  const int kv0 = jt * kBN;
  const int n_tiles = RAGGED ? (Nq + kBM - 1) / kBM : Nq / kBM;   // query tiles per head; the last may be ragged
  // First row of this head in the workspace (whole tiles per head; the
  // workspace has fewer than 2^31 rows).
  const int wrow0 = RAGGED ? bh * n_tiles * kBM : bh * Nq;
  // First query tile with a query that sees a key of this tile: query tile i
  // reaches keys up to 128i + 127 + off, so i ≥ ⌊(kv0 − off) / 128⌋ (kBM == kBN).
  const int i0 = CAUSAL ? (kv0 > off ? (kv0 - off) / kBM : 0) : 0;
  // Loads rows [pos, pos + 128) of this head from a map over heads of `nrows` rows.
  // A debug build checks the destination and the coordinates first and, if a
  // check fails, completes the box's bytes on the barrier without copying.
  auto load_rows = [&](uint32_t dst, const CUtensorMap* map, uint32_t bar_addr, int x, int pos, int nrows) {
    bool chk = dcheck(smem_ok(dst - sbase, kBox, (uint32_t)C::kBar, 1024), wc, kChkSmem, 16) &&
               dcheck(tma_x_ok(x, 64, D), wc, kChkTmaX, 16);
    if constexpr (RAGGED)
      chk = chk && dcheck(tma_head_ok(pos, nrows, bh, a.B * a.H), wc, kChkTmaRows, 16);
    else
      chk = chk && dcheck(tma_rows_ok((long long)bh * nrows + pos, 128, (long long)a.B * a.H * nrows), wc,
                          kChkTmaRows, 16);
    if (!chk) {
      mbar_complete_tx(bar_addr, kBox);
      return;
    }
    if constexpr (RAGGED)
      tma_load_3d(dst, map, bar_addr, x, pos, bh);
    else
      tma_load_2d(dst, map, bar_addr, x, bh * nrows + pos);
  };
  // Bulk copy of `bytes` of a workspace row array; checked like the tile loads.
  auto load_bulk = [&](uint32_t dst, const float* src, uint32_t bytes, uint32_t bar_addr) {
    if (!dcheck(smem_ok(dst - sbase, bytes, (uint32_t)C::kBar, 16) &&
                    bulk_ok(reinterpret_cast<uint64_t>(src), dst, bytes), wc, kChkBulk, 17)) {
      mbar_complete_tx(bar_addr, bytes);
      return;
    }
    bulk_load(dst, src, bytes, bar_addr);
  };
  const int n = n_tiles - i0;                // query tiles visited
  // Step i works on query tile qtile(i).  (Measured on GB300: starting each
  // CTA of a head at its own query tile, so that concurrent CTAs add into
  // different dQ rows, was slower than all walking the tiles in order.)
  auto qtile = [&](int i) -> int { return i0 + i; };

  if (threadIdx.x == 0) {
    mbar_init(bar(kKVFull), 1);
    for (int s = 0; s < QS; ++s) {
      mbar_init(bar(kQFull + s), 1);
      mbar_init(bar(kQEmpty + s), (kDkSplit ? 2 : 1) + 32 * kComputeWarps);   // the issuing thread(s), the compute warps
    }
    mbar_init(bar(kSFull), 1);
    mbar_init(bar(kSFull2), 1);
    mbar_init(bar(kDPFull), 1);
    mbar_init(bar(kPdsFull), 32 * kComputeWarps);
    mbar_init(bar(kDqFull), 1);
    mbar_init(bar(kDqDrained), 32 * kRedWarps);
    mbar_init(bar(kDKVFull), kDkSplit ? 2 : 1);   // dV (warp 13) and dK (warp 14, or 13)
    mbar_init(bar(kSIssued), 1);
    mbar_init(bar(kDkDone), 1);
    mbar_init(bar(kMmaDone2), 1);
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
    setmaxnreg_inc<kRegsCompute>();
    const int g = warp & 3;
    const int h = warp >> 2;                       // query columns [64h, 64h + 64)
    const int r = g * 32 + lane;                   // key row within the tile = TMEM lane
    const int kv = kv0 + r;
    // A key past Nk (last tile of a ragged head) reads as a zero row, so its
    // score is 0 and 2^(−LSE·log2 e) could overflow; its Pᵀ and dSᵀ are
    // masked to 0 so that dQ never sees it.  Causal tiles mask it already
    // (it lies beyond every real query's last key).  Queries past Nq need
    // nothing: their −LSE is −∞ and their dO row is zero.
    const bool dead_key = RAGGED && kv >= Nk;
    [[maybe_unused]] const bool ragged_cta = RAGGED && !CAUSAL && kv0 + kBN > Nk;   // uniform over the CTA
    [[maybe_unused]] const int dead_lim = dead_key ? (1 << 30) : -(1 << 30);        // masks all columns or none
    const uint32_t lane_off = (uint32_t)(g * 32) << 16;
    const float sl2 = a.scale_log2;
    const uint32_t ds_tile = sbase + C::kDS;
    bool ok = true;
    for (int i = 0; i < n; ++i) {
      const int st = i % QS;
      const uint32_t par = (uint32_t)(i & 1);
      const int q0 = qtile(i) * kBM;
      const uint32_t scol = s_cols(i);
      ok = mbar_wait_inl(bar(s_bar_id(i)), s_parity(i), wc, site(1)) &&
           mbar_wait_inl(bar(kQFull + st), (uint32_t)((i / QS) & 1), wc, site(3));
      ok = __all_sync(kFull, ok);
      // The pre-pass stored −LSE·log2(e) and −D, so each pair of columns is
      // one packed FMA (the exponent) and one packed add/multiply (dS).
      const uint64_t* nlse = reinterpret_cast<const uint64_t*>(sgen + C::kLSE + st * kBM * 4);
      const uint64_t* ndv = reinterpret_cast<const uint64_t*>(sgen + C::kDV + st * kBM * 4);
      // Key kv0 + r is visible to query q0 + c iff r − c ≤ delta; the tile
      // masks something iff its largest key passes its first query's limit
      // (square problems: only the diagonal tile, delta = 0).
      const int delta = q0 + off - kv0;
      const bool masked = CAUSAL && delta < kBN - 1;
      const uint64_t sl2x2 = f2_pack(sl2, sl2);
      uint64_t p[32];                              // P for query columns 64h + 2e, 2e + 1
      if (ok) {
        tc_fence_after();
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
          const int c0 = h * 64 + ch * 32;
          uint32_t s[32];
          if (dcheck(tmem_ok(scol + c0, 32, 512), wc, kChkTmem, 18))
            tmem_ld_x32(tmem + lane_off + scol + (uint32_t)c0, s);
          if (masked)
            p_chunk<true, kPolyEvery>(s, sl2x2, nlse + (c0 >> 1), r - c0 - delta, p + ch * 16);
          else if (ragged_cta)
            p_chunk<true, 0>(s, sl2x2, nlse + (c0 >> 1), dead_lim, p + ch * 16);
          else
            p_chunk<false, kPolyEvery>(s, sl2x2, nlse + (c0 >> 1), r - c0, p + ch * 16);
        }
      }
      // dPᵀ is issued after the previous tile's dQ has been drained, so it
      // lands while the exponentials above run: wait for it only now.
      if (ok) ok = mbar_wait_inl(bar(kDPFull), par, wc, site(2));
      // Both warps of the lane quarter have read their Sᵀ columns; Pᵀ may now
      // be written over the first 64 of them.
      ok = pair_sync_and(1 + g, ok);
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float a0, a1;
          f2_unpack(p[half * 16 + e], a0, a1);
          pk[e] = pack2<F16>(a0, a1);
        }
        if (dcheck(tmem_ok(scol + h * 32 + 16 * half, 16, 512), wc, kChkTmem, 19))
          tmem_st_x16(tmem + lane_off + scol + (uint32_t)(h * 32 + 16 * half), pk);
      }
      // dK of the previous step reads dSᵀ from shared memory: it must be done
      // before this step's dSᵀ is written there.
      if (kDkSplit && i > 0) mbar_wait_inl(bar(kDkDone), (uint32_t)((i - 1) & 1), wc, site(15));
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        const int c0 = h * 64 + ch * 32;
        uint32_t dp[32];
        if (dcheck(tmem_ok(C::kColDP + c0, 32, 512), wc, kChkTmem, 20))
          tmem_ld_x32(tmem + lane_off + C::kColDP + (uint32_t)c0, dp);
        uint32_t dk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const uint64_t ds = f2_mul(p[ch * 16 + e], f2_add(f2_pack(u2f(dp[2 * e]), u2f(dp[2 * e + 1])), ndv[(c0 >> 1) + e]));
          float d0, d1;
          f2_unpack(ds, d0, d1);
          dk[e] = pack2<F16>(d0, d1);
        }
        // 32 query columns = four 16-byte chunks of this key row, in box h
        // (queries 64h..64h+63), placed with the 128-byte swizzle.
        const uint32_t row_addr = ds_tile + (uint32_t)(h * kBox + r * 128);
        if (!dcheck(smem_ok(row_addr - sbase, 128, (uint32_t)C::kBar, 128), wc, kChkSmem, 21)) continue;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int chunk = ch * 4 + u;
          st_shared_v4(row_addr + (uint32_t)(((chunk ^ (r & 7)) & 7) * 16), dk[4 * u], dk[4 * u + 1], dk[4 * u + 2],
                       dk[4 * u + 3]);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      fence_proxy_async_smem();
      mbar_arrive(bar(kPdsFull));
      mbar_arrive(bar(kQEmpty + st));
    }
    // ------------------------------------------------------------ dK, dV epilogue
    if (ok) {
      ok = mbar_wait_inl(bar(kDKVFull), 0, wc, site(5));
      ok = __all_sync(kFull, ok);
    }
    if (ok) {
      tc_fence_after();
      const uint32_t col = h == 0 ? C::kColDV : C::kColDK;
      const float mul = h == 0 ? 1.0f : a.scale;
      uint16_t* dst = static_cast<uint16_t*>(h == 0 ? a.dv : a.dk) + ((size_t)bh * (size_t)Nk + (size_t)kv) * DR;
#pragma unroll
      for (int cc = 0; cc < DR / 32; ++cc) {
        uint32_t v[32];
        if (!dcheck(tmem_ok(col + 32 * cc, 32, 512), wc, kChkTmem, 22)) continue;
        tmem_ld_x32(tmem + lane_off + col + 32 * cc, v);   // warp-collective: every lane loads
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) pk[e] = pack2<F16>(u2f(v[2 * e]) * mul, u2f(v[2 * e + 1]) * mul);
        if (!dead_key) {
#pragma unroll
          for (int u = 0; u < 4; ++u)
            st_global_v4(dst + 32 * cc + 8 * u, pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
        }
      }
    }
    tc_fence_before();
    named_bar_arrive(kEndBarrier, kThreads);
  } else if (warp < kRedWarp + kRedWarps) {
    // ------------------------------------------------------------ dQ reductions
    // The MMA thread issues each tile's dQ first after Pᵀ/dSᵀ and the next
    // dPᵀ only after these warps have read dQ out of its columns.  Each thread
    // reads its lane's share into registers, releases the columns, and adds
    // into the fp32 accumulator with global reductions while the compute
    // warps move on to the next tile.
    setmaxnreg_dec<kRegsRed>();
    const int g = warp & 3;                        // TMEM lane quarter
    const int r = g * 32 + lane;
    const uint32_t lane_off = (uint32_t)(g * 32) << 16;
    // Pacing of the reductions issued after the columns are released: they
    // run beside the next dPᵀ product and the compute warps' next tile, and
    // issued in one burst they slow both.  Each thread pauses after every 4
    // floats it adds, so that its reductions span about a quarter of the
    // previous step, as timed between its own dQ hand-overs (no pause on the
    // first step).  Measured on GB300 against unpaced reductions: +10 % for
    // the whole backward at d = 128 (7 longer pauses, after every 8 floats,
    // gained 8 %), +4.5 % at d = 64.
    uint32_t t_prev = 0;
    uint32_t pause_ns = 0;
    for (int i = 0; i < n; ++i) {
      const int q0 = qtile(i) * kBM;
      bool ok = mbar_wait_inl(bar(kDqFull), (uint32_t)(i & 1), wc, site(6));
      ok = __all_sync(kFull, ok);
      if (!ok) break;
      {
        // 15 pauses of step / 120 (cycles read as ns at ~2 GHz: a quarter of
        // the step; `pause_ns` holds step / 40 and is divided at each pause,
        // a form that measured 0.5 % faster than holding step / 120).  Pauses
        // feed back into the step they are measured on: on GB300, pauses
        // adding up to ~60 % of the step already ran away (the backward 15 %
        // slower, ~70 %: 35 %), and a third of the step after every 4 floats
        // (step / 80) was slower than a quarter, so the share stays well short
        // of that and each pause is capped.  32-bit clock: the unsigned
        // difference survives a wrap.
        const uint32_t t_now = (uint32_t)clock();
        if (i > 0) {
          const uint32_t p = (t_now - t_prev) / 40u;
          pause_ns = p < 200u ? p : 200u;
        }
        t_prev = t_now;
      }
      tc_fence_after();
      if constexpr (D == 128) {
        // dQᵀ: lane = head dim r, columns = the tile's 128 queries, read in
        // two halves of 64; a warp's reduction covers 32 consecutive floats of
        // one accumulator row.  Warps whose head dims are all past DR only
        // release the columns.
        if (g * 32 < DR) {
          float* base = a.dqacc + ((size_t)wrow0 + (size_t)q0) * DR + (size_t)r;
          uint32_t v[64];
          if (!dcheck(tmem_ok(C::kColDP, 128, 512), wc, kChkTmem, 23)) {
            tc_fence_before();
            mbar_arrive(bar(kDqDrained));
            continue;
          }
          tmem_ld_x64(tmem + lane_off + C::kColDP, v);
#pragma unroll
          for (int c = 0; c < 64; ++c) red_add_f32(base + (size_t)c * DR, u2f(v[c]));
          tmem_ld_x64(tmem + lane_off + C::kColDP + 64u, v);
          tc_fence_before();
          mbar_arrive(bar(kDqDrained));
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            red_add_f32(base + (size_t)(64 + c) * DR, u2f(v[c]));
            if ((c & 3) == 3 && c < 63 && pause_ns > 0) __nanosleep(pause_ns / 3u);
          }
        } else {
          tc_fence_before();
          mbar_arrive(bar(kDqDrained));
        }
      } else {
        // dQ: lane = query row r, columns = the 64 head dims; 16-byte vector
        // reductions along the row.
        uint32_t v[64];
        const uint32_t dq_col = s_cols(i) + 64u;   // the last 64 columns of step i's Sᵀ buffer
        const bool chk = dcheck(tmem_ok(dq_col, 64, 512), wc, kChkTmem, 24);
        if (chk) tmem_ld_x64(tmem + lane_off + dq_col, v);
        tc_fence_before();
        mbar_arrive(bar(kDqDrained));
        if (!chk) continue;
        float* base = a.dqacc + ((size_t)wrow0 + (size_t)q0 + (size_t)r) * D;
#pragma unroll
        for (int c = 0; c < 64; c += 4) {
          red_add_v4_f32(base + c, u2f(v[c]), u2f(v[c + 1]), u2f(v[c + 2]), u2f(v[c + 3]));
          if (c < 60 && pause_ns > 0) __nanosleep(pause_ns / 3u);
        }
      }
    }
    tc_fence_before();
    named_bar_arrive(kEndBarrier, kThreads);
  } else {
  // Warpgroup 3.  setmaxnreg is .aligned: the four warps execute this one
  // instruction before taking their separate roles.
  setmaxnreg_dec<kRegsMisc>();
  if (warp == kTmaWarp) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tmap(&a.tm_q);
      prefetch_tmap(&a.tm_k);
      prefetch_tmap(&a.tm_v);
      prefetch_tmap(&a.tm_do);
      mbar_arrive_expect_tx(bar(kKVFull), 2u * C::kTile);
      for (int bx = 0; bx < D / 64; ++bx) {
        load_rows(sbase + C::kK + bx * kBox, &a.tm_k, bar(kKVFull), 64 * bx, kv0, Nk);
        load_rows(sbase + C::kV + bx * kBox, &a.tm_v, bar(kKVFull), 64 * bx, kv0, Nk);
      }
      int issued[QS] = {};
      for (int i = 0; i < n; ++i) {
        const int s = i % QS;
        if (i >= QS && !mbar_wait_inl(bar(kQEmpty + s), (uint32_t)((i / QS - 1) & 1), wc, site(7))) break;
        const int q0 = qtile(i) * kBM;
        mbar_arrive_expect_tx(bar(kQFull + s), 2u * C::kTile + 2u * kBM * 4);
        for (int bx = 0; bx < D / 64; ++bx) {
          load_rows(sbase + C::kQ + s * C::kTile + bx * kBox, &a.tm_q, bar(kQFull + s), 64 * bx, q0, Nq);
          load_rows(sbase + C::kDO + s * C::kTile + bx * kBox, &a.tm_do, bar(kQFull + s), 64 * bx, q0, Nq);
        }
        load_bulk(sbase + C::kLSE + s * kBM * 4, a.lse2 + wrow0 + q0, kBM * 4, bar(kQFull + s));
        load_bulk(sbase + C::kDV + s * kBM * 4, a.dvec + wrow0 + q0, kBM * 4, bar(kQFull + s));
        ++issued[s];
      }
      mbar_wait_drain_inl(bar(kKVFull), 0, wc, site(8));
      for (int s = 0; s < QS; ++s)
        if (issued[s] > 0) mbar_wait_drain_inl(bar(kQFull + s), (uint32_t)((issued[s] - 1) & 1), wc, site(8));
    }
    __syncwarp();
    named_bar_arrive(kEndBarrier, kThreads);
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_f16kind(128, kBM, false, false, F16);  // Sᵀ = K Qᵀ, dPᵀ = V dOᵀ
      constexpr uint32_t kIdKV = idesc_f16kind(128, DR, false, true, F16);   // dV += Pᵀ dO, dK += dSᵀ Q
      // d = 128: dQᵀ = Kᵀ dSᵀ (M = head dims, N = 128 queries); d = 64: dQ = dS K (M = queries, N = 64)
      constexpr uint32_t kIdQ =
          D == 128 ? idesc_f16kind(128, kBM, true, true, F16) : idesc_f16kind(128, D, true, true, F16);
      auto issue_sd = [&](int i, uint32_t col, uint32_t a_tile) {    // Sᵀ (A = K) or dPᵀ (A = V)
        const int st = i % QS;
        const uint32_t b_tile = (a_tile == sbase + C::kK ? sbase + C::kQ : sbase + C::kDO) + st * C::kTile;
        if (!(dcheck(tmem_ok(col, kBM, 512), wc, kChkTmem, 25) &&
              dcheck(smem_ok(a_tile - sbase, C::kTile, C::kBar, 1024), wc, kChkSmem, 25) &&
              dcheck(smem_ok(b_tile - sbase, C::kTile, C::kBar, 1024), wc, kChkSmem, 25)))
          return;
#pragma unroll
        for (int ks = 0; ks < DR / 16; ++ks) {
          const uint32_t off = (uint32_t)((ks >> 2) * kBox + (ks & 3) * 32);
          mma_ss(tmem + col, sdesc_sw128(a_tile + off, 16, 1024), sdesc_sw128(b_tile + off, 16, 1024), kIdS,
                 ks > 0 ? 1u : 0u);
        }
      };
      bool ok = mbar_wait_inl(bar(kKVFull), 0, wc, site(9)) && mbar_wait_inl(bar(kQFull), 0, wc, site(10));
      if (ok && n > 0) {
        tc_fence_after();
        issue_sd(0, C::kColS, sbase + C::kK);
        tc_commit(bar(kSFull));
        issue_sd(0, C::kColDP, sbase + C::kV);
        tc_commit(bar(kDPFull));
        if (kSDouble && n > 1) {
          ok = mbar_wait_inl(bar(kQFull + 1), 0, wc, site(12));
          if (ok) {
            tc_fence_after();
            issue_sd(1, C::kColS2, sbase + C::kK);
            tc_commit(bar(kSFull2));
          }
        }
      }
      for (int i = 0; ok && i < n; ++i) {
        const int st = i % QS;
        if (!mbar_wait_inl(bar(kPdsFull), (uint32_t)(i & 1), wc, site(11))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t ds = sbase + C::kDS;
        const uint32_t qb = sbase + C::kQ + st * C::kTile;
        const uint32_t ob = sbase + C::kDO + st * C::kTile;
        // Debug build: every column range and operand tile of this step's products.
        const bool chk = dcheck(tmem_ok(kSDouble ? s_cols(i) + 64 : C::kColDP, D == 128 ? kBM : D, 512) &&
                                    tmem_ok(C::kColDV, DR, 512) && tmem_ok(C::kColDK, DR, 512) &&
                                    tmem_ok(s_cols(i), kBM / 2, 512),
                                wc, kChkTmem, 26) &&
                         dcheck(smem_ok(C::kDS, 2 * kBox, C::kBar, 1024) && smem_ok(qb - sbase, C::kTile, C::kBar, 1024) &&
                                    smem_ok(ob - sbase, C::kTile, C::kBar, 1024),
                                wc, kChkSmem, 26);
        const bool next = i + 1 < n;
        if constexpr (kSDouble) {
          // d = 64.  dQ = dS K into the last 64 columns of this step's Sᵀ
          // buffer (read already; Pᵀ is in the first 64), dK += dSᵀ Q, then
          // the next dPᵀ — its columns are free once dSᵀ is formed, and its
          // barrier tells the compute warps that dQ and dK have read dSᵀ —
          // then dV += Pᵀ dO, and Sᵀ two tiles ahead into this buffer once the
          // reducers have read dQ out of it.
          const uint32_t sb = s_cols(i);
#pragma unroll
          for (int ks = 0; ks < kBN / 16; ++ks) {
            if (!chk) break;
            mma_ss(tmem + sb + 64u, sdesc_sw128(ds + (uint32_t)(ks * 2048), kBox, 1024),
                   sdesc_sw128(sbase + C::kK + (uint32_t)(ks * 2048), kBox, 1024), kIdQ, ks > 0 ? 1u : 0u);
          }
          tc_commit(bar(kDqFull));
#pragma unroll
          for (int ks = 0; ks < kBM / 16; ++ks)
            if (chk) mma_ss(tmem + C::kColDK, sdesc_sw128(ds + (uint32_t)((ks >> 2) * kBox + (ks & 3) * 32), 16, 1024),
                   sdesc_sw128(qb + (uint32_t)(ks * 2048), kBox, 1024), kIdKV, (i > 0 || ks > 0) ? 1u : 0u);
          if (next) {
            issue_sd(i + 1, C::kColDP, sbase + C::kV);
            tc_commit(bar(kDPFull));
          }
#pragma unroll
          for (int ks = 0; ks < kBM / 16; ++ks)
            if (chk) mma_ts(tmem + C::kColDV, tmem + sb + (uint32_t)(8 * ks),
                   sdesc_sw128(ob + (uint32_t)(ks * 2048), kBox, 1024), kIdKV, (i > 0 || ks > 0) ? 1u : 0u);
          tc_commit(bar(kQEmpty + st));
          if (i + 2 < n) {
            if (!mbar_wait_inl(bar(kQFull + (i + 2) % QS), (uint32_t)(((i + 2) / QS) & 1), wc, site(12)) ||
                !mbar_wait_inl(bar(kDqDrained), (uint32_t)(i & 1), wc, site(13))) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_sd(i + 2, sb, sbase + C::kK);
            tc_commit(bar(s_bar_id(i)));
          }
        } else {
          // dQ into the dPᵀ columns first, so its drain overlaps dV and dK.
          // Both operands are read MN-major, dSᵀ [keys][queries] and K [keys][dims].
#pragma unroll
          for (int ks = 0; ks < kBN / 16; ++ks) {
            if (!chk) break;
            const uint64_t dsd = sdesc_sw128(ds + (uint32_t)(ks * 2048), kBox, 1024);
            const uint64_t kd = sdesc_sw128(sbase + C::kK + (uint32_t)(ks * 2048), kBox, 1024);
            mma_ss(tmem + C::kColDP, kd, dsd, kIdQ, ks > 0 ? 1u : 0u);
          }
          tc_commit(bar(kDqFull));
          // dV += Pᵀ dO, Pᵀ from tensor memory
#pragma unroll
          for (int ks = 0; ks < kBM / 16; ++ks)
            if (chk) mma_ts(tmem + C::kColDV, tmem + s_cols(i) + (uint32_t)(8 * ks),
                   sdesc_sw128(ob + (uint32_t)(ks * 2048), kBox, 1024), kIdKV, (i > 0 || ks > 0) ? 1u : 0u);
          // Sᵀ of the next tile overwrites Pᵀ: issued right after dV, which
          // reads it (the products run in issue order), and before dK, so the
          // compute warps can start on it sooner.
          if (next) {
            if (!mbar_wait_inl(bar(kQFull + (i + 1) % QS), (uint32_t)(((i + 1) / QS) & 1), wc, site(12))) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_sd(i + 1, C::kColS, sbase + C::kK);
            tc_commit(bar(kSFull));
          }
          // dK += dSᵀ Q of this step is issued by warp 14, after these products.
          mbar_arrive(bar(kSIssued));
          tc_commit(bar(kQEmpty + st));
          if (next) {
            if (!mbar_wait_inl(bar(kDqDrained), (uint32_t)(i & 1), wc, site(13))) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_sd(i + 1, C::kColDP, sbase + C::kV);
            tc_commit(bar(kDPFull));
          }
        }
      }
      if (ok) tc_commit(bar(kDKVFull));
      tc_commit(bar(kMmaDone));
      mbar_wait_drain_inl(bar(kMmaDone), 0, wc, site(14));
    }
    __syncwarp();
    // Every thread of the CTA has finished with tensor memory once all have
    // arrived here; the allocating warp then frees it.
    named_bar_sync(kEndBarrier, kThreads);
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  } else if (kDkSplit && warp == kDkWarp) {
    // ------------------------------------------------------------ dK issuer
    // dK += dSᵀ Q of step i, once warp 13 has issued step i's dQ, dV and the
    // next Sᵀ (so the pipe sees the products in the single-thread order).
    if (lane == 0) {
      constexpr uint32_t kIdKV = idesc_f16kind(128, DR, false, true, F16);
      bool ok = true;
      for (int i = 0; ok && i < n; ++i) {
        const int st = i % QS;
        if (!mbar_wait_inl(bar(kSIssued), (uint32_t)(i & 1), wc, site(16))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t ds = sbase + C::kDS;
        const uint32_t qb = sbase + C::kQ + st * C::kTile;
        const bool chk = dcheck(tmem_ok(C::kColDK, DR, 512), wc, kChkTmem, 27) &&
                         dcheck(smem_ok(C::kDS, 2 * kBox, C::kBar, 1024) && smem_ok(qb - sbase, C::kTile, C::kBar, 1024),
                                wc, kChkSmem, 27);
#pragma unroll
        for (int ks = 0; ks < kBM / 16; ++ks)
          if (chk) mma_ss(tmem + C::kColDK, sdesc_sw128(ds + (uint32_t)((ks >> 2) * kBox + (ks & 3) * 32), 16, 1024),
                 sdesc_sw128(qb + (uint32_t)(ks * 2048), kBox, 1024), kIdKV, (i > 0 || ks > 0) ? 1u : 0u);
        tc_commit(bar(kDkDone));
        tc_commit(bar(kQEmpty + st));
      }
      if (ok) tc_commit(bar(kDKVFull));
      tc_commit(bar(kMmaDone2));
      mbar_wait_drain_inl(bar(kMmaDone2), 0, wc, site(17));
    }
    __syncwarp();
    named_bar_arrive(kEndBarrier, kThreads);
  } else {
    named_bar_arrive(kEndBarrier, kThreads);   // warp 15 (and 14 at d = 64)
  }
  }
  // No code after the roles: their register counts differ (setmaxnreg).
}

// Persistent form of the backward at d = 64 for problems without the mask
// whose CTAs would visit few query tiles: one CTA per SM walks the units
// (K/V tiles, head-major) u = blockIdx.x, blockIdx.x + gridDim.x, ...  The
// steps of all its units form one sequence: the Q/dO ring, the score
// buffers and every step barrier count on across units; K and V alternate
// between two buffers, so the next unit's K/V tile loads while the current
// one runs; the next unit's first scores and dPᵀ are issued during the
// current unit's last steps, and its first dK and dV products (which start
// the accumulators afresh) wait only until the compute warps have read the
// current unit's dK and dV out of tensor memory.  Per step it is the d = 64
// kernel above: two score buffers, dQ in the spent half of a buffer.
struct BwdCfgP64 {
  static constexpr int kQS = 3;
  static constexpr int kTile = 128 * 64 * 2;       // one 128 × 64 bf16 tile = one box
  static constexpr int kK = 0;                     // 2 unit buffers
  static constexpr int kV = kK + 2 * kTile;        // 2 unit buffers
  static constexpr int kQ = kV + 2 * kTile;        // kQS stages
  static constexpr int kDO = kQ + kQS * kTile;     // kQS stages
  static constexpr int kDS = kDO + kQS * kTile;    // dSᵀ [128 keys][128 queries]: 2 boxes
  static constexpr int kLSE = kDS + 2 * kBox;      // kQS stages of 128 floats
  static constexpr int kDV = kLSE + kQS * kBM * 4; // kQS stages of 128 floats
  static constexpr int kBar = kDV + kQS * kBM * 4;
  static constexpr int kBytes = kBar + 256;
  static constexpr uint32_t kColDV = 0, kColDK = 64, kColS = 128, kColDP = 256, kColS2 = 384;
  // barriers
  static constexpr int kKVFull = 0;                // +buffer
  static constexpr int kKVEmpty = 2;               // +buffer
  static constexpr int kQFull = 4;                 // +stage
  static constexpr int kQEmpty = kQFull + kQS;     // +stage
  static constexpr int kSFull = kQEmpty + kQS;
  static constexpr int kSFull2 = kSFull + 1;
  static constexpr int kDPFull = kSFull + 2;
  static constexpr int kPdsFull = kSFull + 3;
  static constexpr int kDqFull = kSFull + 4;
  static constexpr int kDqDrained = kSFull + 5;
  static constexpr int kDKVFull = kSFull + 6;      // a unit's dK and dV are complete
  static constexpr int kDKVEmpty = kSFull + 7;     // ... and have been read out
  static constexpr int kMmaDone = kSFull + 8;
  static constexpr int kNumBars = kSFull + 9;
};
static_assert(BwdCfgP64::kBytes <= 232448, "shared memory exceeds the 227 KB a CTA may use");
static_assert(8 * BwdCfgP64::kNumBars + 8 <= 256, "barrier block too small");

template <bool RAGGED, bool F16>
__global__ void __launch_bounds__(kThreads, 1) fa_bwd_bf16_persist64_kernel(const __grid_constant__ BwdArgs a) {
  constexpr int D = 64, DR = 64;
  using C = BwdCfgP64;
  constexpr int QS = C::kQS;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t sbase = smem_u32(smem_raw);
  uint8_t* sgen = smem_raw;
  if (sbase & 1023u) {
    if (threadIdx.x == 0) atomicCAS(a.fault, 0u, site(0));
    return;
  }
  const uint32_t bars = sbase + C::kBar;
  auto bar = [&](int i) -> uint32_t { return bars + 8u * (uint32_t)i; };
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sgen + C::kBar + 8 * C::kNumBars);
  int* abort_flag = reinterpret_cast<int*>(sgen + C::kBar + 8 * C::kNumBars + 4);
  const WaitCtx wc{abort_flag, a.fault};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int Nq = a.Nq, Nk = a.Nk;
  const int n_kv = (Nk + kBN - 1) / kBN;                           // K/V tiles per head
  const int n = RAGGED ? (Nq + kBM - 1) / kBM : Nq / kBM;          // query tiles per head = steps per unit
  const int units = a.B * a.H * n_kv;
  // This CTA's units and steps: unit k (k-th of the CTA) is u = blockIdx.x + k·gridDim.x;
  // step g of the CTA is step g mod n of its unit g / n.
  const int my_units = (int)blockIdx.x < units ? (units - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  const int total = my_units * n;
  auto unit_of = [&](int k) -> int { return (int)blockIdx.x + k * (int)gridDim.x; };
  auto s_cols = [](int g) -> uint32_t { return (g & 1) ? C::kColS2 : C::kColS; };
  auto s_bar_id = [](int g) -> int { return (g & 1) ? C::kSFull2 : C::kSFull; };
  auto s_parity = [](int g) -> uint32_t { return (uint32_t)((g >> 1) & 1); };
  auto load_rows = [&](uint32_t dst, const CUtensorMap* map, uint32_t bar_addr, int x, int pos, int nrows, int bh) {
    bool chk = dcheck(smem_ok(dst - sbase, kBox, (uint32_t)C::kBar, 1024), wc, kChkSmem, 40) &&
               dcheck(tma_x_ok(x, 64, D), wc, kChkTmaX, 40);
    if constexpr (RAGGED)
      chk = chk && dcheck(tma_head_ok(pos, nrows, bh, a.B * a.H), wc, kChkTmaRows, 40);
    else
      chk = chk && dcheck(tma_rows_ok((long long)bh * nrows + pos, 128, (long long)a.B * a.H * nrows), wc,
                          kChkTmaRows, 40);
    if (!chk) {
      mbar_complete_tx(bar_addr, kBox);
      return;
    }
    if constexpr (RAGGED)
      tma_load_3d(dst, map, bar_addr, x, pos, bh);
    else
      tma_load_2d(dst, map, bar_addr, x, bh * nrows + pos);
  };
  auto load_bulk = [&](uint32_t dst, const float* src, uint32_t bytes, uint32_t bar_addr) {
    if (!dcheck(smem_ok(dst - sbase, bytes, (uint32_t)C::kBar, 16) &&
                    bulk_ok(reinterpret_cast<uint64_t>(src), dst, bytes), wc, kChkBulk, 41)) {
      mbar_complete_tx(bar_addr, bytes);
      return;
    }
    bulk_load(dst, src, bytes, bar_addr);
  };
  // Workspace row of query 0 of head bh (whole tiles per head when ragged).
  auto wrow_of = [&](int bh) -> int { return RAGGED ? bh * n * kBM : bh * Nq; };

  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(C::kKVFull + b), 1);
      mbar_init(bar(C::kKVEmpty + b), 1);
    }
    for (int s = 0; s < QS; ++s) {
      mbar_init(bar(C::kQFull + s), 1);
      mbar_init(bar(C::kQEmpty + s), 1 + 32 * kComputeWarps);   // the MMA thread and the compute warps
    }
    mbar_init(bar(C::kSFull), 1);
    mbar_init(bar(C::kSFull2), 1);
    mbar_init(bar(C::kDPFull), 1);
    mbar_init(bar(C::kPdsFull), 32 * kComputeWarps);
    mbar_init(bar(C::kDqFull), 1);
    mbar_init(bar(C::kDqDrained), 32 * kRedWarps);
    mbar_init(bar(C::kDKVFull), 1);
    mbar_init(bar(C::kDKVEmpty), 32 * kComputeWarps);
    mbar_init(bar(C::kMmaDone), 1);
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
    // ------------------------------------------------------------ Pᵀ, dSᵀ, and each unit's dK, dV
    setmaxnreg_inc<kRegsCompute>();
    const int gq = warp & 3;
    const int h = warp >> 2;                       // query columns [64h, 64h + 64)
    const int r = gq * 32 + lane;                  // key row within the tile = TMEM lane
    const uint32_t lane_off = (uint32_t)(gq * 32) << 16;
    const float sl2 = a.scale_log2;
    const uint32_t ds_tile = sbase + C::kDS;
    const uint64_t sl2x2 = f2_pack(sl2, sl2);
    bool ok = true;
    // Unit k of this CTA, step i within it, Q/dO stage st of step g and the
    // parity of that stage's use, all kept incrementally (no divisions).
    int k = 0, i = 0, st = 0, qph = 0;
    int bh = 0, kv0 = 0, dead_lim = 0;
    bool dead_key = false, ragged_cta = false;
    for (int g = 0; g < total; ++g) {
      if (i == 0) {
        const int u = unit_of(k);
        bh = u / n_kv;
        kv0 = (u - bh * n_kv) * kBN;
        dead_key = RAGGED && kv0 + r >= Nk;
        ragged_cta = RAGGED && kv0 + kBN > Nk;
        dead_lim = dead_key ? (1 << 30) : -(1 << 30);
      }
      const int kv = kv0 + r;
      const uint32_t scol = s_cols(g);
      ok = mbar_wait_inl(bar(s_bar_id(g)), s_parity(g), wc, site(40)) &&
           mbar_wait_inl(bar(C::kQFull + st), (uint32_t)qph, wc, site(41));
      ok = __all_sync(kFull, ok);
      const uint64_t* nlse = reinterpret_cast<const uint64_t*>(sgen + C::kLSE + st * kBM * 4);
      const uint64_t* ndv = reinterpret_cast<const uint64_t*>(sgen + C::kDV + st * kBM * 4);
      uint64_t p[32];
      if (ok) {
        tc_fence_after();
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
          const int c0 = h * 64 + ch * 32;
          uint32_t s[32];
          if (dcheck(tmem_ok(scol + c0, 32, 512), wc, kChkTmem, 40))
            tmem_ld_x32(tmem + lane_off + scol + (uint32_t)c0, s);
          if (ragged_cta)
            p_chunk<true, 0>(s, sl2x2, nlse + (c0 >> 1), dead_lim, p + ch * 16);
          else
            p_chunk<false, kPolyEvery>(s, sl2x2, nlse + (c0 >> 1), r - c0, p + ch * 16);
        }
      }
      if (ok) ok = mbar_wait_inl(bar(C::kDPFull), (uint32_t)(g & 1), wc, site(42));
      ok = pair_sync_and(1 + gq, ok);
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float a0, a1;
          f2_unpack(p[half * 16 + e], a0, a1);
          pk[e] = pack2<F16>(a0, a1);
        }
        if (dcheck(tmem_ok(scol + h * 32 + 16 * half, 16, 512), wc, kChkTmem, 41))
          tmem_st_x16(tmem + lane_off + scol + (uint32_t)(h * 32 + 16 * half), pk);
      }
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        const int c0 = h * 64 + ch * 32;
        uint32_t dp[32];
        if (dcheck(tmem_ok(C::kColDP + c0, 32, 512), wc, kChkTmem, 42))
          tmem_ld_x32(tmem + lane_off + C::kColDP + (uint32_t)c0, dp);
        uint32_t dk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const uint64_t ds = f2_mul(p[ch * 16 + e], f2_add(f2_pack(u2f(dp[2 * e]), u2f(dp[2 * e + 1])), ndv[(c0 >> 1) + e]));
          float d0, d1;
          f2_unpack(ds, d0, d1);
          dk[e] = pack2<F16>(d0, d1);
        }
        const uint32_t row_addr = ds_tile + (uint32_t)(h * kBox + r * 128);
        if (!dcheck(smem_ok(row_addr - sbase, 128, (uint32_t)C::kBar, 128), wc, kChkSmem, 43)) continue;
#pragma unroll
        for (int w4 = 0; w4 < 4; ++w4) {
          const int chunk = ch * 4 + w4;
          st_shared_v4(row_addr + (uint32_t)(((chunk ^ (r & 7)) & 7) * 16), dk[4 * w4], dk[4 * w4 + 1],
                       dk[4 * w4 + 2], dk[4 * w4 + 3]);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      fence_proxy_async_smem();
      mbar_arrive(bar(C::kPdsFull));
      mbar_arrive(bar(C::kQEmpty + st));
      if (i == n - 1) {
        // The unit's dK and dV: read them out (then the next unit's first
        // dK and dV products may start the accumulators afresh) and store.
        ok = mbar_wait_inl(bar(C::kDKVFull), (uint32_t)(k & 1), wc, site(43));
        ok = __all_sync(kFull, ok);
        if (!ok) break;
        tc_fence_after();
        const uint32_t col = h == 0 ? C::kColDV : C::kColDK;
        const float mul = h == 0 ? 1.0f : a.scale;
        uint32_t v0[32], v1[32];
        if (dcheck(tmem_ok(col, 64, 512), wc, kChkTmem, 44)) {
          tmem_ld_x32(tmem + lane_off + col, v0);
          tmem_ld_x32(tmem + lane_off + col + 32, v1);
        }
        tc_fence_before();
        mbar_arrive(bar(C::kDKVEmpty));
        uint16_t* dst = static_cast<uint16_t*>(h == 0 ? a.dv : a.dk) + ((size_t)bh * (size_t)Nk + (size_t)kv) * DR;
        if (!dead_key) {
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const uint32_t x0 = cc ? v1[2 * e] : v0[2 * e], x1 = cc ? v1[2 * e + 1] : v0[2 * e + 1];
              pk[e] = pack2<F16>(u2f(x0) * mul, u2f(x1) * mul);
            }
#pragma unroll
            for (int w4 = 0; w4 < 4; ++w4)
              st_global_v4(dst + 32 * cc + 8 * w4, pk[4 * w4], pk[4 * w4 + 1], pk[4 * w4 + 2], pk[4 * w4 + 3]);
          }
        }
      }
      if (++st == QS) {
        st = 0;
        qph ^= 1;
      }
      if (++i == n) {
        i = 0;
        ++k;
      }
    }
    tc_fence_before();
    named_bar_arrive(kEndBarrier, kThreads);
  } else if (warp < kRedWarp + kRedWarps) {
    // ------------------------------------------------------------ dQ reductions (as in the d = 64 kernel)
    setmaxnreg_dec<kRegsRed>();
    const int gq = warp & 3;
    const int r = gq * 32 + lane;
    const uint32_t lane_off = (uint32_t)(gq * 32) << 16;
    uint32_t t_prev = 0;
    uint32_t pause_ns = 0;
    int k = 0, i = 0, wrow0 = wrow_of(unit_of(0) / n_kv);
    for (int g = 0; g < total; ++g) {
      if (g > 0 && ++i == n) {
        i = 0;
        ++k;
        wrow0 = wrow_of(unit_of(k) / n_kv);
      }
      bool ok = mbar_wait_inl(bar(C::kDqFull), (uint32_t)(g & 1), wc, site(44));
      ok = __all_sync(kFull, ok);
      if (!ok) break;
      {
        const uint32_t t_now = (uint32_t)clock();
        if (g > 0) {
          const uint32_t pp = (t_now - t_prev) / 40u;
          pause_ns = pp < 200u ? pp : 200u;
        }
        t_prev = t_now;
      }
      tc_fence_after();
      uint32_t v[64];
      const uint32_t dq_col = s_cols(g) + 64u;
      const bool chk = dcheck(tmem_ok(dq_col, 64, 512), wc, kChkTmem, 45);
      if (chk) tmem_ld_x64(tmem + lane_off + dq_col, v);
      tc_fence_before();
      mbar_arrive(bar(C::kDqDrained));
      if (!chk) continue;
      float* base = a.dqacc + ((size_t)wrow0 + (size_t)(i * kBM) + (size_t)r) * D;
#pragma unroll
      for (int c = 0; c < 64; c += 4) {
        red_add_v4_f32(base + c, u2f(v[c]), u2f(v[c + 1]), u2f(v[c + 2]), u2f(v[c + 3]));
        if (c < 60 && pause_ns > 0) __nanosleep(pause_ns / 3u);
      }
    }
    tc_fence_before();
    named_bar_arrive(kEndBarrier, kThreads);
  } else {
  setmaxnreg_dec<kRegsMisc>();
  if (warp == kTmaWarp) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tmap(&a.tm_q);
      prefetch_tmap(&a.tm_k);
      prefetch_tmap(&a.tm_v);
      prefetch_tmap(&a.tm_do);
      int issued_kv[2] = {}, issued_q[QS] = {};
      int g = 0;
      bool ok = true;
      for (int k = 0; ok && k < my_units; ++k) {
        const int u = unit_of(k);
        const int bh = u / n_kv, kv0 = (u % n_kv) * kBN;
        const int b = k & 1;
        // Buffer b last held unit k − 2: its products must be done.
        if (k >= 2 && !mbar_wait_inl(bar(C::kKVEmpty + b), (uint32_t)(((k >> 1) - 1) & 1), wc, site(45))) break;
        mbar_arrive_expect_tx(bar(C::kKVFull + b), 2u * C::kTile);
        load_rows(sbase + C::kK + b * C::kTile, &a.tm_k, bar(C::kKVFull + b), 0, kv0, Nk, bh);
        load_rows(sbase + C::kV + b * C::kTile, &a.tm_v, bar(C::kKVFull + b), 0, kv0, Nk, bh);
        ++issued_kv[b];
        const int wrow0 = wrow_of(bh);
        for (int i = 0; i < n; ++i, ++g) {
          const int s = g % QS;
          if (g >= QS && !mbar_wait_inl(bar(C::kQEmpty + s), (uint32_t)((g / QS - 1) & 1), wc, site(46))) {
            ok = false;
            break;
          }
          const int q0 = i * kBM;
          mbar_arrive_expect_tx(bar(C::kQFull + s), 2u * C::kTile + 2u * kBM * 4);
          load_rows(sbase + C::kQ + s * C::kTile, &a.tm_q, bar(C::kQFull + s), 0, q0, Nq, bh);
          load_rows(sbase + C::kDO + s * C::kTile, &a.tm_do, bar(C::kQFull + s), 0, q0, Nq, bh);
          load_bulk(sbase + C::kLSE + s * kBM * 4, a.lse2 + wrow0 + q0, kBM * 4, bar(C::kQFull + s));
          load_bulk(sbase + C::kDV + s * kBM * 4, a.dvec + wrow0 + q0, kBM * 4, bar(C::kQFull + s));
          ++issued_q[s];
        }
      }
      for (int b = 0; b < 2; ++b)
        if (issued_kv[b] > 0) mbar_wait_drain_inl(bar(C::kKVFull + b), (uint32_t)((issued_kv[b] - 1) & 1), wc, site(47));
      for (int s = 0; s < QS; ++s)
        if (issued_q[s] > 0) mbar_wait_drain_inl(bar(C::kQFull + s), (uint32_t)((issued_q[s] - 1) & 1), wc, site(47));
    }
    __syncwarp();
    named_bar_arrive(kEndBarrier, kThreads);
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_f16kind(128, kBM, false, false, F16);  // Sᵀ = K Qᵀ, dPᵀ = V dOᵀ
      constexpr uint32_t kIdKV = idesc_f16kind(128, DR, false, true, F16);   // dV += Pᵀ dO, dK += dSᵀ Q
      constexpr uint32_t kIdQ = idesc_f16kind(128, D, true, true, F16);      // dQ = dS K (M = queries, N = 64)
      int kv_ready = -1;          // last unit whose K/V tile was seen complete
      auto need_kv = [&](int k) -> bool {
        if (kv_ready >= k) return true;
        if (!mbar_wait_inl(bar(C::kKVFull + (k & 1)), (uint32_t)((k >> 1) & 1), wc, site(48))) return false;
        kv_ready = k;
        return true;
      };
      // Sᵀ (A = K) or dPᵀ (A = V) of a step whose unit uses K/V buffer b and
      // whose Q/dO sit in stage st, into `col`.
      auto issue_sd = [&](int b, int st, uint32_t col, bool scores) {
        const uint32_t a_tile = sbase + (scores ? C::kK : C::kV) + b * C::kTile;
        const uint32_t b_tile = sbase + (scores ? C::kQ : C::kDO) + st * C::kTile;
        if (!(dcheck(tmem_ok(col, kBM, 512), wc, kChkTmem, 46) &&
              dcheck(smem_ok(a_tile - sbase, C::kTile, C::kBar, 1024), wc, kChkSmem, 46) &&
              dcheck(smem_ok(b_tile - sbase, C::kTile, C::kBar, 1024), wc, kChkSmem, 46)))
          return;
#pragma unroll
        for (int ks = 0; ks < DR / 16; ++ks)
          mma_ss(tmem + col, sdesc_sw128(a_tile + (uint32_t)(ks * 32), 16, 1024),
                 sdesc_sw128(b_tile + (uint32_t)(ks * 32), 16, 1024), kIdS, ks > 0 ? 1u : 0u);
      };
      bool ok = total > 0 && need_kv(0) && mbar_wait_inl(bar(C::kQFull), 0, wc, site(49));
      if (ok) {
        tc_fence_after();
        issue_sd(0, 0, s_cols(0), true);
        tc_commit(bar(s_bar_id(0)));
        issue_sd(0, 0, C::kColDP, false);
        tc_commit(bar(C::kDPFull));
        if (total > 1) {
          const int k1 = n == 1 ? 1 : 0;
          ok = need_kv(k1) && mbar_wait_inl(bar(C::kQFull + 1), 0, wc, site(49));
          if (ok) {
            tc_fence_after();
            issue_sd(k1 & 1, 1, s_cols(1), true);
            tc_commit(bar(s_bar_id(1)));
          }
        }
      }
      // Unit k, step i within it and Q/dO stage st of step g, kept incrementally.
      int k = 0, i = 0, st = 0;
      for (int g = 0; ok && g < total; ++g) {
        const int b = k & 1;
        if (!mbar_wait_inl(bar(C::kPdsFull), (uint32_t)(g & 1), wc, site(50))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t ds = sbase + C::kDS;
        const uint32_t kb = sbase + C::kK + b * C::kTile;
        const uint32_t qb = sbase + C::kQ + st * C::kTile;
        const uint32_t ob = sbase + C::kDO + st * C::kTile;
        const uint32_t sb = s_cols(g);
        const bool chk = dcheck(tmem_ok(sb, 128, 512) && tmem_ok(C::kColDV, DR, 512) && tmem_ok(C::kColDK, DR, 512),
                                wc, kChkTmem, 47) &&
                         dcheck(smem_ok(C::kDS, 2 * kBox, C::kBar, 1024) && smem_ok(qb - sbase, C::kTile, C::kBar, 1024) &&
                                    smem_ok(ob - sbase, C::kTile, C::kBar, 1024) &&
                                    smem_ok(kb - sbase, C::kTile, C::kBar, 1024),
                                wc, kChkSmem, 47);
        // dQ = dS K into the spent half of this step's score buffer.
#pragma unroll
        for (int ks = 0; ks < kBN / 16; ++ks) {
          if (!chk) break;
          mma_ss(tmem + sb + 64u, sdesc_sw128(ds + (uint32_t)(ks * 2048), kBox, 1024),
                 sdesc_sw128(kb + (uint32_t)(ks * 2048), kBox, 1024), kIdQ, ks > 0 ? 1u : 0u);
        }
        tc_commit(bar(C::kDqFull));
        // The unit's first dK and dV start the accumulators afresh: the
        // previous unit's must have been read out.
        if (i == 0 && k > 0 && !mbar_wait_inl(bar(C::kDKVEmpty), (uint32_t)((k - 1) & 1), wc, site(51))) {
          ok = false;
          break;
        }
#pragma unroll
        for (int ks = 0; ks < kBM / 16; ++ks)
          if (chk) mma_ss(tmem + C::kColDK, sdesc_sw128(ds + (uint32_t)((ks >> 2) * kBox + (ks & 3) * 32), 16, 1024),
                 sdesc_sw128(qb + (uint32_t)(ks * 2048), kBox, 1024), kIdKV, (i > 0 || ks > 0) ? 1u : 0u);
        const int st1 = st + 1 == QS ? 0 : st + 1;
        if (g + 1 < total) {
          // Its Q/dO stage and K/V buffer were waited for when its scores were issued.
          issue_sd(i + 1 == n ? (b ^ 1) : b, st1, C::kColDP, false);
          tc_commit(bar(C::kDPFull));
        }
#pragma unroll
        for (int ks = 0; ks < kBM / 16; ++ks)
          if (chk) mma_ts(tmem + C::kColDV, tmem + sb + (uint32_t)(8 * ks),
                 sdesc_sw128(ob + (uint32_t)(ks * 2048), kBox, 1024), kIdKV, (i > 0 || ks > 0) ? 1u : 0u);
        tc_commit(bar(C::kQEmpty + st));
        if (i == n - 1) {
          tc_commit(bar(C::kDKVFull));
          tc_commit(bar(C::kKVEmpty + b));
        }
        if (g + 2 < total) {
          // Step g + 2 belongs to unit k + (i + 2) / n (two units on when n = 1).
          const int k2 = k + (i + 2 >= n ? 1 : 0) + (n == 1 ? 1 : 0);
          const int st2 = st1 + 1 == QS ? 0 : st1 + 1;
          if (!need_kv(k2) ||
              !mbar_wait_inl(bar(C::kQFull + st2), (uint32_t)(((g + 2) / QS) & 1), wc, site(52)) ||
              !mbar_wait_inl(bar(C::kDqDrained), (uint32_t)(g & 1), wc, site(53))) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_sd(k2 & 1, st2, sb, true);
          tc_commit(bar(s_bar_id(g)));
        }
        st = st1;
        if (++i == n) {
          i = 0;
          ++k;
        }
      }
      tc_commit(bar(C::kMmaDone));
      mbar_wait_drain_inl(bar(C::kMmaDone), 0, wc, site(54));
    }
    __syncwarp();
    named_bar_sync(kEndBarrier, kThreads);
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  } else {
    named_bar_arrive(kEndBarrier, kThreads);   // warps 14, 15
  }
  }
}

template <bool RAGGED, bool F16>
cudaError_t launch_persist64(const BwdArgs& a, cudaStream_t s) {
  auto kern = fa_bwd_bf16_persist64_kernel<RAGGED, F16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)BwdCfgP64::kBytes);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)a.persist_ctas, kThreads, BwdCfgP64::kBytes, s>>>(a);
  return cudaGetLastError();
}

template <int DR, bool CAUSAL, bool RAGGED, bool F16>
cudaError_t launch_impl(const BwdArgs& a, cudaStream_t s) {
  auto kern = fa_bwd_bf16_kernel<DR, CAUSAL, RAGGED, F16>;
  const size_t smem = BwdCfg<(DR <= 64 ? 64 : 128)>::kBytes;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const unsigned tiles = (unsigned)((a.Nk + kBN - 1) / kBN), heads = (unsigned)(a.B * a.H);
  const dim3 grid = CAUSAL ? dim3(heads, tiles) : dim3(tiles, heads);
  kern<<<grid, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ pre-pass and dQ finish

// Grid (n_pad·D/8 / 256, heads): one group of D/8 threads per workspace row
// (n_pad rows per head, a multiple of 128, so every thread has a row); each
// thread reads 8 16-bit elements of O and of dO (16 bytes each), so a warp
// covers 32·8 contiguous elements.  Rows past Nq in a head are padding: D = 0,
// −LSE = −∞.
// DR = 96: groups of 16 threads (a power of two, for the shuffle sum) of
// which the last 4 hold no columns.
template <int DR, bool F16>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const uint16_t* __restrict__ o,
                                                       const uint16_t* __restrict__ dO,
                                                       const float* __restrict__ lse, float* __restrict__ dvec,
                                                       float* __restrict__ lse2, float* __restrict__ dqacc, int Nq,
                                                       int n_pad) {
  constexpr int G = DR == 96 ? 16 : DR / 8;   // threads per row
  const int tid = (int)(blockIdx.x * blockDim.x + threadIdx.x);
  const int pos = tid / G;                  // row within the head
  const int part = tid % G;
  const bool has_cols = part * 8 < DR;
  const long long head = blockIdx.y;
  const long long row = head * n_pad + pos;   // workspace row
  const long long src = head * Nq + pos;       // row of O, dO and LSE
  const bool live = pos < Nq;
  float acc = 0.f;
  if (has_cols && dqacc != nullptr) {
    float4* z = reinterpret_cast<float4*>(dqacc + row * DR + part * 8);
    z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if (live && has_cols) {
    const uint4 ov = *reinterpret_cast<const uint4*>(o + src * DR + part * 8);
    const uint4 gv = *reinterpret_cast<const uint4*>(dO + src * DR + part * 8);
    const uint32_t op[4] = {ov.x, ov.y, ov.z, ov.w};
    const uint32_t gp[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 a2 = unpack2<F16>(op[i]);
      const float2 b2 = unpack2<F16>(gp[i]);
      acc = fmaf(a2.x, b2.x, acc);
      acc = fmaf(a2.y, b2.y, acc);
    }
  }
#pragma unroll
  for (int off = G / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(kFull, acc, off);
  if (part == 0) {
    // Stored negated: the tiled kernel adds them with packed f32x2 operations.
    dvec[row] = live ? -acc : 0.f;
    lse2[row] = live ? -lse[src] * 1.4426950408889634074f : -INFINITY;
  }
}

// Grid (⌈Nq·D/8 / 256⌉, heads): one thread per 8 consecutive dQ elements of a
// row below Nq; the accumulator has n_pad rows per head, dQ has Nq.
template <int DR, bool F16>
__global__ void __launch_bounds__(256) dq_finish_kernel(const float* __restrict__ acc, uint16_t* __restrict__ dq,
                                                        int Nq, int n_pad, float scale) {
  constexpr int G = DR / 8;
  const int tid = (int)(blockIdx.x * blockDim.x + threadIdx.x);
  const int pos = tid / G;
  if (pos >= Nq) return;
  const int part = tid % G;
  const long long head = blockIdx.y;
  const long long arow = head * n_pad + pos;
  const long long i = (head * Nq + pos) * G + part;   // 16-byte chunk of dQ
  const float4* a = reinterpret_cast<const float4*>(acc + arow * DR + part * 8);
  const float4 a0 = a[0];
  const float4 a1 = a[1];
  uint4 out;
  out.x = pack2<F16>(a0.x * scale, a0.y * scale);
  out.y = pack2<F16>(a0.z * scale, a0.w * scale);
  out.z = pack2<F16>(a1.x * scale, a1.y * scale);
  out.w = pack2<F16>(a1.z * scale, a1.w * scale);
  reinterpret_cast<uint4*>(dq)[i] = out;
}

}  // namespace

int bwd_bf16_block_m(int) { return kBM; }

int bwd_kv_box_rows(int d) { return d == 256 ? 64 : kBN; }

size_t bwd_bf16_smem_bytes(int d) { return d <= 64 ? BwdCfg<64>::kBytes : BwdCfg<128>::kBytes; }

template <bool F16>
static cudaError_t dispatch_bwd(const BwdArgs& a, bool ragged, cudaStream_t s) {
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

cudaError_t launch_bwd_bf16(const BwdArgs& a, cudaStream_t s) {
  if (a.d == 256) return launch_bwd_d256(a, s);
  const bool ragged = a.Nq % kBM != 0 || a.Nk % kBN != 0;
  if (a.persist_ctas > 0 && a.d == 64 && !a.causal) {
    if (a.f16) return ragged ? launch_persist64<true, true>(a, s) : launch_persist64<false, true>(a, s);
    return ragged ? launch_persist64<true, false>(a, s) : launch_persist64<false, false>(a, s);
  }
  return a.f16 ? dispatch_bwd<true>(a, ragged, s) : dispatch_bwd<false>(a, ragged, s);
}

template <int D, bool F16>
static void launch_prep(dim3 grid, const void* o, const void* dO, const float* lse, float* dvec, float* lse2,
                        float* dqacc, int Nq, int n_pad, cudaStream_t s) {
  bwd_prep_kernel<D, F16><<<grid, 256, 0, s>>>(static_cast<const uint16_t*>(o), static_cast<const uint16_t*>(dO), lse,
                                               dvec, lse2, dqacc, Nq, n_pad);
}

cudaError_t launch_bwd_prep_bf16(const void* o, const void* dO, const float* lse, float* dvec, float* lse2,
                                 float* dqacc, long long heads, int Nq, int n_pad, int d, int f16, cudaStream_t s) {
  if (heads <= 0 || heads > 65535 || n_pad % 128 != 0) return cudaErrorInvalidValue;
  const int threads_per_row = d == 96 ? 16 : d / 8;
  const dim3 grid((unsigned)((long long)n_pad * threads_per_row / 256), (unsigned)heads);
  if (d == 256)
    f16 ? launch_prep<256, true>(grid, o, dO, lse, dvec, lse2, dqacc, Nq, n_pad, s)
        : launch_prep<256, false>(grid, o, dO, lse, dvec, lse2, dqacc, Nq, n_pad, s);
  else if (d == 128)
    f16 ? launch_prep<128, true>(grid, o, dO, lse, dvec, lse2, dqacc, Nq, n_pad, s)
        : launch_prep<128, false>(grid, o, dO, lse, dvec, lse2, dqacc, Nq, n_pad, s);
  else if (d == 96)
    f16 ? launch_prep<96, true>(grid, o, dO, lse, dvec, lse2, dqacc, Nq, n_pad, s)
        : launch_prep<96, false>(grid, o, dO, lse, dvec, lse2, dqacc, Nq, n_pad, s);
  else if (d == 64)
    f16 ? launch_prep<64, true>(grid, o, dO, lse, dvec, lse2, dqacc, Nq, n_pad, s)
        : launch_prep<64, false>(grid, o, dO, lse, dvec, lse2, dqacc, Nq, n_pad, s);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

template <int D, bool F16>
static void launch_finish(dim3 grid, const float* dqacc, void* dq, int Nq, int n_pad, float scale, cudaStream_t s) {
  dq_finish_kernel<D, F16><<<grid, 256, 0, s>>>(dqacc, static_cast<uint16_t*>(dq), Nq, n_pad, scale);
}

cudaError_t launch_dq_finish_bf16(const float* dqacc, void* dq, long long heads, int Nq, int n_pad, int d, float scale,
                                  int f16, cudaStream_t s) {
  if (heads <= 0 || heads > 65535) return cudaErrorInvalidValue;
  const dim3 grid((unsigned)(((long long)Nq * (d / 8) + 255) / 256), (unsigned)heads);
  if (d == 128)
    f16 ? launch_finish<128, true>(grid, dqacc, dq, Nq, n_pad, scale, s)
        : launch_finish<128, false>(grid, dqacc, dq, Nq, n_pad, scale, s);
  else if (d == 96)
    f16 ? launch_finish<96, true>(grid, dqacc, dq, Nq, n_pad, scale, s)
        : launch_finish<96, false>(grid, dqacc, dq, Nq, n_pad, scale, s);
  else if (d == 64)
    f16 ? launch_finish<64, true>(grid, dqacc, dq, Nq, n_pad, scale, s)
        : launch_finish<64, false>(grid, dqacc, dq, Nq, n_pad, scale, s);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace fa
