// fa_kernels.h — launch parameters and host launchers shared between the C-ABI
// layer (fa_abi.cu) and the kernel translation units.  Internal to libfa.so.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <mutex>

namespace fa {

// ---------------------------------------------------------------- device addresses of library arrays

// A device address that cudaGetSymbolAddress returns belongs to the context
// that was current: after cudaDeviceReset (or any teardown of the primary
// context) the next context loads the module again and the array may sit
// elsewhere.  So a cached address is kept together with the id of the context
// it was looked up in, per device, and looked up again when that id changes.
constexpr int kMaxDevices = 64;
struct SymbolCache {
  std::mutex mu;
  unsigned long long ctx[kMaxDevices] = {};
  void* ptr[kMaxDevices] = {};
};
// Id of the context current on the calling thread (cuCtxGetId), 0 if there is
// none yet or it cannot be queried.
unsigned long long current_context_id();
// The address cached for the current device and context, or the result of
// `lookup` (a function in the array's own translation unit that calls
// cudaGetSymbolAddress on it), cached.  Returns null, with the runtime's
// last error cleared, if the lookup fails.
void* cached_symbol_address(SymbolCache& cache, void* (*lookup)());

// ---------------------------------------------------------------- bf16 tensor-core path

// Q, O, dO, dQ are [B·H, Nq, d]; K, V, dK, dV are [B·H, Nk, d]; LSE [B·H, Nq].
// Under the causal mask query i sees keys j ≤ i + Nk − Nq (Nq ≤ Nk).
//
// Forward: tensor maps over Q, K, V with boxes of 64 columns (128 bytes) ×
// 128 rows and 128-byte swizzle: 2-D over the [B·H·Nq, d] / [B·H·Nk, d] row
// views when Nq and Nk are multiples of 128, else 3-D over [B·H, N, d] with
// rows past N read as zero.
// Element type of the 16-bit tensors: bf16, or fp16 when f16 = 1.
struct FwdArgs {
  CUtensorMap tm_q, tm_k, tm_v;
  void* o;                // [B·H, Nq, d] in the 16-bit type
  float* lse;
  int B, H, Nq, Nk, d;
  int f16;
  float scale_log2;       // scale · log2(e): scores are handled in base 2
  int causal;
  unsigned int* fault;
  // Load balancing: units [0, n_full) run whole; each of the remaining
  // units runs as `splits` CTAs over K/V sub-ranges writing fp32 partials
  // (opart [slots·part_rows, d], lpart [slots·part_rows]; part_rows ≤ the
  // unit's rows: every row of a unit, or only the queries that exist when a
  // problem has at most 128) that a combine kernel merges.  splits = 1 (or
  // n_full = all units) disables it.  Under the causal mask only problems
  // with at most 128 queries split (the d ≤ 128 kernel).
  int n_full, splits, part_rows;
  float* opart;
  float* lpart;
  // > 0: the persistent forward (d ≤ 128, no mask, no split) on this many
  // CTAs, each walking the units with a stride of persist_ctas.
  int persist_ctas;
};
// Largest K/V tile count per unit for which the forward runs persistent when
// there are more units than SMs (its start-up and drain then weigh most).
constexpr int kFwdPersistMaxTiles = 16;
// Work units of the forward: 256 query rows (two tiles) per CTA, 128 at d = 256.
int fwd_unit_rows(int d);
int fwd_units(int B, int H, int Nq, int d);
// Split plan for `units` equal units of `n_kv` K/V tiles on `num_sms` SMs: the
// units of the last, partial wave are split when that fills the GPU better.
void fwd_split_plan(int units, int num_sms, int n_kv, int* n_full, int* splits);
// Parts per unit for a problem with at most 128 queries and fewer units
// than SMs, every unit split over its n_kv visible K/V tiles.
int fwd_split_short(int units, int num_sms, int n_kv);
size_t fwd_bf16_smem_bytes(int d);
// Dispatches on d (64, 96, 128; 256 goes to launch_fwd_d256).
cudaError_t launch_fwd_bf16(const FwdArgs& a, cudaStream_t s);
// d = 256: one 128-row query tile per CTA, double-buffered scores.
cudaError_t launch_fwd_d256(const FwdArgs& a, cudaStream_t s);
// Merges the fp32 partials of the `tail` split units (unit_rows rows each).
cudaError_t launch_fwd_combine(const FwdArgs& a, int tail, int unit_rows, cudaStream_t s);

// Backward tiled loop.  Tensor maps as in the forward (128-row boxes).
// The workspace arrays hold n_pad = 128·⌈Nq/128⌉ rows per head.
struct BwdArgs {
  CUtensorMap tm_q, tm_k, tm_v, tm_do;
  const float* lse2;      // workspace: −LSE · log2(e), [B·H·n_pad]
  const float* dvec;      // workspace: −D = −rowsum(dO ⊙ O), [B·H·n_pad]
  float* dqacc;           // workspace: fp32 dQ accumulator, [B·H·n_pad, d] (not used at d = 256)
  void* dq;               // [B·H, Nq, d], written directly at d = 256 (else by the finish pass)
  void* dk;               // [B·H, Nk, d] in the 16-bit type
  void* dv;
  int B, H, Nq, Nk, d;
  int f16;
  float scale_log2;
  float scale;
  int causal;
  unsigned int* fault;
  // > 0: the persistent backward (d = 64, no mask) on this many CTAs, each
  // walking the K/V tiles with a stride of persist_ctas.
  int persist_ctas;
};
// Largest query-tile count per head for which the d = 64 backward runs
// persistent when there are more K/V tiles than SMs.  Measured on GB300
// (B·H·N fixed at 128·1024, d = 64): 2 tiles +13.5 %, 4 +7.7 %, 8 +1.2 %,
// 16 −4.1 % against one K/V tile per CTA: its steps are a little slower, so
// it pays only where a CTA's start-up and drain weigh most.
constexpr int kBwdPersistMaxTiles = 8;
int bwd_bf16_block_m(int d);
size_t bwd_bf16_smem_bytes(int d);
// Dispatches on d (64, 96, 128; 256 goes to launch_bwd_d256).
cudaError_t launch_bwd_bf16(const BwdArgs& a, cudaStream_t s);
// d = 256: a dK/dV kernel over 64-key tiles and a dQ kernel over 128-query
// tiles (K and V maps with 64-row boxes); dQ is written scaled, in the 16-bit
// type, so no accumulator and no finish pass.
cudaError_t launch_bwd_d256(const BwdArgs& a, cudaStream_t s);
// Rows of the K/V boxes the backward's tensor maps use.
int bwd_kv_box_rows(int d);

// Backward pre-pass: −D = −rowsum(dO ⊙ O) and −LSE·log2(e) per query row, dQ
// accumulator zeroed (dqacc may be null: d = 256 has none).  The workspace arrays hold n_pad ≥ Nq rows per head
// (whole 128-row tiles); padding rows get −LSE = −∞ (so P = 0) and D = 0.
cudaError_t launch_bwd_prep_bf16(const void* o, const void* dO, const float* lse, float* dvec, float* lse2,
                                 float* dqacc, long long heads, int Nq, int n_pad, int d, int f16, cudaStream_t s);
// dQ = scale · accumulator (n_pad rows per head), rounded to the 16-bit type [heads, Nq, d].
cudaError_t launch_dq_finish_bf16(const float* dqacc, void* dq, long long heads, int Nq, int n_pad, int d, float scale,
                                  int f16, cudaStream_t s);

// ---------------------------------------------------------------- merge of partial results

// O = Σ_k e^{LSE_k − LSE} O_k, LSE = ln Σ_k e^{LSE_k} over n_parts partial
// results of the same rows ([rows, d] in the dtype, LSE fp32 [rows]).  Rows
// every part missed (LSE_k = −∞) get O = 0, LSE = −∞.  `o` / `lse` may be one
// of the parts (each row is read completely before it is written).
constexpr int kMaxMergeParts = 16;
struct MergeArgs {
  const void* o_parts[kMaxMergeParts];
  const float* lse_parts[kMaxMergeParts];
  int n_parts;
  void* o;
  float* lse;
  long long rows;
  int d;
  int elem;   // O element type: 0 fp32, 1 bf16, 2 fp16
};
cudaError_t launch_merge(const MergeArgs& a, cudaStream_t s);

// ---------------------------------------------------------------- self-test

// One CTA whose pipeline wait can never complete: the bounded wait gives up
// after its time limit and records a fault code in `fault` (no trap, no hang).
cudaError_t launch_wait_timeout_selftest(unsigned int* fault, cudaStream_t s);
// One thread evaluates the debug-build checks on FA_SELFTEST_BOUNDS_CASES fixed
// cases and writes 1 (passed) / 0 (failed) for each into `results`.
cudaError_t launch_bounds_check_selftest(unsigned int* fault, int* results, cudaStream_t s);

// ---------------------------------------------------------------- fp32 SIMT path

cudaError_t launch_fwd_f32(const float* q, const float* k, const float* v, float* o, float* lse, int BH, int Nq,
                           int Nk, int d, float scale, int causal, cudaStream_t s);
cudaError_t launch_bwd_prep_f32(const float* o, const float* dO, const float* lse, float* dvec, float* lse_copy,
                                long long rows, int d, cudaStream_t s);
cudaError_t launch_bwd_f32(const float* q, const float* k, const float* v, const float* dO, const float* lse,
                           const float* dvec, float* dq, float* dk, float* dv, int BH, int Nq, int Nk, int d,
                           float scale, int causal, cudaStream_t s);

}  // namespace fa
