// fa_kernels.h — launch parameters and host launchers shared between the C-ABI
// layer (fa_abi.cu) and the kernel translation units.  Internal to libfa.so.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace fa {

// ---------------------------------------------------------------- bf16 tensor-core path

// Forward: tensor maps over Q, K, V with boxes of 64 columns (128 bytes) ×
// 128 rows and 128-byte swizzle: 2-D over the [B·H·N, d] row view when N is a
// multiple of 128, else 3-D over [B·H, N, d] with rows past N read as zero.
struct FwdArgs {
  CUtensorMap tm_q, tm_k, tm_v;
  __nv_bfloat16* o;
  float* lse;
  int B, H, N, d;
  float scale_log2;       // scale · log2(e): scores are handled in base 2
  int causal;
  unsigned int* fault;
  // Non-causal load balancing: two-tile units [0, n_full) run whole; each of
  // the remaining units runs as `splits` CTAs over K/V sub-ranges writing
  // fp32 partials (opart [slots·256, d], lpart [slots·256]) that a combine
  // kernel merges.  splits = 1 (or n_full = all units) disables it.
  int n_full, splits;
  float* opart;
  float* lpart;
};
// Two-tile (256-query) work units of the forward.
int fwd_units(int B, int H, int N);
// Split plan for `units` equal units of `n_kv` K/V tiles on `num_sms` SMs: the
// units of the last, partial wave are split when that fills the GPU better.
void fwd_split_plan(int units, int num_sms, int n_kv, int* n_full, int* splits);
size_t fwd_bf16_smem_bytes(int d);
cudaError_t launch_fwd_bf16(const FwdArgs& a, cudaStream_t s);

// Backward tiled loop.  Tensor maps as in the forward (3-D, 128-row boxes).
// The workspace arrays hold n_pad = 128·⌈N/128⌉ rows per head.
struct BwdArgs {
  CUtensorMap tm_q, tm_k, tm_v, tm_do;
  const float* lse2;      // workspace: −LSE · log2(e), [B·H·n_pad]
  const float* dvec;      // workspace: −D = −rowsum(dO ⊙ O), [B·H·n_pad]
  float* dqacc;           // workspace: fp32 dQ accumulator, [B·H·n_pad, d]
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int B, H, N, d;
  float scale_log2;
  float scale;
  int causal;
  unsigned int* fault;
};
int bwd_bf16_block_m(int d);
size_t bwd_bf16_smem_bytes(int d);
cudaError_t launch_bwd_bf16(const BwdArgs& a, cudaStream_t s);

// Backward pre-pass: −D = −rowsum(dO ⊙ O) and −LSE·log2(e) per row, dQ
// accumulator zeroed.  The workspace arrays hold n_pad ≥ N rows per head
// (whole 128-row tiles); padding rows get −LSE = −∞ (so P = 0) and D = 0.
cudaError_t launch_bwd_prep_bf16(const __nv_bfloat16* o, const __nv_bfloat16* dO, const float* lse,
                                 float* dvec, float* lse2, float* dqacc, long long heads, int N, int n_pad, int d,
                                 cudaStream_t s);
// dQ = scale · accumulator (n_pad rows per head), rounded to bf16 [heads, N, d].
cudaError_t launch_dq_finish_bf16(const float* dqacc, __nv_bfloat16* dq, long long heads, int N, int n_pad, int d,
                                  float scale, cudaStream_t s);

// ---------------------------------------------------------------- fp32 SIMT path

cudaError_t launch_fwd_f32(const float* q, const float* k, const float* v, float* o, float* lse, int BH, int N,
                           int d, float scale, int causal, cudaStream_t s);
cudaError_t launch_bwd_prep_f32(const float* o, const float* dO, const float* lse, float* dvec, float* lse_copy,
                                long long rows, int d, cudaStream_t s);
cudaError_t launch_bwd_f32(const float* q, const float* k, const float* v, const float* dO, const float* lse,
                           const float* dvec, float* dq, float* dk, float* dv, int BH, int N, int d, float scale,
                           int causal, cudaStream_t s);

}  // namespace fa
