// fa_decode.h — the decoding-step kernel (fa_decode.cu): one query row per
// (batch, head) over Nk keys, streamed on the CUDA cores.  Internal to libfa.so.
#pragma once

#include <cuda_runtime.h>

namespace fa {

// q [BH, d], k and v [BH, Nk, d] in the 16-bit type (bf16, or fp16 when
// f16 = 1); o [BH, d], lse [BH] (natural log of the scaled scores).  With
// splits > 1 each head's keys are cut into `splits` equal ranges whose fp32
// partials (opart [BH·splits, d], lpart [BH·splits]) are merged afterwards.
struct DecodeArgs {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  int BH, Nk, d, f16;
  float scale_log2;
  int splits;
  float* opart;
  float* lpart;
};

// Key ranges per head for `heads` heads on `num_sms` SMs (1 = no split).
int decode_splits(int heads, int num_sms, int Nk);
// Launches the step and, when split, the merge of the partials.
cudaError_t launch_fwd_decode(const DecodeArgs& a, cudaStream_t s);

}  // namespace fa
