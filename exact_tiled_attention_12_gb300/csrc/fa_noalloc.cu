// fa_noalloc.cu — fa_bwd_noalloc: the backward pass without a caller-provided
// workspace, for callers that cannot allocate device memory.
//
// Some callers can't call cudaMalloc at the point where they need gradients: a
// host runtime that forbids allocation after start-up (fixed memory budgets,
// real-time or safety-certified loops), a plug-in whose host owns every device
// allocation, or a process whose allocator state must not change between two
// checkpoints.  fa_bwd needs a scratch workspace (D, the base-2 LSE and the
// float32 dQ accumulator); this entry point takes that scratch from a
// fixed-size array compiled into the library instead.
//
// The array is a file-scope __device__ variable, so every GPU that loads
// libfa.so holds FA_NOALLOC_SCRATCH_BYTES of device memory for it until the
// process exits.  Host code cannot use the array's name as a device address
// (on the host it names a shadow object), so the first call on each device
// asks the runtime for the device address with cudaGetSymbolAddress, with that
// device current, and caches it together with the id of the context it was
// looked up in (after cudaDeviceReset the array is looked up again).  That
// first call should therefore come before any stream capture starts.  No call
// here allocates memory.
#include "fa.h"
#include "fa_kernels.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch array in the current context.
void* lookup_scratch() {
  void* p = nullptr;
  return cudaGetSymbolAddress(&p, g_noalloc_scratch) == cudaSuccess ? p : nullptr;
}

fa::SymbolCache g_scratch_cache;

}  // namespace

extern "C" fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dO,
                                    const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                                    float scale, int causal, fa_dtype dtype, fa_stream_t stream) {
  const size_t need = fa_bwd_workspace_size(B, H, N, d, dtype);
  if (need > (size_t)FA_NOALLOC_SCRATCH_BYTES) return FA_ERR_WORKSPACE;   // problem larger than the built-in scratch
  if (need == 0)   // empty or invalid: fa_bwd returns the same status it would with any workspace
    return fa_bwd(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d, scale, causal, dtype, nullptr, 0, stream);
  void* scratch = fa::cached_symbol_address(g_scratch_cache, lookup_scratch);
  if (scratch == nullptr) return FA_ERR_CUDA;
  // fa_bwd's pre-pass overwrites D and the LSE copy and zeroes the dQ
  // accumulator, so whatever an earlier call left in the array is harmless.
  return fa_bwd(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d, scale, causal, dtype, scratch,
                (size_t)FA_NOALLOC_SCRATCH_BYTES, stream);
}
