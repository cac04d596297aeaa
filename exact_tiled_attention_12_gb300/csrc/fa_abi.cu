// fa_abi.cu — the extern "C" boundary of libfa.so (declared in include/fa.h).
//
// Host-side only: argument validation, TMA tensor-map encoding, workspace
// carving and kernel dispatch.  Every argument check runs before any CUDA call,
// so invalid calls return an error with no side effect (and need no GPU).
#include <cudaTypedefs.h>
#include <math.h>
#include <stdint.h>

#include <atomic>

#include "fa.h"
#include "fa_checks.h"
#include "fa_decode.h"
#include "fa_kernels.h"

namespace {

// One fault word per device; kernels record the first timed-out wait here.
__device__ unsigned int g_fault_word;

void* lookup_fault_word() {
  void* addr = nullptr;
  return cudaGetSymbolAddress(&addr, g_fault_word) == cudaSuccess ? addr : nullptr;
}

fa::SymbolCache g_fault_cache;

unsigned int* fault_word_for_current_device() {
  return static_cast<unsigned int*>(fa::cached_symbol_address(g_fault_cache, lookup_fault_word));
}

template <class PFN>
PFN driver_entry(const char* name, int version) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, version, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<PFN>(p);
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::atomic<PFN_cuTensorMapEncodeTiled_v12000> fn{nullptr};
  PFN_cuTensorMapEncodeTiled_v12000 f = fn.load(std::memory_order_acquire);
  if (f) return f;
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || p == nullptr)
    return nullptr;
  f = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  fn.store(f, std::memory_order_release);
  return f;
}

// Tensor map over a [B·H, N, d] bf16 (or fp16) tensor with boxes of 64 columns (128
// bytes) × box_rows rows and 128-byte swizzle.  rows_view (every sequence
// length of the call a multiple of 128): a 2-D map over the [B·H·N, d] row
// view (a tile never straddles two heads).  Otherwise a 3-D map whose rows
// past N read as zero, so the last tile of a head never picks up the next
// head's rows.  The kernels take the matching copy form from the same test.
bool encode_bf16_heads(CUtensorMap* m, const void* base, long long heads, long long N, int d, int box_rows,
                       bool rows_view, bool f16) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)(rows_view ? heads * N : N), (cuuint64_t)heads};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)N * (cuuint64_t)d * 2};
  cuuint32_t box[3] = {64u, (cuuint32_t)box_rows, 1u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = enc(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rows_view ? 2 : 3, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

inline size_t pad256(size_t x) { return (x + 255) & ~(size_t)255; }

bool valid_dtype(fa_dtype t) { return t == FA_DTYPE_BF16 || t == FA_DTYPE_FP32 || t == FA_DTYPE_FP16; }
// The 16-bit dtypes run on the tensor cores; float32 runs the SIMT kernels.
bool is16(fa_dtype t) { return t == FA_DTYPE_BF16 || t == FA_DTYPE_FP16; }

// ------------------------------------------------------------------ validation

// Nq queries over Nk keys per (batch, head).
struct Shape {
  long long B, H, Nq, Nk, d;
  long long heads() const { return B * H; }
  long long rows() const { return B * H * Nq; }            // query rows
  long long q_elems() const { return B * H * Nq * d; }
  long long k_elems() const { return B * H * Nk * d; }
  // bf16 per-row workspace arrays are padded to whole 128-row tiles per head
  long long nq_pad() const { return (Nq + 127) / 128 * 128; }
  long long nk_pad() const { return (Nk + 127) / 128 * 128; }
  long long rows_pad() const { return B * H * nq_pad(); }
  bool rows_view() const { return Nq % 128 == 0 && Nk % 128 == 0; }
  bool no_heads() const { return B == 0 || H == 0; }
  bool empty() const { return no_heads() || Nq == 0; }    // nothing to compute for any query
};

fa_status check_shape(int B, int H, int Nq, int Nk, int d, fa_dtype dtype, int causal, Shape* out) {
  if (B < 0 || H < 0 || Nq < 0 || Nk < 0 || d <= 0) return FA_ERR_INVALID_ARG;
  if (!valid_dtype(dtype)) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  Shape s{B, H, Nq, Nk, d};
  if (s.q_elems() > (1ll << 40) || s.k_elems() > (1ll << 40)) return FA_ERR_UNSUPPORTED;
  if (!s.no_heads() && Nq > 0 && Nk == 0) return FA_ERR_INVALID_ARG;     // queries with no key at all
  if (s.no_heads() || (Nq == 0 && Nk == 0)) {
    *out = s;
    return FA_OK;
  }
  // The causal mask aligns the queries with the last Nq keys; more queries
  // than keys would leave rows with no visible key.
  if (causal && Nq > Nk) return FA_ERR_UNSUPPORTED;
  if (s.heads() > 65535) return FA_ERR_UNSUPPORTED;
  if (is16(dtype)) {
    if (d != 64 && d != 96 && d != 128 && d != 256) return FA_ERR_UNSUPPORTED;
    if (s.rows_pad() >= (1ll << 31) || s.heads() * s.nk_pad() >= (1ll << 31) || s.nk_pad() / 128 > 65535)
      return FA_ERR_UNSUPPORTED;
  } else {
    if (d > 128) return FA_ERR_UNSUPPORTED;
    if (s.rows() >= (1ll << 31) || s.heads() * Nk >= (1ll << 31)) return FA_ERR_UNSUPPORTED;
  }
  *out = s;
  return FA_OK;
}

fa_status check_scale(float scale) {
  return (isfinite(scale) && scale > 0.f) ? FA_OK : FA_ERR_INVALID_ARG;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

fa_status check_ptrs(std::initializer_list<const void*> ptrs, fa_dtype dtype) {
  for (const void* p : ptrs)
    if (p == nullptr) return FA_ERR_INVALID_ARG;
  if (is16(dtype))
    for (const void* p : ptrs)
      if (!aligned16(p)) return FA_ERR_MISALIGNED;
  for (const void* p : ptrs)
    if ((reinterpret_cast<uintptr_t>(p) & 3u) != 0) return FA_ERR_MISALIGNED;
  return FA_OK;
}

size_t workspace_bytes_for(const Shape& s, fa_dtype dtype) {
  if (s.empty()) return 0;
  if (dtype == FA_DTYPE_FP32) return 2 * pad256((size_t)s.rows() * 4);
  const size_t rows = (size_t)s.rows_pad();
  // d = 256 writes dQ directly (no fp32 accumulator).
  return 2 * pad256(rows * 4) + (s.d == 256 ? 0 : pad256(rows * (size_t)s.d * 4));
}

// Workspace parts: D (float32 per query row), the forward's LSE per row (base
// 2 for bf16, natural-log copy for fp32), and for bf16 the float32 dQ
// accumulator.  The bf16 parts hold whole 128-row tiles per head.
struct Workspace {
  float* dvec;
  float* lse2;
  float* dqacc;
};

fa_status carve_workspace(const Shape& s, fa_dtype dtype, void* ws, size_t bytes, Workspace* w) {
  const size_t need = workspace_bytes_for(s, dtype);
  if (need == 0) return FA_OK;
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0 || bytes < need) return FA_ERR_WORKSPACE;
  char* p = static_cast<char*>(ws);
  const size_t rows = dtype == FA_DTYPE_FP32 ? (size_t)s.rows() : (size_t)s.rows_pad();
  w->dvec = reinterpret_cast<float*>(p);
  w->lse2 = reinterpret_cast<float*>(p + pad256(rows * 4));
  w->dqacc = (dtype == FA_DTYPE_FP32 || s.d == 256) ? nullptr : reinterpret_cast<float*>(p + 2 * pad256(rows * 4));
  return FA_OK;
}

inline fa_status from_cuda(cudaError_t e) { return e == cudaSuccess ? FA_OK : FA_ERR_CUDA; }

// SM count of the current device (0 if it cannot be queried), cached per device.
int sm_count_current_device() {
  static std::atomic<int> cache[fa::kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= fa::kMaxDevices) return 0;
  int n = cache[dev].load(std::memory_order_relaxed);
  if (n > 0) return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 0;
  cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

struct FwdPlan {
  int n_full, splits, part_rows;
  size_t opart_bytes;
};

// Workspace the forward's load balancing needs on the current device (0 when
// it does not split: fp32, or a long problem with no partial last wave worth
// splitting, or a long causal one).  One query (a decoding step) sees every
// key under the causal mask, so it runs as the unmasked problem, which may
// split its keys over several CTAs.  A problem with 2 to 128 queries per
// head and fewer units than SMs streams its K/V far more than it computes
// and would leave SMs idle: every unit is split over its K/V tiles so the
// grid fills whole waves (under the mask too, except at d = 256), and each
// part keeps one partial row per query.  (Measured on GB300: with as many
// units as SMs or more, the unsplit grid already keeps HBM busy and
// splitting every unit only adds start-up and merge work.)
int forward_causal(int causal, const Shape& s) { return causal && s.Nq > 1 ? 1 : 0; }

size_t fwd_workspace_bytes(const Shape& s, int causal, fa_dtype dtype, FwdPlan* plan) {
  causal = forward_causal(causal, s);
  if (s.empty() || !is16(dtype)) return 0;
  const int sms = sm_count_current_device();
  const bool short_q =
      s.Nq >= 2 && s.Nq <= 128 && fa::fwd_units((int)s.B, (int)s.H, (int)s.Nq, (int)s.d) < sms;
  if (causal && !(short_q && s.d != 256)) return 0;
  if (s.Nq == 1) {
    // A decoding step: the streaming kernel's key ranges per head.
    const int splits = fa::decode_splits((int)s.heads(), sm_count_current_device(), (int)s.Nk);
    if (splits <= 1) return 0;
    const size_t rows = (size_t)s.heads() * (size_t)splits;
    const size_t opart = pad256(rows * (size_t)s.d * 4);
    if (plan) *plan = FwdPlan{0, splits, 1, opart};
    return opart + pad256(rows * 4);
  }
  const int units = fa::fwd_units((int)s.B, (int)s.H, (int)s.Nq, (int)s.d);
  int n_full, splits, part_rows = fa::fwd_unit_rows((int)s.d);
  if (short_q) {
    // Every query row of a head sees (under the mask) keys up to Nk − 1, so
    // each unit's visible K/V tiles are all of them.
    n_full = 0;
    splits = fa::fwd_split_short(units, sms, (int)(s.nk_pad() / 128));
    part_rows = (int)s.Nq;
  } else {
    fa::fwd_split_plan(units, sms, (int)(s.nk_pad() / 128), &n_full, &splits);
  }
  if (splits <= 1 || n_full >= units) return 0;
  const size_t rows = (size_t)(units - n_full) * (size_t)splits * (size_t)part_rows;
  const size_t opart = pad256(rows * (size_t)s.d * 4);
  if (plan) *plan = FwdPlan{n_full, splits, part_rows, opart};
  return opart + pad256(rows * 4);
}

constexpr float kLog2e = 1.4426950408889634074f;

size_t elem_bytes(fa_dtype dtype) { return is16(dtype) ? 2 : 4; }

// ------------------------------------------------------------------ implementations (Nq queries, Nk keys)

fa_status fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq, int Nk,
                   int d, float scale, int causal, fa_dtype dtype, void* workspace, size_t workspace_bytes,
                   fa_stream_t stream) {
  Shape s;
  fa_status st = check_shape(B, H, Nq, Nk, d, dtype, causal, &s);
  if (st != FA_OK) return st;
  if ((st = check_scale(scale)) != FA_OK) return st;
  if (s.empty()) return FA_OK;
  causal = forward_causal(causal, s);
  if ((st = check_ptrs({q, k, v, o, lse}, dtype)) != FA_OK) return st;
  if (workspace != nullptr && (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return FA_ERR_WORKSPACE;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  unsigned int* fault = fault_word_for_current_device();
  if (!fault) return FA_ERR_CUDA;
  if (dtype == FA_DTYPE_FP32)
    return from_cuda(fa::launch_fwd_f32(static_cast<const float*>(q), static_cast<const float*>(k),
                                        static_cast<const float*>(v), static_cast<float*>(o), lse, (int)s.heads(), Nq,
                                        Nk, d, scale, causal, cs));
  const bool f16 = dtype == FA_DTYPE_FP16;
  if (Nq == 1) {
    // A decoding step (the causal mask was dropped above: one query sees
    // every key): streamed on the CUDA cores, keys split over CTAs when a
    // workspace is given.
    fa::DecodeArgs da{q, k, v, o, lse, (int)s.heads(), Nk, d, f16 ? 1 : 0, scale * kLog2e, 1, nullptr, nullptr};
    FwdPlan plan;
    const size_t need = fwd_workspace_bytes(s, causal, dtype, &plan);
    if (need > 0 && workspace != nullptr) {
      if (workspace_bytes < need) return FA_ERR_WORKSPACE;
      da.splits = plan.splits;
      da.opart = static_cast<float*>(workspace);
      da.lpart = reinterpret_cast<float*>(static_cast<char*>(workspace) + plan.opart_bytes);
    }
    return from_cuda(fa::launch_fwd_decode(da, cs));
  }
  fa::FwdArgs a;
  const long long heads = s.heads();
  const bool rv = s.rows_view();
  if (!encode_bf16_heads(&a.tm_q, q, heads, Nq, d, 128, rv, f16) ||
      !encode_bf16_heads(&a.tm_k, k, heads, Nk, d, 128, rv, f16) ||
      !encode_bf16_heads(&a.tm_v, v, heads, Nk, d, 128, rv, f16))
    return FA_ERR_CUDA;
  a.o = o;
  a.f16 = f16 ? 1 : 0;
  a.lse = lse;
  a.B = B;
  a.H = H;
  a.Nq = Nq;
  a.Nk = Nk;
  a.d = d;
  a.scale_log2 = scale * kLog2e;
  a.causal = causal;
  a.fault = fault;
  // Load balancing needs the workspace; without one (NULL) every unit runs whole.
  FwdPlan plan;
  const size_t need = fwd_workspace_bytes(s, causal, dtype, &plan);
  a.n_full = fa::fwd_units(B, H, Nq, d);
  a.splits = 1;
  a.part_rows = fa::fwd_unit_rows(d);
  a.opart = nullptr;
  a.lpart = nullptr;
  if (need > 0 && workspace != nullptr) {
    if (workspace_bytes < need) return FA_ERR_WORKSPACE;
    a.n_full = plan.n_full;
    a.splits = plan.splits;
    a.part_rows = plan.part_rows;
    a.opart = static_cast<float*>(workspace);
    a.lpart = reinterpret_cast<float*>(static_cast<char*>(workspace) + plan.opart_bytes);
  }
  // Short K/V ranges without the mask and with more units than SMs: one
  // persistent CTA per SM, so units' start-up and drain overlap.
  a.persist_ctas = 0;
  const int sms = sm_count_current_device();
  if (d != 256 && !causal && a.splits <= 1 && s.nk_pad() / 128 <= fa::kFwdPersistMaxTiles && sms > 0 &&
      fa::fwd_units(B, H, Nq, d) > sms)
    a.persist_ctas = sms;
  return from_cuda(fa::launch_fwd_bf16(a, cs));
}

fa_status prep_impl(const void* o, const void* dO, const float* lse, int B, int H, int Nq, int Nk, int d,
                    fa_dtype dtype, void* workspace, size_t workspace_bytes, fa_stream_t stream) {
  Shape s;
  fa_status st = check_shape(B, H, Nq, Nk, d, dtype, 0, &s);
  if (st != FA_OK) return st;
  if (s.empty()) return FA_OK;
  if ((st = check_ptrs({o, dO, lse}, dtype)) != FA_OK) return st;
  Workspace w;
  if ((st = carve_workspace(s, dtype, workspace, workspace_bytes, &w)) != FA_OK) return st;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (dtype == FA_DTYPE_FP32)
    return from_cuda(fa::launch_bwd_prep_f32(static_cast<const float*>(o), static_cast<const float*>(dO), lse, w.dvec,
                                             w.lse2, s.rows(), d, cs));
  return from_cuda(fa::launch_bwd_prep_bf16(o, dO, lse, w.dvec, w.lse2, w.dqacc, s.heads(), Nq, (int)s.nq_pad(), d,
                                            dtype == FA_DTYPE_FP16 ? 1 : 0, cs));
}

// The d = 256 backward tiles the keys by 64 and, under the causal mask, puts
// those tiles in the grid's second dimension (at most 65,535): past that it
// cannot launch, so such shapes are refused before any work is queued.
fa_status check_bwd_grid(const Shape& s, int causal, fa_dtype dtype) {
  if (is16(dtype) && s.d == 256 && causal && (s.Nk + 63) / 64 > 65535) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

fa_status tiles_impl(const void* q, const void* k, const void* v, const void* dO, void* dq, void* dk, void* dv, int B,
                     int H, int Nq, int Nk, int d, float scale, int causal, fa_dtype dtype, void* workspace,
                     size_t workspace_bytes, fa_stream_t stream) {
  Shape s;
  fa_status st = check_shape(B, H, Nq, Nk, d, dtype, causal, &s);
  if (st != FA_OK) return st;
  if ((st = check_bwd_grid(s, causal, dtype)) != FA_OK) return st;
  if ((st = check_scale(scale)) != FA_OK) return st;
  if (s.empty()) return FA_OK;
  if ((st = check_ptrs({q, k, v, dO, dk, dv}, dtype)) != FA_OK) return st;
  if ((dtype == FA_DTYPE_FP32 || d == 256) && (st = check_ptrs({dq}, dtype)) != FA_OK) return st;
  Workspace w;
  if ((st = carve_workspace(s, dtype, workspace, workspace_bytes, &w)) != FA_OK) return st;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (dtype == FA_DTYPE_FP32)
    return from_cuda(fa::launch_bwd_f32(static_cast<const float*>(q), static_cast<const float*>(k),
                                        static_cast<const float*>(v), static_cast<const float*>(dO), w.lse2, w.dvec,
                                        static_cast<float*>(dq), static_cast<float*>(dk), static_cast<float*>(dv),
                                        (int)s.heads(), Nq, Nk, d, scale, causal, cs));
  unsigned int* fault = fault_word_for_current_device();
  if (!fault) return FA_ERR_CUDA;
  fa::BwdArgs a;
  const int bm = fa::bwd_bf16_block_m(d);
  const int bn = fa::bwd_kv_box_rows(d);
  const long long heads = s.heads();
  const bool rv = s.rows_view();
  const bool f16 = dtype == FA_DTYPE_FP16;
  if (!encode_bf16_heads(&a.tm_q, q, heads, Nq, d, bm, rv, f16) ||
      !encode_bf16_heads(&a.tm_k, k, heads, Nk, d, bn, rv, f16) ||
      !encode_bf16_heads(&a.tm_v, v, heads, Nk, d, bn, rv, f16) ||
      !encode_bf16_heads(&a.tm_do, dO, heads, Nq, d, bm, rv, f16))
    return FA_ERR_CUDA;
  a.f16 = f16 ? 1 : 0;
  a.lse2 = w.lse2;
  a.dvec = w.dvec;
  a.dqacc = w.dqacc;
  a.dq = d == 256 ? dq : nullptr;
  a.dk = dk;
  a.dv = dv;
  a.B = B;
  a.H = H;
  a.Nq = Nq;
  a.Nk = Nk;
  a.d = d;
  a.scale_log2 = scale * kLog2e;
  a.scale = scale;
  a.causal = causal;
  a.fault = fault;
  // d = 64 without the mask, few query tiles per head and more K/V tiles than
  // SMs: one persistent CTA per SM, so K/V tiles' start-up and drain overlap.
  a.persist_ctas = 0;
  const int sms = sm_count_current_device();
  if (d == 64 && !causal && sms > 0 && s.nq_pad() / 128 <= fa::kBwdPersistMaxTiles &&
      heads * (s.nk_pad() / 128) > sms)
    a.persist_ctas = sms;
  return from_cuda(fa::launch_bwd_bf16(a, cs));
}

fa_status finish_impl(void* dq, int B, int H, int Nq, int Nk, int d, float scale, fa_dtype dtype, void* workspace,
                      size_t workspace_bytes, fa_stream_t stream) {
  Shape s;
  fa_status st = check_shape(B, H, Nq, Nk, d, dtype, 0, &s);
  if (st != FA_OK) return st;
  if ((st = check_scale(scale)) != FA_OK) return st;
  // fp32 and d = 256 write dQ in the tiled pass.
  if (s.empty() || dtype == FA_DTYPE_FP32 || d == 256) return FA_OK;
  if ((st = check_ptrs({dq}, dtype)) != FA_OK) return st;
  Workspace w;
  if ((st = carve_workspace(s, dtype, workspace, workspace_bytes, &w)) != FA_OK) return st;
  return from_cuda(fa::launch_dq_finish_bf16(w.dqacc, dq, s.heads(), Nq, (int)s.nq_pad(), d, scale,
                                             dtype == FA_DTYPE_FP16 ? 1 : 0, reinterpret_cast<cudaStream_t>(stream)));
}

fa_status bwd_impl(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                   void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int d, float scale, int causal,
                   fa_dtype dtype, void* workspace, size_t workspace_bytes, fa_stream_t stream) {
  Shape s;
  fa_status st = check_shape(B, H, Nq, Nk, d, dtype, causal, &s);
  if (st != FA_OK) return st;
  if ((st = check_bwd_grid(s, causal, dtype)) != FA_OK) return st;
  if ((st = check_scale(scale)) != FA_OK) return st;
  if (s.no_heads() || (Nq == 0 && Nk == 0)) return FA_OK;
  if (Nq == 0) {
    // No query sees the keys: their gradients are zero.
    if ((st = check_ptrs({dk, dv}, dtype)) != FA_OK) return st;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    const size_t bytes = (size_t)s.k_elems() * elem_bytes(dtype);
    if (cudaMemsetAsync(dk, 0, bytes, cs) != cudaSuccess || cudaMemsetAsync(dv, 0, bytes, cs) != cudaSuccess)
      return FA_ERR_CUDA;
    return FA_OK;
  }
  if ((st = check_ptrs({q, k, v, o, dO, lse, dq, dk, dv}, dtype)) != FA_OK) return st;
  Workspace w;
  if ((st = carve_workspace(s, dtype, workspace, workspace_bytes, &w)) != FA_OK) return st;
  if ((st = prep_impl(o, dO, lse, B, H, Nq, Nk, d, dtype, workspace, workspace_bytes, stream)) != FA_OK) return st;
  if ((st = tiles_impl(q, k, v, dO, dq, dk, dv, B, H, Nq, Nk, d, scale, causal, dtype, workspace, workspace_bytes,
                       stream)) != FA_OK)
    return st;
  return finish_impl(dq, B, H, Nq, Nk, d, scale, dtype, workspace, workspace_bytes, stream);
}

}  // namespace

namespace fa {

unsigned long long current_context_id() {
  static const auto get_current = driver_entry<PFN_cuCtxGetCurrent_v4000>("cuCtxGetCurrent", 4000);
  static const auto get_id = driver_entry<PFN_cuCtxGetId_v12000>("cuCtxGetId", 12000);
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

void* cached_symbol_address(SymbolCache& cache, void* (*lookup)()) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(cache.mu);
  const unsigned long long id = current_context_id();
  if (id != 0 && cache.ctx[dev] == id && cache.ptr[dev] != nullptr) return cache.ptr[dev];
  // The lookup makes the device's primary context current if none was yet.
  void* p = lookup();
  if (p == nullptr) {
    cudaGetLastError();   // leave no stale error for the next launch to report as its own
    return nullptr;
  }
  cache.ctx[dev] = current_context_id();
  cache.ptr[dev] = p;
  return p;
}

}  // namespace fa

extern "C" {

const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG: null pointer, negative size or bad scale/causal/dtype";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED: shape or dtype not implemented";
    case FA_ERR_MISALIGNED: return "FA_ERR_MISALIGNED: pointer not aligned (bf16 needs 16 bytes)";
    case FA_ERR_WORKSPACE: return "FA_ERR_WORKSPACE: workspace missing, misaligned (256 B) or too small";
    case FA_ERR_CUDA: return "FA_ERR_CUDA: a CUDA call or kernel launch failed";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT: a kernel abandoned a pipeline wait";
    case FA_ERR_BOUNDS: return "FA_ERR_BOUNDS: a device-side bounds or alignment check failed (debug build)";
  }
  return "unknown fa_status";
}

int fa_version(void) { return 110; }

size_t fa_fwd_kv_workspace_size(int B, int H, int Nq, int Nk, int d, int causal, fa_dtype dtype) {
  Shape s;
  if (check_shape(B, H, Nq, Nk, d, dtype, causal, &s) != FA_OK) return 0;
  return fwd_workspace_bytes(s, causal, dtype, nullptr);
}

size_t fa_fwd_workspace_size(int B, int H, int N, int d, int causal, fa_dtype dtype) {
  return fa_fwd_kv_workspace_size(B, H, N, N, d, causal, dtype);
}

fa_status fa_fwd_kv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq, int Nk,
                    int d, float scale, int causal, fa_dtype dtype, void* workspace, size_t workspace_bytes,
                    fa_stream_t stream) {
  return fwd_impl(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, dtype, workspace, workspace_bytes, stream);
}

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                 float scale, int causal, fa_dtype dtype, void* workspace, size_t workspace_bytes,
                 fa_stream_t stream) {
  return fwd_impl(q, k, v, o, lse, B, H, N, N, d, scale, causal, dtype, workspace, workspace_bytes, stream);
}

size_t fa_bwd_kv_workspace_size(int B, int H, int Nq, int Nk, int d, fa_dtype dtype) {
  Shape s;
  if (check_shape(B, H, Nq, Nk, d, dtype, 0, &s) != FA_OK) return 0;
  return workspace_bytes_for(s, dtype);
}

size_t fa_bwd_workspace_size(int B, int H, int N, int d, fa_dtype dtype) {
  return fa_bwd_kv_workspace_size(B, H, N, N, d, dtype);
}

fa_status fa_bwd_prep(const void* o, const void* dO, const float* lse, int B, int H, int N, int d, fa_dtype dtype,
                      void* workspace, size_t workspace_bytes, fa_stream_t stream) {
  return prep_impl(o, dO, lse, B, H, N, N, d, dtype, workspace, workspace_bytes, stream);
}

fa_status fa_bwd_tiles(const void* q, const void* k, const void* v, const void* dO, void* dq, void* dk, void* dv,
                       int B, int H, int N, int d, float scale, int causal, fa_dtype dtype, void* workspace,
                       size_t workspace_bytes, fa_stream_t stream) {
  return tiles_impl(q, k, v, dO, dq, dk, dv, B, H, N, N, d, scale, causal, dtype, workspace, workspace_bytes, stream);
}

fa_status fa_bwd_dq_finish(void* dq, int B, int H, int N, int d, float scale, fa_dtype dtype, void* workspace,
                           size_t workspace_bytes, fa_stream_t stream) {
  return finish_impl(dq, B, H, N, N, d, scale, dtype, workspace, workspace_bytes, stream);
}

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                 void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale, int causal, fa_dtype dtype,
                 void* workspace, size_t workspace_bytes, fa_stream_t stream) {
  return bwd_impl(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, N, d, scale, causal, dtype, workspace, workspace_bytes,
                  stream);
}

fa_status fa_bwd_kv(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                    void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int d, float scale, int causal,
                    fa_dtype dtype, void* workspace, size_t workspace_bytes, fa_stream_t stream) {
  return bwd_impl(q, k, v, o, dO, lse, dq, dk, dv, B, H, Nq, Nk, d, scale, causal, dtype, workspace, workspace_bytes,
                  stream);
}

static_assert(FA_MERGE_MAX_PARTS == fa::kMaxMergeParts, "merge part limit differs between fa.h and the kernel");

fa_status fa_merge(const void* const* o_parts, const float* const* lse_parts, int n_parts, void* o, float* lse,
                   int B, int H, int N, int d, fa_dtype dtype, fa_stream_t stream) {
  if (B < 0 || H < 0 || N < 0 || d <= 0) return FA_ERR_INVALID_ARG;
  if (!valid_dtype(dtype)) return FA_ERR_INVALID_ARG;
  if (n_parts < 1 || n_parts > FA_MERGE_MAX_PARTS) return FA_ERR_INVALID_ARG;
  if (d > 256) return FA_ERR_UNSUPPORTED;
  const long long rows = (long long)B * H * N;
  if (rows == 0) return FA_OK;
  if (rows * d > (1ll << 40) || (rows + 7) / 8 >= (1ll << 31)) return FA_ERR_UNSUPPORTED;
  if (o_parts == nullptr || lse_parts == nullptr) return FA_ERR_INVALID_ARG;
  fa_status st;
  if ((st = check_ptrs({o, lse}, dtype)) != FA_OK) return st;
  fa::MergeArgs a;
  for (int i = 0; i < n_parts; ++i) {
    if ((st = check_ptrs({o_parts[i], lse_parts[i]}, dtype)) != FA_OK) return st;
    a.o_parts[i] = o_parts[i];
    a.lse_parts[i] = lse_parts[i];
  }
  for (int i = n_parts; i < fa::kMaxMergeParts; ++i) {
    a.o_parts[i] = nullptr;
    a.lse_parts[i] = nullptr;
  }
  a.n_parts = n_parts;
  a.o = o;
  a.lse = lse;
  a.rows = rows;
  a.d = d;
  a.elem = dtype == FA_DTYPE_BF16 ? 1 : dtype == FA_DTYPE_FP16 ? 2 : 0;
  return from_cuda(fa::launch_merge(a, reinterpret_cast<cudaStream_t>(stream)));
}

fa_status fa_selftest_wait_timeout(fa_stream_t stream) {
  unsigned int* fault = fault_word_for_current_device();
  if (!fault) return FA_ERR_CUDA;
  return from_cuda(fa::launch_wait_timeout_selftest(fault, reinterpret_cast<cudaStream_t>(stream)));
}

fa_status fa_sync_status(fa_stream_t stream) {
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return FA_ERR_CUDA;
  unsigned int word = 0;
  if (cudaMemcpyFromSymbol(&word, g_fault_word, sizeof(word)) != cudaSuccess) return FA_ERR_CUDA;
  if (word != 0) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(g_fault_word, &zero, sizeof(zero)) != cudaSuccess) return FA_ERR_CUDA;
    return fa::is_check_code(word) ? FA_ERR_BOUNDS : FA_ERR_TIMEOUT;
  }
  return FA_OK;
}

int fa_debug_checks_enabled(void) { return fa::kDebugChecks ? 1 : 0; }

fa_status fa_selftest_bounds_check(int* results, fa_stream_t stream) {
  if (!fa::kDebugChecks) return FA_ERR_UNSUPPORTED;
  if (results == nullptr) return FA_ERR_INVALID_ARG;
  unsigned int* fault = fault_word_for_current_device();
  if (!fault) return FA_ERR_CUDA;
  return from_cuda(fa::launch_bounds_check_selftest(fault, results, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
