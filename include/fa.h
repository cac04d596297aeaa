/*
 * fa.h — C ABI of the exact tiled attention library (libfa.so) for GB300 (sm_103a).
 *
 * What is computed (pages cited by title and section):
 *   Forward  — "Flash Attention" tutorial, 1.FlashAttention 整体结构 一 and
 *              2.Online Softmax §4.2: O = softmax(scale · Q Kᵀ) V computed one
 *              K/V tile at a time with the online (m, ℓ) rescaling of §3.1 and
 *              §4.1, normalised once at the end; the N×N score matrix never
 *              reaches global memory.  The per-row statistic is the one of
 *              3.Recomputation 三: LSE_i = m_i + ln ℓ_i.
 *   Backward — same tutorial, 3.Recomputation 四 and 4.附录A
 *              "反向传播的公式推导" 五-六: only O and LSE are kept; each tile of
 *              P is rebuilt as exp(S - LSE); D = rowsum(dO ⊙ O);
 *              dV = Pᵀ dO, dP = dO Vᵀ, dS = P ⊙ (dP - D), dQ = scale · dS K,
 *              dK = scale · dSᵀ Q (the factor scale = 1/sqrt(d_k) on dQ and dK
 *              as on the coreui.cn page "FlashAttention 反向传播").
 *
 * Conventions shared by every entry point:
 *   Layout      Q, K, V, O, dO, dQ, dK, dV are dense row-major [B, H, N, d]
 *               (d innermost, no padding).  LSE is dense [B, H, N] float32,
 *               the natural-log log-sum-exp of row i of scale · Q Kᵀ over the
 *               visible keys.  All pointers are DEVICE pointers.
 *   dtype       FA_DTYPE_BF16: every [B,H,N,d] tensor is bfloat16; arithmetic
 *               is fp32 accumulation on the tensor cores, P and dS are rounded
 *               to bf16 before their products.  Supported: d ∈ {64, 96, 128,
 *               256}, any N ≥ 1 (tiles of 128 rows; a ragged last tile reads
 *               zero rows past N and masks those keys), base pointers 16-byte
 *               aligned.
 *               FA_DTYPE_FP16: the same with IEEE half precision (P and dS
 *               rounded to fp16; outputs that pass ±65504 become ±inf).
 *               FA_DTYPE_FP32: every tensor is float32 and computed with
 *               fp32 arithmetic (no tensor cores); any N ≥ 1, 1 ≤ d ≤ 128.
 *   causal      0: every key visible.  1: key j visible to query i iff j ≤ i
 *               (square, top-left aligned; no row is ever empty).  The _kv
 *               entry points take Nq queries over Nk keys; there the queries
 *               are the last Nq positions of the sequence ("Flash Attention"
 *               tutorial, 2.Online Softmax §七 item 3: later tokens extend a
 *               cached prefix), so query i sees keys j ≤ i + Nk − Nq, which
 *               needs Nq ≤ Nk (FA_ERR_UNSUPPORTED otherwise).
 *   scale       finite and > 0; callers usually pass 1/sqrt(d).
 *   Limits      (FA_ERR_UNSUPPORTED past them; the grids' second dimension)
 *               at most 65,535 heads (B·H) and 65,535 tiles of 128 keys per
 *               head (8,388,480 keys); the d = 256 backward under the causal
 *               mask at most 65,535 tiles of 64 keys (4,194,240 keys); fewer
 *               than 2^31 query rows and 2^31 key rows in all (counted in
 *               whole 128-row tiles per head for the 16-bit types).
 *   Empty       B, H or N equal to 0 is a valid empty problem: FA_OK, nothing
 *               launched, pointers may be NULL.
 *   Ownership   the caller owns every buffer.  The library allocates no device
 *               or host memory.
 *   Streams     every call only enqueues work on `stream` (NULL = legacy
 *               default stream) and returns without synchronising.  Outputs
 *               are fully overwritten.  Calls on different streams must not
 *               share output or workspace buffers.
 *   Errors      argument checks happen on the host before anything is
 *               enqueued and return FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED,
 *               FA_ERR_MISALIGNED or FA_ERR_WORKSPACE with no side effects.
 *               A launch failure returns FA_ERR_CUDA.  Kernels never trap: a
 *               pipeline wait that runs past its time limit records a fault
 *               word and the kernel exits; fa_sync_status() reports it as
 *               FA_ERR_TIMEOUT.  No exception crosses the ABI; nothing is
 *               printed.
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque CUDA stream handle; identical to cudaStream_t / CUstream. */
typedef struct CUstream_st* fa_stream_t;

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,  /* null pointer, negative size, bad scale/causal/dtype */
  FA_ERR_UNSUPPORTED = 2,  /* valid but not implemented (bf16/fp16 d∉{64,96,128,256}, fp32 d>128, sizes past the grid limits) */
  FA_ERR_MISALIGNED = 3,   /* bf16/fp16 base pointer not 16-byte aligned */
  FA_ERR_WORKSPACE = 4,    /* workspace NULL, misaligned (256 B) or too small */
  FA_ERR_CUDA = 5,         /* a CUDA runtime/driver call or launch failed */
  FA_ERR_TIMEOUT = 6,      /* a kernel abandoned a pipeline wait (see fa_sync_status) */
  FA_ERR_BOUNDS = 7        /* debug build only: a device-side bounds or alignment check failed */
} fa_status;

typedef enum { FA_DTYPE_BF16 = 0, FA_DTYPE_FP32 = 1, FA_DTYPE_FP16 = 2 } fa_dtype;

/* Human-readable name of a status code (static string, never NULL). */
const char* fa_status_string(fa_status s);

/* Library ABI version (major*100 + minor): 110 adds the _kv entry points,
 * fa_merge and FA_DTYPE_FP16. */
int fa_version(void);

/*
 * Bytes of optional device workspace that lets fa_fwd balance its last wave
 * of work across the GPU (0 when it would not: causal masks, FA_DTYPE_FP32,
 * or no partial last wave).  Depends on the current device's SM count (one
 * CUDA attribute query, cached); returns 0 for invalid arguments or when no
 * device is available.
 */
size_t fa_fwd_workspace_size(int B, int H, int N, int d, int causal, fa_dtype dtype);

/*
 * Forward.  Reads q, k, v; writes o [B,H,N,d] and lse [B,H,N] (float32).
 * Cited: "Flash Attention" tutorial, 2.Online Softmax §4.2 (one pass over
 * K/V tiles, deferred normalisation) and 3.Recomputation 三 (the saved L).
 * `workspace` is optional: NULL runs every 256-query unit of work in one CTA.
 * With at least fa_fwd_workspace_size() bytes (256-byte aligned) the units of
 * the last, partial wave are split over K/V ranges whose partial results are
 * merged on the device with the log-sum-exp form of the two-block merge
 * (2.Online Softmax §3.1, §七); results differ from the unsplit run only by
 * floating-point rounding.  A non-NULL workspace that is misaligned or too
 * small returns FA_ERR_WORKSPACE.
 */
fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                 int B, int H, int N, int d, float scale, int causal,
                 fa_dtype dtype, void* workspace, size_t workspace_bytes,
                 fa_stream_t stream);

/*
 * Nq queries over Nk keys: Q and O are [B,H,Nq,d], K and V [B,H,Nk,d], LSE
 * [B,H,Nq].  Otherwise as fa_fwd_workspace_size / fa_fwd (which are these with
 * Nq = Nk = N).  Nq = 0 is an empty problem; Nk = 0 with Nq > 0 (queries with
 * no key) is FA_ERR_INVALID_ARG.  With causal = 1 the queries are the last Nq
 * positions (see "causal" above): e.g. a decode step is Nq = 1 over the Nk
 * cached keys plus itself, and prefix caching runs the new tokens' queries
 * over all keys.
 * Nq = 1 with a 16-bit dtype (a decoding step; the causal flag changes
 * nothing there, the one query sees every key) runs a streaming kernel that
 * reads K and V once with 16-byte loads on the CUDA cores: the step is bound
 * by HBM bandwidth.  With the workspace each head's keys are cut into ranges
 * (about four CTAs per SM, ≥ 256 keys each) merged as above; with NULL one
 * CTA per head does all of its keys.
 */
size_t fa_fwd_kv_workspace_size(int B, int H, int Nq, int Nk, int d, int causal, fa_dtype dtype);
fa_status fa_fwd_kv(const void* q, const void* k, const void* v, void* o, float* lse,
                    int B, int H, int Nq, int Nk, int d, float scale, int causal,
                    fa_dtype dtype, void* workspace, size_t workspace_bytes,
                    fa_stream_t stream);

/*
 * Bytes of device workspace fa_bwd needs for this problem (0 for an empty
 * one).  BF16: D and the base-2 LSE (4·B·H·Np bytes each) plus a float32 dQ
 * accumulator (4·B·H·Np·d bytes; none at d = 256), Np = 128·⌈N/128⌉ (whole
 * tiles per head), each part padded to 256 bytes.  FP32: D and
 * a copy of LSE (4·B·H·N bytes each, padded to 256).
 * Pure host arithmetic; returns 0 for invalid arguments.
 */
size_t fa_bwd_workspace_size(int B, int H, int N, int d, fa_dtype dtype);

/*
 * Backward.  Reads q, k, v, o, dO and the forward's lse; writes dq, dk, dv
 * (same dtype and layout as q).  `workspace` is caller-owned device memory of
 * at least fa_bwd_workspace_size() bytes, 256-byte aligned; its contents on
 * entry do not matter and are clobbered.  The bf16 path accumulates dQ in
 * float32 with reductions whose order varies, so dQ is not bitwise
 * reproducible run to run; O, LSE, dK and dV are.  At d = 256 dQ comes from
 * its own pass over the keys (no reductions) and is reproducible too.
 * Cited: "Flash Attention" tutorial, 4.附录A "反向传播的公式推导" 六 (tiled
 * backward with the D precompute; here K/V tiles are the outer loop).
 * Equivalent to fa_bwd_prep + fa_bwd_tiles + fa_bwd_dq_finish on one stream.
 */
fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o,
                 const void* dO, const float* lse, void* dq, void* dk, void* dv,
                 int B, int H, int N, int d, float scale, int causal,
                 fa_dtype dtype, void* workspace, size_t workspace_bytes,
                 fa_stream_t stream);

/*
 * Backward for Nq queries over Nk keys (layouts as fa_fwd_kv; dq like q, dk
 * and dv like k).  The workspace depends on Nq only (the same formula as
 * fa_bwd_workspace_size with N = Nq).  Nq = 0 with Nk > 0 writes dk = dv = 0.
 */
size_t fa_bwd_kv_workspace_size(int B, int H, int Nq, int Nk, int d, fa_dtype dtype);
fa_status fa_bwd_kv(const void* q, const void* k, const void* v, const void* o,
                    const void* dO, const float* lse, void* dq, void* dk, void* dv,
                    int B, int H, int Nq, int Nk, int d, float scale, int causal,
                    fa_dtype dtype, void* workspace, size_t workspace_bytes,
                    fa_stream_t stream);

/* Most partial results one fa_merge call takes. */
#define FA_MERGE_MAX_PARTS 16

/*
 * Merge of partial results of the same queries over disjoint key sets
 * ("Flash Attention" tutorial, 2.Online Softmax §3.1/§4.1, the two-block
 * merge, in log-sum-exp form; §七 lists its uses: ring attention, streaming
 * inference / prefix caching).  For every row:
 *   LSE = ln Σ_k e^{LSE_k},   O = Σ_k e^{LSE_k − LSE} · O_k.
 * A part whose LSE_k is −∞ saw no key of that row and contributes nothing;
 * a row no part saw gets O = 0 and LSE = −∞.
 *   o_parts, lse_parts  HOST arrays of n_parts DEVICE pointers: part k's O
 *                       [B,H,N,d] in `dtype` and LSE [B,H,N] float32 (as
 *                       fa_fwd / fa_fwd_kv write them).  1 ≤ n_parts ≤
 *                       FA_MERGE_MAX_PARTS; the host arrays are read before
 *                       the call returns.
 *   o, lse              outputs, same layouts; may be the same buffers as
 *                       one of the parts (each row is read before it is
 *                       written), so a running state can be extended in place.
 *   d                   1 ≤ d ≤ 256 for either dtype.
 * Errors as the other entry points (null or misaligned pointers, sizes).
 */
fa_status fa_merge(const void* const* o_parts, const float* const* lse_parts, int n_parts,
                   void* o, float* lse, int B, int H, int N, int d, fa_dtype dtype,
                   fa_stream_t stream);

/*
 * The three stages of fa_bwd, exposed so each can be timed on its own.  They
 * must run in this order on one stream with the same workspace and sizes.
 *   fa_bwd_prep      — "反向传播的公式推导" 五 (预处理): D_i = Σ_k dO_ik O_ik in
 *                      float32 and a copy of LSE (bf16 stores −D and
 *                      −LSE·log2(e) for the tiled stage), dQ accumulator zeroed.
 *   fa_bwd_tiles     — the tiled loop of 六: recompute S and P per tile, then
 *                      dV += Pᵀ dO, dP = dO Vᵀ, dS = P ⊙ (dP - D), dK += dSᵀ Q
 *                      and dQ += dS K (into the accumulator); writes dk, dv.
 *   fa_bwd_dq_finish — dQ = scale · accumulator, rounded to the output dtype.
 * For FA_DTYPE_FP32, and for d = 256 (where fa_bwd_tiles runs a dK/dV kernel
 * over 64-key tiles and a dQ kernel over 128-query tiles), fa_bwd_tiles
 * writes dq directly and fa_bwd_dq_finish is a no-op.
 */
fa_status fa_bwd_prep(const void* o, const void* dO, const float* lse,
                      int B, int H, int N, int d, fa_dtype dtype,
                      void* workspace, size_t workspace_bytes, fa_stream_t stream);
fa_status fa_bwd_tiles(const void* q, const void* k, const void* v, const void* dO,
                       void* dq, void* dk, void* dv,
                       int B, int H, int N, int d, float scale, int causal,
                       fa_dtype dtype, void* workspace, size_t workspace_bytes,
                       fa_stream_t stream);
fa_status fa_bwd_dq_finish(void* dq, int B, int H, int N, int d, float scale,
                           fa_dtype dtype, void* workspace, size_t workspace_bytes,
                           fa_stream_t stream);

/*
 * Synchronises `stream`, then reports and clears the kernels' fault words on
 * the current device: FA_ERR_TIMEOUT if any kernel abandoned a pipeline wait
 * since the last call, FA_ERR_BOUNDS if (debug build) a device-side check
 * failed, FA_ERR_CUDA if the stream reports an error, else FA_OK.  The only
 * entry point that blocks the host.
 */
fa_status fa_sync_status(fa_stream_t stream);

/*
 * Self-test of the failure path (not part of the computation).  Enqueues one
 * small kernel whose pipeline wait can never complete, so the wait gives up
 * after its time limit (2 s), records the fault word and raises the CTA's
 * abort flag, and the CTA's other wait gives up on seeing it; the kernel then
 * exits normally — nothing faults, traps or hangs.  Returns FA_OK if the
 * launch succeeded; a following fa_sync_status() returns FA_ERR_TIMEOUT (and
 * clears the word), after which the device is fully usable.  This is the
 * path every tensor-core kernel takes when a wait runs out.
 */
fa_status fa_selftest_wait_timeout(fa_stream_t stream);

/*
 * Debug build.  The library also builds as libfa_debug.so (same symbols,
 * compiled with FA_DEBUG_CHECKS) whose tensor-core kernels check, before
 * each access, that every TMA tile load starts its innermost coordinate on a
 * 16-byte boundary inside the row and its rows inside the tensor, that every
 * shared-memory destination or MMA operand lies inside the kernel's dynamic
 * shared memory with its alignment, that every tensor-memory load, store and
 * MMA accumulator stays inside the 512 allocated columns, and that every bulk
 * copy is 16-byte aligned.  A failed check records its code in the fault
 * word, raises the CTA's abort flag and skips the access (a skipped load
 * still completes its bytes on the barrier), so the CTA unwinds through its
 * bounded waits: nothing traps, and fa_sync_status() returns FA_ERR_BOUNDS.
 * Results of a debug build are bit-identical to the release build's except
 * for dQ's float32 summation order.  (compute-sanitizer is not available
 * everywhere; this is the substitute.)
 *
 * fa_debug_checks_enabled() returns 1 in libfa_debug.so and 0 in libfa.so.
 */
int fa_debug_checks_enabled(void);

/*
 * Self-test of the debug build's device-side checks (not part of the
 * computation).  One thread evaluates FA_SELFTEST_BOUNDS_CASES checks on
 * fixed integer arguments — alternately valid and invalid: a TMA coordinate
 * off its 16-byte boundary, box rows past the tensor, tensor-memory columns
 * past the allocation, a misaligned shared-memory operand — and writes 1
 * (passed) or 0 (failed) for each into `results` (device memory, at least
 * FA_SELFTEST_BOUNDS_CASES ints).  The kernel performs no access with those
 * arguments: it only evaluates the checks.  The first failed check's code is
 * recorded, so a following fa_sync_status() returns FA_ERR_BOUNDS.  Returns
 * FA_ERR_UNSUPPORTED from the release library (checks compiled out) and
 * FA_ERR_INVALID_ARG for a NULL `results`.
 */
#define FA_SELFTEST_BOUNDS_CASES 8
fa_status fa_selftest_bounds_check(int* results, fa_stream_t stream);

/*
 * Size of the scratch array compiled into libfa.so for fa_bwd_noalloc:
 * 32 MiB, held on every GPU that loads the library until the process exits.
 */
#define FA_NOALLOC_SCRATCH_BYTES (32u << 20)

/*
 * Backward without a workspace argument.  The pages have no counterpart to
 * this entry point; it exists for callers that cannot allocate device memory
 * (for example a runtime that forbids allocation after start-up, or a plug-in
 * whose host owns every device allocation).  Same arguments, results and
 * errors as fa_bwd, except that the scratch comes from a fixed array inside
 * the library instead of the caller:
 *   - nothing is allocated, by this call or by anything it calls;
 *   - problems whose fa_bwd_workspace_size() exceeds FA_NOALLOC_SCRATCH_BYTES
 *     are rejected with FA_ERR_WORKSPACE before anything is enqueued (for
 *     bf16 that is 4·B·H·Np·(d + 2) bytes plus padding, e.g. B·H·Np up to
 *     about 64,000 rows at d = 128);
 *   - the first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current and caches it with the
 *     id of the current context (a call after cudaDeviceReset, in a new
 *     context, looks it up again); make that first call before any stream
 *     capture begins;
 *   - every call on a device shares the one array and it keeps the last
 *     call's contents (the pre-pass rewrites what must start at zero), so
 *     calls whose work can overlap on the GPU — on different streams, or from
 *     different host threads — race and must not be issued.
 */
fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                         const void* dO, const float* lse, void* dq, void* dk, void* dv,
                         int B, int H, int N, int d, float scale, int causal,
                         fa_dtype dtype, fa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
