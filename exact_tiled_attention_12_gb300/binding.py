"""ctypes binding for libfa.so — argument marshalling only.

Every step of the computation runs in the library's CUDA kernels; this module
allocates outputs with torch (the library allocates nothing), passes device
pointers and the current CUDA stream, and turns status codes into exceptions.
If libfa.so is missing the calls raise: there is no fallback.
"""

from __future__ import annotations

import contextlib
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = None

FA_DTYPE_BF16 = 0
FA_DTYPE_FP32 = 1
FA_DTYPE_FP16 = 2
_CODES = {torch.bfloat16: FA_DTYPE_BF16, torch.float32: FA_DTYPE_FP32, torch.float16: FA_DTYPE_FP16}
_STATUS = {
    0: "FA_OK", 1: "FA_ERR_INVALID_ARG", 2: "FA_ERR_UNSUPPORTED", 3: "FA_ERR_MISALIGNED",
    4: "FA_ERR_WORKSPACE", 5: "FA_ERR_CUDA", 6: "FA_ERR_TIMEOUT", 7: "FA_ERR_BOUNDS",
}
# Every function include/fa.h declares, with (restype, argtypes).
_P, _I, _F, _Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
SIGNATURES = {
    "fa_status_string": (ctypes.c_char_p, [_I]),
    "fa_version": (_I, []),
    "fa_fwd_workspace_size": (_Z, [_I, _I, _I, _I, _I, _I]),
    "fa_fwd": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _I, _P, _Z, _P]),
    "fa_bwd_workspace_size": (_Z, [_I, _I, _I, _I, _I]),
    "fa_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _I, _P, _Z, _P]),
    "fa_bwd_prep": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _P, _Z, _P]),
    "fa_bwd_tiles": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _I, _P, _Z, _P]),
    "fa_bwd_dq_finish": (_I, [_P, _I, _I, _I, _I, _F, _I, _P, _Z, _P]),
    "fa_sync_status": (_I, [_P]),
    "fa_bwd_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _F, _I, _I, _P]),
    "fa_fwd_kv_workspace_size": (_Z, [_I, _I, _I, _I, _I, _I, _I]),
    "fa_fwd_kv": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _I, _P, _Z, _P]),
    "fa_bwd_kv_workspace_size": (_Z, [_I, _I, _I, _I, _I, _I]),
    "fa_bwd_kv": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _I, _P, _Z, _P]),
    "fa_merge": (_I, [_P, _P, _I, _P, _P, _I, _I, _I, _I, _I, _P]),
    "fa_selftest_wait_timeout": (_I, [_P]),
    "fa_debug_checks_enabled": (_I, []),
    "fa_selftest_bounds_check": (_I, [_P, _P]),
}
FA_SELFTEST_BOUNDS_CASES = 8
MERGE_MAX_PARTS = 16


class FaError(RuntimeError):
    """A non-zero fa_status returned by the library."""

    def __init__(self, fn: str, code: int):
        self.code = code
        super().__init__(f"{fn} failed: {status_string(code)}")


def library_path() -> str:
    return os.path.join(_HERE, "libfa.so")


def _load(path):
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`")
    handle = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(handle, name)
        fn.restype = res
        fn.argtypes = args
    return handle


def lib():
    """Loads libfa.so once (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        _LIB = _load(library_path())
    return _LIB


_DEBUG_LIB = None


def debug_library_path() -> str:
    return os.path.join(_HERE, "libfa_debug.so")


def debug_lib():
    """Loads libfa_debug.so once: the same entry points with device-side bounds
    and alignment checks compiled into the kernels (raises if not built)."""
    global _DEBUG_LIB
    if _DEBUG_LIB is None:
        _DEBUG_LIB = _load(debug_library_path())
    return _DEBUG_LIB


@contextlib.contextmanager
def debug_checks():
    """Within the block, every call of this module runs the debug build
    (libfa_debug.so); a failed device-side check then shows up as
    FA_ERR_BOUNDS from sync_status().  Not thread-safe: it swaps the library
    handle this module uses."""
    global _LIB
    saved = lib()
    _LIB = debug_lib()
    try:
        yield
    finally:
        _LIB = saved


def status_string(code: int) -> str:
    try:
        return lib().fa_status_string(int(code)).decode()
    except Exception:  # library not loadable: fall back to the static table
        return _STATUS.get(int(code), f"status {code}")


def _check(fn: str, code: int) -> None:
    if code != 0:
        raise FaError(fn, code)


def _dtype_code(t: torch.Tensor) -> int:
    return _code(t.dtype)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None and t.numel() > 0 else ctypes.c_void_p(0)


def _stream(t: torch.Tensor) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _check_tensors(qside, kside):
    """q-side tensors (q, o, dO) are [B, H, Nq, d]; k-side (k, v) [B, H, Nk, d]."""
    ref = qside[0]
    if ref.dim() != 4:
        raise ValueError("tensors must be [B, H, N, d]")
    for t in qside + kside:
        if not t.is_cuda:
            raise ValueError("tensors must be CUDA tensors")
        if t.dim() != 4 or t.dtype != ref.dtype or t.device != ref.device:
            raise ValueError("q, k, v (and o, dO) must be [B, H, N, d] with one dtype and device")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous [B, H, N, d]")
    for t in qside:
        if t.shape != ref.shape:
            raise ValueError("q, o and dO must share one shape [B, H, Nq, d]")
    kref = kside[0]
    for t in kside:
        if t.shape != kref.shape:
            raise ValueError("k and v must share one shape [B, H, Nk, d]")
    if kref.shape[:2] != ref.shape[:2] or kref.shape[3] != ref.shape[3]:
        raise ValueError("q and k must agree on B, H and d")


def _code(dtype) -> int:
    if dtype not in _CODES:
        raise TypeError(f"unsupported dtype {dtype}; use torch.bfloat16, torch.float16 or torch.float32")
    return _CODES[dtype]


def fwd_workspace_size(B, H, N, d, causal=False, dtype=torch.bfloat16, Nk=None) -> int:
    """Bytes of the forward's optional load-balancing workspace (N queries over Nk keys, Nk = N by default)."""
    Nk = N if Nk is None else Nk
    return int(lib().fa_fwd_kv_workspace_size(B, H, N, Nk, d, int(bool(causal)), _code(dtype)))


def fwd(q, k, v, scale=None, causal=False, workspace=None):
    """Attention forward.  q [B,H,Nq,d], k and v [B,H,Nk,d]; returns
    (o [B,H,Nq,d] in q's dtype, lse [B,H,Nq] float32).  Under ``causal`` the
    queries are the last Nq positions: query i sees keys j <= i + Nk - Nq.

    ``workspace``: None allocates the optional load-balancing workspace with
    torch when the library asks for one; a uint8 CUDA tensor is used as given;
    False runs without one.
    """
    _check_tensors([q], [k, v])
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    scale = float(d ** -0.5 if scale is None else scale)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    with torch.cuda.device(q.device):
        if workspace is None:
            n = fwd_workspace_size(B, H, Nq, d, causal, q.dtype, Nk)
            workspace = torch.empty(n, dtype=torch.uint8, device=q.device) if n else False
        ws, n = (None, 0) if workspace is False else (workspace, workspace.numel())
        _check("fa_fwd_kv", lib().fa_fwd_kv(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Nq, Nk, d, scale,
                                            int(bool(causal)), _dtype_code(q), _ptr(ws), n, _stream(q)))
    return o, lse


def bwd_workspace_size(B, H, N, d, dtype=torch.bfloat16, Nk=None) -> int:
    """Bytes of the backward's workspace (N queries over Nk keys, Nk = N by default)."""
    Nk = N if Nk is None else Nk
    return int(lib().fa_bwd_kv_workspace_size(B, H, N, Nk, d, _code(dtype)))


def _workspace(q, k):
    B, H, Nq, d = q.shape
    n = bwd_workspace_size(B, H, Nq, d, q.dtype, k.shape[2])
    # torch's caching allocator returns blocks aligned to at least 512 bytes
    return torch.empty(max(n, 1), dtype=torch.uint8, device=q.device), n


def bwd(q, k, v, o, do, lse, scale=None, causal=False, workspace=None):
    """Attention backward.  Returns (dq like q, dk and dv like k)."""
    _check_tensors([q, o, do], [k, v])
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if lse.shape != (B, H, Nq) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 [B, H, Nq] tensor")
    scale = float(d ** -0.5 if scale is None else scale)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws, n = _workspace(q, k) if workspace is None else (workspace, workspace.numel())
    with torch.cuda.device(q.device):
        _check("fa_bwd_kv", lib().fa_bwd_kv(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq),
                                            _ptr(dk), _ptr(dv), B, H, Nq, Nk, d, scale, int(bool(causal)),
                                            _dtype_code(q), _ptr(ws), n, _stream(q)))
    return dq, dk, dv


def merge(o_parts, lse_parts, out=None):
    """Merge partial results of the same queries over disjoint key sets.

    o_parts: list of [B,H,N,d] tensors (one dtype); lse_parts: list of
    [B,H,N] float32 tensors.  Returns (o, lse); ``out`` = (o, lse) writes into
    given tensors, which may be one of the parts (in-place running state).
    """
    if not o_parts or len(o_parts) != len(lse_parts) or len(o_parts) > MERGE_MAX_PARTS:
        raise ValueError(f"need 1..{MERGE_MAX_PARTS} parts with one LSE each")
    ref = o_parts[0]
    for t in o_parts:
        if not t.is_cuda or t.shape != ref.shape or t.dtype != ref.dtype or not t.is_contiguous():
            raise ValueError("O parts must be contiguous CUDA tensors of one shape and dtype")
    B, H, N, d = ref.shape
    for t in lse_parts:
        if t.shape != (B, H, N) or t.dtype != torch.float32 or not t.is_contiguous() or not t.is_cuda:
            raise ValueError("LSE parts must be contiguous float32 CUDA tensors [B, H, N]")
    o, lse = out if out is not None else (torch.empty_like(ref), torch.empty_like(lse_parts[0]))
    n = len(o_parts)
    o_arr = (ctypes.c_void_p * n)(*[t.data_ptr() for t in o_parts])
    l_arr = (ctypes.c_void_p * n)(*[t.data_ptr() for t in lse_parts])
    with torch.cuda.device(ref.device):
        _check("fa_merge", lib().fa_merge(ctypes.cast(o_arr, ctypes.c_void_p), ctypes.cast(l_arr, ctypes.c_void_p), n,
                                          _ptr(o), _ptr(lse), B, H, N, d, _dtype_code(ref), _stream(ref)))
    return o, lse


def bwd_stages(q, k, v, o, do, lse, dq, dk, dv, workspace, scale=None, causal=False, between=None):
    """fa_bwd as its three stages on the current stream, writing into dq/dk/dv.

    ``between`` is an optional pair of callables run just before and just
    after the tiled stage (the bench records CUDA events there).
    """
    _check_tensors([q, o, do, dq], [k, v, dk, dv])
    B, H, N, d = q.shape
    if k.shape[2] != N:
        raise ValueError("the stage entry points take square problems (Nq = Nk)")
    scale = float(d ** -0.5 if scale is None else scale)
    code = _dtype_code(q)
    s = _stream(q)
    L = lib()
    n = workspace.numel()
    _check("fa_bwd_prep", L.fa_bwd_prep(_ptr(o), _ptr(do), _ptr(lse), B, H, N, d, code, _ptr(workspace), n, s))
    if between:
        between[0]()
    _check("fa_bwd_tiles", L.fa_bwd_tiles(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(dq), _ptr(dk), _ptr(dv), B, H, N,
                                          d, scale, int(bool(causal)), code, _ptr(workspace), n, s))
    if between:
        between[1]()
    _check("fa_bwd_dq_finish", L.fa_bwd_dq_finish(_ptr(dq), B, H, N, d, scale, code, _ptr(workspace), n, s))


def sync_status(device=None) -> int:
    """Synchronises the current stream and returns the library's fault status (0 = OK)."""
    dev = torch.device("cuda") if device is None else torch.device(device)
    with torch.cuda.device(dev):
        return int(lib().fa_sync_status(ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)))
