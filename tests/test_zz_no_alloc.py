"""fa_bwd_noalloc: the backward for callers that cannot allocate device memory.

Such callers (a runtime that forbids allocation after start-up, a plug-in whose
host owns every device allocation) cannot hand fa_bwd a workspace, so this
entry point uses a fixed scratch array compiled into the library.  The test
calls it through the C ABI twice in a row, with different inputs, and checks
each result against fa_bwd with a caller-provided workspace, within the
tolerances the other tests use: dK and dV are reproducible bit for bit, dQ
(float32 reductions in varying order) within 1e-2.  Between a warm-up call
and the end of the two checked calls the device's free memory must not
change: the calls allocate nothing.  It also checks that a problem larger
than the built-in scratch is refused.  This file sorts last so that a run
stopping at the first failure has already run every other test.
"""

import ctypes

import pytest
import torch

from exact_tiled_attention_12_gb300.synthetic import make_inputs

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 32 << 20   # FA_NOALLOC_SCRATCH_BYTES in include/fa.h


@pytest.fixture(scope="module")
def fa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    import exact_tiled_attention_12_gb300 as fa

    return fa


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


_CODES = {torch.bfloat16: 0, torch.float32: 1, torch.float16: 2}


def _noalloc_into(fa, q, k, v, o, do, lse, causal, out):
    """fa_bwd_noalloc through the C ABI, into preallocated dq, dk, dv."""
    B, H, N, d = q.shape
    dq, dk, dv = out
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = fa.lib().fa_bwd_noalloc(_p(q), _p(k), _p(v), _p(o), _p(do), _p(lse), _p(dq), _p(dk), _p(dv),
                                 B, H, N, d, d ** -0.5, int(causal), _CODES[q.dtype], stream)
    assert st == 0, fa.status_string(st)


@pytest.mark.parametrize("dtype,shape,causal", [
    ("bf16", (1, 2, 512, 128), True),
    ("bf16", (2, 2, 384, 64), False),
    ("fp16", (1, 3, 256, 128), False),
    ("bf16", (1, 2, 300, 256), True),   # d = 256: dQ from its own kernel, no accumulator in the scratch
    ("fp32", (1, 2, 200, 64), True),
])
def test_noalloc_matches_fa_bwd_twice(fa, dtype, shape, causal):
    # Everything the checked calls need is allocated first; fa_bwd with a
    # caller workspace gives the expected results.
    cases = []
    for seed in (21, 22):   # two calls in a row; the second sees the first's leftovers
        q, k, v, do = make_inputs(*shape, dtype, "normal", seed, device="cuda")
        o, lse = fa.fwd(q, k, v, causal=causal)
        want = fa.bwd(q, k, v, o, do, lse, causal=causal)
        out = tuple(torch.empty_like(t) for t in (q, k, v))
        cases.append(((q, k, v, o, do, lse), want, out))
    warm = tuple(torch.empty_like(t) for t in cases[0][2])
    _noalloc_into(fa, *cases[0][0], causal, warm)   # warm-up: the library's modules are loaded by now
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    for args, _, out in cases:
        _noalloc_into(fa, *args, causal, out)
    assert fa.sync_status() == 0
    assert torch.cuda.mem_get_info()[0] == free_before, "fa_bwd_noalloc changed the device's free memory"
    for _, want, got in cases:
        if dtype in ("bf16", "fp16"):
            assert torch.equal(got[1], want[1]) and torch.equal(got[2], want[2])
            assert float((got[0].float() - want[0].float()).abs().max()) <= 1e-2
        else:
            for g, w_ in zip(got, want):
                assert float((g - w_).abs().max()) <= 1e-5


def test_noalloc_rejects_problems_beyond_the_scratch(fa):
    B, H, N, d = 1, 16, 4096, 128
    assert fa.bwd_workspace_size(B, H, N, d) > SCRATCH_BYTES
    fake = ctypes.c_void_p(0x10000)
    st = fa.lib().fa_bwd_noalloc(*([fake] * 9), B, H, N, d, d ** -0.5, 0, 0, None)
    assert st == 4   # FA_ERR_WORKSPACE, returned before anything is enqueued
