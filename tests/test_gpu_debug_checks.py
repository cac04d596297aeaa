"""The debug build (libfa_debug.so) on the GPU.

Its kernels check every TMA coordinate, shared-memory operand, tensor-memory
column range and bulk copy before using it.  On every kind of shape the
library runs (d = 64, 96, 128, 256; causal and not; ragged N; fewer queries
than keys; a split forward; a decoding step; fp16 and fp32), no check may
fire and the results must equal the release build's: O, LSE, dK and dV bit
for bit, dQ (float32 reductions in a varying order) within 1e-2.  The
self-test kernel evaluates the checks on fixed valid and invalid arguments,
without using them for any access, and must report exactly the invalid ones
and FA_ERR_BOUNDS.
"""

import pytest
import torch

from exact_tiled_attention_12_gb300.synthetic import make_inputs, make_inputs_kv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    import exact_tiled_attention_12_gb300 as fa

    assert fa.debug_lib().fa_debug_checks_enabled() == 1
    return fa


def test_bounds_selftest_reports_exactly_the_invalid_cases(fa):
    import ctypes

    from exact_tiled_attention_12_gb300.binding import FA_SELFTEST_BOUNDS_CASES

    L = fa.debug_lib()
    out = torch.full((FA_SELFTEST_BOUNDS_CASES,), -1, dtype=torch.int32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert L.fa_selftest_bounds_check(ctypes.c_void_p(out.data_ptr()), stream) == 0
    assert L.fa_sync_status(stream) == 7          # FA_ERR_BOUNDS, and the word is cleared
    assert L.fa_sync_status(stream) == 0
    assert out.tolist() == [1, 0, 1, 0, 1, 0, 1, 0]


CASES = [
    # dtype, B, H, Nq, Nk, d, causal
    ("bf16", 1, 2, 512, 512, 128, False),
    ("bf16", 2, 1, 384, 384, 64, True),
    ("bf16", 1, 2, 300, 300, 128, True),     # ragged
    ("bf16", 2, 1, 333, 333, 64, False),     # ragged, masked keys past N
    ("bf16", 1, 2, 256, 640, 96, True),      # fewer queries than keys, d = 96
    ("bf16", 1, 1, 256, 2048, 128, False),   # a split forward (K/V ranges merged on the device)
    ("fp16", 1, 1, 256, 256, 128, False),
    ("bf16", 1, 2, 256, 256, 256, False),    # d = 256
    ("bf16", 1, 2, 300, 300, 256, True),     # d = 256, ragged
    ("bf16", 2, 2, 1, 4096, 128, False),     # a decoding step
    ("fp32", 1, 1, 96, 96, 64, True),
    ("bf16", 8, 32, 1000, 1000, 64, False),  # persistent forward and persistent d = 64 backward, ragged
    ("bf16", 4, 40, 2048, 2048, 128, False), # persistent forward at d = 128
]


@pytest.mark.parametrize("dtype,B,H,Nq,Nk,d,causal", CASES)
def test_debug_build_passes_its_checks_and_matches_release(fa, dtype, B, H, Nq, Nk, d, causal):
    if Nq == Nk:
        q, k, v, do = make_inputs(B, H, Nq, d, dtype, "normal", 31 + Nq, device="cuda")
    else:
        q, k, v, do = make_inputs_kv(B, H, Nq, Nk, d, dtype, "normal", 31 + Nq, device="cuda")
    want_o, want_lse = fa.fwd(q, k, v, causal=causal)
    want = fa.bwd(q, k, v, want_o, do, want_lse, causal=causal)
    assert fa.sync_status() == 0
    with fa.debug_checks():
        o, lse = fa.fwd(q, k, v, causal=causal)
        dq, dk, dv = fa.bwd(q, k, v, o, do, lse, causal=causal)
        assert fa.sync_status() == 0          # no check fired (FA_ERR_BOUNDS would be 7)
    assert torch.equal(o, want_o) and torch.equal(lse, want_lse)
    assert torch.equal(dk, want[1]) and torch.equal(dv, want[2])
    assert float((dq.float() - want[0].float()).abs().max()) <= 1e-2
