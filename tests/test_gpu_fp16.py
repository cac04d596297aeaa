"""GPU parity for the fp16 dtype (IEEE half inputs and outputs, P and dS
rounded to fp16 before their tensor-core products, fp32 accumulation).

Same tolerances as bf16 (fp16 keeps 3 more mantissa bits over a smaller
range); shapes cover aligned and ragged lengths, both masks, Nq != Nk, the
split forward, large scores, the merge and autograd.
"""

import numpy as np
import pytest
import torch

from exact_tiled_attention_12_gb300.synthetic import make_inputs, make_inputs_kv

from ._helpers import compare, run_library, run_oracle_heads, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()


def _heads(B, H):
    return [(b, h) for b in range(B) for h in range(H)]


@pytest.mark.parametrize("B,H,N,d", [(1, 2, 256, 128), (2, 1, 384, 64), (1, 2, 200, 128), (1, 1, 1000, 64)])
@pytest.mark.parametrize("causal", [False, True])
def test_fp16_parity(B, H, N, d, causal):
    q, k, v, do = make_inputs(B, H, N, d, "fp16", "normal", 300 + N + d, device="cuda")
    gpu = run_library(q, k, v, do, causal, d ** -0.5)
    ref = run_oracle_heads(q, k, v, do, causal, d ** -0.5, _heads(B, H))
    errs = compare({key: val.reshape((-1,) + val.shape[2:]) for key, val in gpu.items()}, ref, "fp16")
    # fp16 rounds P, dS and the outputs with 11-bit significands: tighter than bf16
    assert errs["O"] <= 3e-3


@pytest.mark.parametrize("causal", [False, True])
def test_fp16_kv_and_stress(causal):
    import exact_tiled_attention_12_gb300 as fa

    q, k, v, do = make_inputs_kv(2, 1, 150, 333, 64, "fp16", "stress", 301, device="cuda")
    o, lse = fa.fwd(q, k, v, causal=causal)
    dq, dk, dv = fa.bwd(q, k, v, o, do, lse, causal=causal)
    assert fa.sync_status() == 0
    gpu = {"O": to64(o), "LSE": to64(lse), "dQ": to64(dq), "dK": to64(dk), "dV": to64(dv)}
    ref = run_oracle_heads(q, k, v, do, causal, 64 ** -0.5, _heads(2, 1))
    compare({key: val.reshape((-1,) + val.shape[2:]) for key, val in gpu.items()}, ref, "fp16")


def test_fp16_split_forward_and_merge():
    import oracle

    import exact_tiled_attention_12_gb300 as fa

    B, H, N, d = 1, 1, 2048, 128
    assert fa.fwd_workspace_size(B, H, N, d, dtype=torch.float16) > 0
    q, k, v, _ = make_inputs(B, H, N, d, "fp16", "normal", 302, device="cuda")
    o, lse = fa.fwd(q, k, v)
    parts = [fa.fwd(q, k[:, :, a:b].contiguous(), v[:, :, a:b].contiguous()) for a, b in ((0, 700), (700, N))]
    om, lsem = fa.merge([p[0] for p in parts], [p[1] for p in parts])
    assert fa.sync_status() == 0
    ref_o, ref_lse = oracle.attention_forward_head(to64(q[0, 0]), to64(k[0, 0]), to64(v[0, 0]), d ** -0.5)
    for oo, ll in ((o, lse), (om, lsem)):
        assert np.max(np.abs(to64(oo[0, 0]) - ref_o)) <= 3e-3
        assert np.max(np.abs(to64(ll[0, 0]) - ref_lse)) <= 1e-3


def test_fp16_autograd():
    import exact_tiled_attention_12_gb300 as fa

    B, H, N, d = 1, 2, 256, 64
    q, k, v, do = make_inputs(B, H, N, d, "fp16", "normal", 303, device="cuda")
    q, k, v = (t.clone().requires_grad_(True) for t in (q, k, v))
    o = fa.attention(q, k, v, causal=True)
    o.backward(do)
    ref = run_oracle_heads(q.detach(), k.detach(), v.detach(), do, True, d ** -0.5, _heads(B, H))
    gpu = {"O": to64(o.detach()[0]), "LSE": ref["LSE"], "dQ": to64(q.grad[0]), "dK": to64(k.grad[0]),
           "dV": to64(v.grad[0])}
    compare(gpu, ref, "fp16")
