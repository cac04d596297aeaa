"""GPU parity at head dimension 256 (bf16 and fp16) against the fp64 oracle.

d = 256 runs its own kernels: the forward keeps one 128-row query tile per
CTA with two score buffers; the backward computes dK/dV over 64-key tiles and
dQ over 128-query tiles in two kernels.  Shapes cover several tiles, ragged
Nq and Nk, fewer queries than keys under the offset causal mask, a decode
step whose keys are split over several CTAs and merged, and large scores.
"""

import numpy as np
import pytest
import torch

from exact_tiled_attention_12_gb300.synthetic import make_inputs_kv

from ._helpers import BF16_LSE_ATOL, BF16_O_ATOL, compare, run_oracle_heads, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()


def _heads(B, H):
    return [(b, h) for b in range(B) for h in range(H)]


def _oracle_forward(q, k, v, causal):
    import oracle

    d = q.shape[-1]
    out = {"O": [], "LSE": []}
    for b, h in _heads(q.shape[0], q.shape[1]):
        o, lse = oracle.attention_forward_head(to64(q[b, h]), to64(k[b, h]), to64(v[b, h]), d ** -0.5, causal)
        out["O"].append(o)
        out["LSE"].append(lse)
    return {key: np.stack(val) for key, val in out.items()}


def _flat(res):
    return {key: val.reshape((-1,) + val.shape[2:]) for key, val in res.items()}


FWD_SHAPES = [
    (1, 2, 512, 512),      # four query tiles, four K/V tiles
    (2, 1, 333, 333),      # ragged: the last tiles hold 77 rows / keys
    (1, 2, 200, 1000),     # Nq < Nk, both ragged; causal offset 800
    (1, 2, 1, 8192),       # a decode step: the keys split over several CTAs
    (1, 1, 1024, 8192),    # eight query tiles per head, keys split (combine indexing)
    (1, 1, 130, 130),      # two query tiles, the second with 2 rows
]


@pytest.mark.parametrize("B,H,Nq,Nk", FWD_SHAPES)
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_d256_forward(B, H, Nq, Nk, causal, dtype):
    import exact_tiled_attention_12_gb300 as fa

    d = 256
    q, k, v, do = make_inputs_kv(B, H, Nq, Nk, d, dtype, "normal", 300 + Nq + Nk, device="cuda")
    o, lse = fa.fwd(q, k, v, causal=causal)
    assert fa.sync_status() == 0
    ref = _oracle_forward(q, k, v, causal)
    go, gl = to64(o).reshape((-1, Nq, d)), to64(lse).reshape((-1, Nq))
    assert np.all(np.isfinite(go)) and np.all(np.isfinite(gl))
    assert np.max(np.abs(go - ref["O"])) <= BF16_O_ATOL
    assert np.max(np.abs(gl - ref["LSE"])) <= BF16_LSE_ATOL


BWD_SHAPES = [
    (1, 2, 512, 512),      # four query tiles, eight 64-key tiles
    (2, 1, 333, 333),      # ragged: 77-row query tile, 13-key last key tile
    (1, 2, 200, 1000),     # Nq < Nk, both ragged; causal offset 800 (not a tile multiple)
    (1, 1, 130, 130),      # two query tiles, the second with 2 rows
    (1, 1, 1, 300),        # one query
]


@pytest.mark.parametrize("B,H,Nq,Nk", BWD_SHAPES)
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_d256_forward_backward(B, H, Nq, Nk, causal, dtype):
    import exact_tiled_attention_12_gb300 as fa

    d = 256
    q, k, v, do = make_inputs_kv(B, H, Nq, Nk, d, dtype, "normal", 400 + Nq + Nk, device="cuda")
    o, lse = fa.fwd(q, k, v, causal=causal)
    dq, dk, dv = fa.bwd(q, k, v, o, do, lse, causal=causal)
    assert fa.sync_status() == 0
    gpu = {"O": to64(o), "LSE": to64(lse), "dQ": to64(dq), "dK": to64(dk), "dV": to64(dv)}
    ref = run_oracle_heads(q, k, v, do, causal, d ** -0.5, _heads(B, H))
    compare(_flat(gpu), ref, "bf16")


def test_d256_large_scores():
    """Scores of magnitude ~ 8·8·√256 / 16: the online max and the recomputed P stay exact."""
    import exact_tiled_attention_12_gb300 as fa

    B, H, N, d = 1, 2, 384, 256
    q, k, v, do = make_inputs_kv(B, H, N, N, d, "bf16", "stress", 77, device="cuda")
    for causal in (False, True):
        o, lse = fa.fwd(q, k, v, causal=causal)
        dq, dk, dv = fa.bwd(q, k, v, o, do, lse, causal=causal)
        assert fa.sync_status() == 0
        gpu = {"O": to64(o), "LSE": to64(lse), "dQ": to64(dq), "dK": to64(dk), "dV": to64(dv)}
        ref = run_oracle_heads(q, k, v, do, causal, d ** -0.5, _heads(B, H))
        compare(_flat(gpu), ref, "bf16")


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_d256_more_queries_than_keys_without_mask(dtype):
    import exact_tiled_attention_12_gb300 as fa

    B, H, Nq, Nk, d = 1, 2, 300, 77, 256
    q, k, v, do = make_inputs_kv(B, H, Nq, Nk, d, dtype, "normal", 9 + Nq, device="cuda")
    o, lse = fa.fwd(q, k, v)
    dq, dk, dv = fa.bwd(q, k, v, o, do, lse)
    assert fa.sync_status() == 0
    gpu = {"O": to64(o), "LSE": to64(lse), "dQ": to64(dq), "dK": to64(dk), "dV": to64(dv)}
    ref = run_oracle_heads(q, k, v, do, False, d ** -0.5, _heads(B, H))
    compare(_flat(gpu), ref, "bf16")


def test_d256_autograd():
    """attention() at d = 256: gradients through .backward() against the oracle."""
    import exact_tiled_attention_12_gb300 as fa

    B, H, Nq, Nk, d = 1, 2, 150, 420, 256
    q, k, v, do = make_inputs_kv(B, H, Nq, Nk, d, "bf16", "normal", 81, device="cuda")
    q, k, v = (t.clone().requires_grad_(True) for t in (q, k, v))
    o = fa.attention(q, k, v, causal=True)
    o.backward(do)
    assert fa.sync_status() == 0
    ref = run_oracle_heads(q.detach(), k.detach(), v.detach(), do, True, d ** -0.5, _heads(B, H))
    gpu = {"O": to64(o.detach()[0]), "LSE": ref["LSE"], "dQ": to64(q.grad[0]), "dK": to64(k.grad[0]),
           "dV": to64(v.grad[0])}
    compare(gpu, ref, "bf16")
