"""GPU parity of the decoding step (one query per head over Nk keys), and of
a few queries per head over a long cache.

A single query runs a streaming kernel on the CUDA cores (the step is bound
by reading K and V, not by arithmetic), its keys split over several CTAs when
a workspace is given and merged afterwards.  Covered: every supported head
dimension, bf16 and fp16, key counts from 1 to tens of thousands (ragged
against every split), with and without the workspace (one CTA per head),
the causal flag (one query sees every key), large scores, and the state a
decoding loop keeps (each step's O and LSE merged with the next chunk's).
Two to five queries per head (e.g. checking draft tokens; under the mask
the last positions) run the tensor-core forward.
"""

import numpy as np
import pytest
import torch

from exact_tiled_attention_12_gb300.synthetic import make_inputs_kv

from ._helpers import BF16_LSE_ATOL, BF16_O_ATOL, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()


def _oracle(q, k, v, scale, causal=False):
    import oracle

    B, H = q.shape[:2]
    o = np.zeros(q.shape, dtype=np.float64)
    lse = np.zeros(q.shape[:3], dtype=np.float64)
    for b in range(B):
        for h in range(H):
            o[b, h], lse[b, h] = oracle.attention_forward_head(to64(q[b, h]), to64(k[b, h]), to64(v[b, h]), scale, causal)
    return o, lse


def _check(o, lse, ref_o, ref_lse):
    go, gl = to64(o), to64(lse)
    assert np.all(np.isfinite(go)) and np.all(np.isfinite(gl))
    assert np.max(np.abs(go - ref_o)) <= BF16_O_ATOL, np.max(np.abs(go - ref_o))
    assert np.max(np.abs(gl - ref_lse)) <= BF16_LSE_ATOL, np.max(np.abs(gl - ref_lse))


@pytest.mark.parametrize("d", [64, 96, 128, 256])
@pytest.mark.parametrize("Nk", [1, 7, 300, 4099, 20000])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_decode_parity(d, Nk, dtype):
    import exact_tiled_attention_12_gb300 as fa

    B, H = 2, 3
    q, k, v, _ = make_inputs_kv(B, H, 1, Nk, d, dtype, "normal", 500 + d + Nk, device="cuda")
    o, lse = fa.fwd(q, k, v, causal=True)
    assert fa.sync_status() == 0
    _check(o, lse, *_oracle(q, k, v, d ** -0.5))


@pytest.mark.parametrize("d", [64, 128, 256])
def test_decode_without_workspace(d):
    """workspace=False: one CTA per head writes O and LSE itself (no merge)."""
    import exact_tiled_attention_12_gb300 as fa

    B, H, Nk = 1, 4, 5000
    q, k, v, _ = make_inputs_kv(B, H, 1, Nk, d, "bf16", "normal", 600 + d, device="cuda")
    o, lse = fa.fwd(q, k, v, workspace=False)
    o2, lse2 = fa.fwd(q, k, v)
    assert fa.sync_status() == 0
    ref = _oracle(q, k, v, d ** -0.5)
    _check(o, lse, *ref)
    _check(o2, lse2, *ref)


def test_decode_large_scores():
    import exact_tiled_attention_12_gb300 as fa

    B, H, Nk, d = 2, 2, 3000, 128
    q, k, v, _ = make_inputs_kv(B, H, 1, Nk, d, "bf16", "stress", 71, device="cuda")
    o, lse = fa.fwd(q, k, v)
    assert fa.sync_status() == 0
    _check(o, lse, *_oracle(q, k, v, d ** -0.5))


def test_decode_split_boundaries_match_one_cta():
    """The split result equals the single-CTA result to rounding: the merge is exact."""
    import exact_tiled_attention_12_gb300 as fa

    q, k, v, _ = make_inputs_kv(1, 8, 1, 12345, 128, "bf16", "normal", 9, device="cuda")
    o1, l1 = fa.fwd(q, k, v, workspace=False)
    o2, l2 = fa.fwd(q, k, v)
    assert fa.sync_status() == 0
    assert float((l1 - l2).abs().max()) <= 1e-4
    assert float((o1.float() - o2.float()).abs().max()) <= 1e-2


def test_decode_loop_keeps_running_state():
    """A decoding loop: each step's (O, LSE) over the cache so far, merged with
    the next chunk of keys, equals one call over all keys."""
    import exact_tiled_attention_12_gb300 as fa

    B, H, d = 1, 2, 128
    q, k, v, _ = make_inputs_kv(B, H, 1, 3000, d, "bf16", "normal", 31, device="cuda")
    cuts = [0, 1000, 1001, 2500, 3000]
    o = lse = None
    for a, b in zip(cuts[:-1], cuts[1:]):
        oc, lc = fa.fwd(q, k[:, :, a:b].contiguous(), v[:, :, a:b].contiguous())
        if o is None:
            o, lse = oc, lc
        else:
            o, lse = fa.merge([o, oc], [lse, lc])
    assert fa.sync_status() == 0
    _check(o, lse, *_oracle(q, k, v, d ** -0.5))


@pytest.mark.parametrize("d", [64, 96, 128])
@pytest.mark.parametrize("Nq", [2, 3, 4])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nk", [4, 300, 9000])
def test_decode_few_queries(d, Nq, causal, Nk):
    """Two to four queries per head (e.g. checking draft tokens); under the
    mask they are the last Nq positions."""
    import exact_tiled_attention_12_gb300 as fa

    B, H = 2, 3
    q, k, v, _ = make_inputs_kv(B, H, Nq, Nk, d, "bf16", "normal", 700 + d + Nq + Nk, device="cuda")
    o, lse = fa.fwd(q, k, v, causal=causal)
    assert fa.sync_status() == 0
    _check(o, lse, *_oracle(q, k, v, d ** -0.5, causal))


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_decode_few_queries_without_workspace_and_equal_lengths(dtype):
    import exact_tiled_attention_12_gb300 as fa

    for Nq, Nk in ((4, 4), (3, 3), (4, 5000)):
        q, k, v, _ = make_inputs_kv(1, 2, Nq, Nk, 128, dtype, "normal", 17 + Nk, device="cuda")
        for ws in (None, False):
            o, lse = fa.fwd(q, k, v, causal=True, workspace=ws)
            assert fa.sync_status() == 0
            _check(o, lse, *_oracle(q, k, v, 128 ** -0.5, True))


def test_five_queries():
    import exact_tiled_attention_12_gb300 as fa

    q, k, v, _ = make_inputs_kv(1, 2, 5, 3000, 128, "bf16", "normal", 23, device="cuda")
    o, lse = fa.fwd(q, k, v, causal=True)
    assert fa.sync_status() == 0
    _check(o, lse, *_oracle(q, k, v, 128 ** -0.5, True))
