"""GPU parity for Nq queries over Nk keys, and for the merge of partial results.

Under the causal mask the queries are the last Nq positions (query i sees
keys j <= i + Nk - Nq).  Shapes cover a query/key offset that is a multiple
of the 128-row tile and one that is not (the mask then crosses two K/V
tiles), ragged Nq and Nk, a single query over a long key sequence (a decode
step) and more queries than keys without the mask.  The merge tests rebuild
full attention from parts over disjoint key ranges, in place as a running
state, and the prefix-caching split (cached keys without the mask, new keys
with it).  Everything is compared with the fp64 oracle.
"""

import numpy as np
import pytest
import torch

from exact_tiled_attention_12_gb300.synthetic import make_inputs_kv

from ._helpers import compare, run_oracle_heads, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()


def _heads(B, H):
    return [(b, h) for b in range(B) for h in range(H)]


def _run(q, k, v, do, causal):
    import exact_tiled_attention_12_gb300 as fa

    o, lse = fa.fwd(q, k, v, causal=causal)
    dq, dk, dv = fa.bwd(q, k, v, o, do, lse, causal=causal)
    assert fa.sync_status() == 0
    return {"O": to64(o), "LSE": to64(lse), "dQ": to64(dq), "dK": to64(dk), "dV": to64(dv)}


KV_SHAPES = [
    (1, 2, 128, 384, 128),   # offset 256: a whole number of tiles
    (1, 2, 256, 320, 64),    # offset 64: the mask crosses two K/V tiles; ragged Nk
    (2, 1, 200, 1000, 128),  # ragged Nq and Nk, offset 800
    (1, 1, 77, 589, 64),     # offset 512 with a 77-row query tile
    (1, 2, 1, 4096, 128),    # one query over 4096 keys (a decode step)
    (2, 2, 130, 430, 128),   # offset 300, two query tiles, the second with 2 rows
    (1, 2, 1, 32768, 128),   # one query over 32768 keys: the keys split over 16 CTAs
]


@pytest.mark.parametrize("B,H,Nq,Nk,d", KV_SHAPES)
@pytest.mark.parametrize("causal", [False, True])
def test_bf16_kv_parity(B, H, Nq, Nk, d, causal):
    q, k, v, do = make_inputs_kv(B, H, Nq, Nk, d, "bf16", "normal", 100 + Nq + Nk + d, device="cuda")
    gpu = _run(q, k, v, do, causal)
    ref = run_oracle_heads(q, k, v, do, causal, d ** -0.5, _heads(B, H))
    compare({key: val.reshape((-1,) + val.shape[2:]) for key, val in gpu.items()}, ref, "bf16")


@pytest.mark.parametrize("B,H,Nq,Nk,d", [(1, 2, 384, 128, 128), (1, 1, 300, 77, 64)])
def test_bf16_more_queries_than_keys_without_mask(B, H, Nq, Nk, d):
    q, k, v, do = make_inputs_kv(B, H, Nq, Nk, d, "bf16", "normal", 7 + Nq, device="cuda")
    gpu = _run(q, k, v, do, False)
    ref = run_oracle_heads(q, k, v, do, False, d ** -0.5, _heads(B, H))
    compare({key: val.reshape((-1,) + val.shape[2:]) for key, val in gpu.items()}, ref, "bf16")


@pytest.mark.parametrize("B,H,Nq,Nk,d", [(1, 2, 37, 100, 40), (2, 1, 1, 300, 64), (1, 1, 64, 64 + 33, 128)])
@pytest.mark.parametrize("causal", [False, True])
def test_fp32_kv_parity(B, H, Nq, Nk, d, causal):
    q, k, v, do = make_inputs_kv(B, H, Nq, Nk, d, "fp32", "normal", 200 + Nq + Nk, device="cuda")
    gpu = _run(q, k, v, do, causal)
    ref = run_oracle_heads(q, k, v, do, causal, d ** -0.5, _heads(B, H))
    compare({key: val.reshape((-1,) + val.shape[2:]) for key, val in gpu.items()}, ref, "fp32")


def test_bf16_kv_stress_ragged_causal():
    """Large scores, offset not a multiple of the tile, ragged tail keys."""
    q, k, v, do = make_inputs_kv(2, 1, 150, 333, 64, "bf16", "stress", 9, device="cuda")
    for causal in (False, True):
        gpu = _run(q, k, v, do, causal)
        ref = run_oracle_heads(q, k, v, do, causal, 64 ** -0.5, _heads(2, 1))
        compare({key: val.reshape((-1,) + val.shape[2:]) for key, val in gpu.items()}, ref, "bf16")


def test_suffix_queries_match_the_square_problem():
    """The last Nq queries of a square causal problem, run alone over all keys,
    give that problem's last Nq rows (both on the GPU, within bf16 rounding)."""
    import exact_tiled_attention_12_gb300 as fa

    q, k, v, _ = make_inputs_kv(1, 2, 640, 640, 128, "bf16", "normal", 31, device="cuda")
    o_full, lse_full = fa.fwd(q, k, v, causal=True)
    for nq in (128, 200, 1):
        o_s, lse_s = fa.fwd(q[:, :, 640 - nq:].contiguous(), k, v, causal=True)
        assert float((o_s.float() - o_full[:, :, 640 - nq:].float()).abs().max()) <= 1e-2
        assert float((lse_s - lse_full[:, :, 640 - nq:]).abs().max()) <= 1e-4


# ------------------------------------------------------------------ merge


def _oracle_forward(q, k, v, causal, scale):
    import oracle

    B, H = q.shape[:2]
    o = np.stack([np.stack([oracle.attention_forward_head(to64(q[b, h]), to64(k[b, h]), to64(v[b, h]), scale,
                                                          causal)[0] for h in range(H)]) for b in range(B)])
    lse = np.stack([np.stack([oracle.attention_forward_head(to64(q[b, h]), to64(k[b, h]), to64(v[b, h]), scale,
                                                            causal)[1] for h in range(H)]) for b in range(B)])
    return o, lse


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_merge_of_key_ranges_equals_full_attention(dtype):
    import exact_tiled_attention_12_gb300 as fa

    B, H, Nq, Nk, d = 2, 2, 96, 1000, 64
    q, k, v, _ = make_inputs_kv(B, H, Nq, Nk, d, dtype, "normal", 51, device="cuda")
    cuts = [0, 129, 130, 700, Nk]
    parts = [fa.fwd(q, k[:, :, a:b].contiguous(), v[:, :, a:b].contiguous()) for a, b in zip(cuts, cuts[1:])]
    o, lse = fa.merge([p[0] for p in parts], [p[1] for p in parts])
    assert fa.sync_status() == 0
    ref_o, ref_lse = _oracle_forward(q, k, v, False, d ** -0.5)
    tol_o = 1e-2 if dtype == "bf16" else 1e-5
    assert np.max(np.abs(to64(o) - ref_o)) <= tol_o
    assert np.max(np.abs(to64(lse) - ref_lse)) <= (1e-3 if dtype == "bf16" else 1e-5)


def test_streaming_decode_merges_in_place():
    """A running (O, LSE) state extended block by block in place (out= one of
    the parts) equals one pass over all keys: the prefix-caching use of the
    merge.  One query per head, 5 key blocks of uneven length."""
    import exact_tiled_attention_12_gb300 as fa

    B, H, Nk, d = 2, 4, 2000, 128
    q, k, v, _ = make_inputs_kv(B, H, 1, Nk, d, "bf16", "normal", 52, device="cuda")
    cuts = [0, 300, 301, 1024, 1500, Nk]
    state = None
    for a, b in zip(cuts, cuts[1:]):
        o_b, lse_b = fa.fwd(q, k[:, :, a:b].contiguous(), v[:, :, a:b].contiguous())
        if state is None:
            state = (o_b, lse_b)
        else:
            fa.merge([state[0], o_b], [state[1], lse_b], out=state)
    assert fa.sync_status() == 0
    ref_o, ref_lse = _oracle_forward(q, k, v, False, d ** -0.5)
    # each merge step rounds the running O to bf16 once more
    assert np.max(np.abs(to64(state[0]) - ref_o)) <= 2e-2
    assert np.max(np.abs(to64(state[1]) - ref_lse)) <= 1e-3


@pytest.mark.parametrize("n_new", [1, 64, 200])
def test_prefix_caching_split(n_new):
    """New tokens' queries over cached keys (no mask) merged with the same
    queries over the new keys (causal, square) equal the causal problem of the
    new queries over all keys, computed directly by fa_fwd_kv."""
    import exact_tiled_attention_12_gb300 as fa

    B, H, n_cache, d = 1, 2, 700, 128
    q, k, v, _ = make_inputs_kv(B, H, n_new, n_cache + n_new, d, "bf16", "normal", 53 + n_new, device="cuda")
    o_direct, lse_direct = fa.fwd(q, k, v, causal=True)
    o_a, lse_a = fa.fwd(q, k[:, :, :n_cache].contiguous(), v[:, :, :n_cache].contiguous())
    o_b, lse_b = fa.fwd(q, k[:, :, n_cache:].contiguous(), v[:, :, n_cache:].contiguous(), causal=True)
    o_m, lse_m = fa.merge([o_a, o_b], [lse_a, lse_b])
    assert fa.sync_status() == 0
    ref_o, ref_lse = _oracle_forward(q, k, v, True, d ** -0.5)
    for o, lse in ((o_direct, lse_direct), (o_m, lse_m)):
        assert np.max(np.abs(to64(o) - ref_o)) <= 1e-2
        assert np.max(np.abs(to64(lse) - ref_lse)) <= 1e-3


def test_merge_parts_that_saw_nothing():
    import exact_tiled_attention_12_gb300 as fa

    B, H, N, d = 1, 2, 10, 64
    g = torch.Generator().manual_seed(3)
    o1 = torch.randn((B, H, N, d), generator=g).to(torch.bfloat16).cuda()
    junk = torch.randn((B, H, N, d), generator=g).to(torch.bfloat16).cuda()
    lse1 = torch.randn((B, H, N), generator=g).cuda()
    none = torch.full((B, H, N), float("-inf")).cuda()
    o, lse = fa.merge([junk, o1, junk], [none, lse1, none])
    assert torch.equal(o, o1) and torch.equal(lse, lse1)
    o, lse = fa.merge([junk, junk], [none, none])
    assert fa.sync_status() == 0
    assert bool((o == 0).all()) and bool((lse == float("-inf")).all())


def test_merge_two_parts_closed_form():
    """Weights e^{a}/(e^{a}+e^{b}) and e^{b}/(e^{a}+e^{b}) in fp32 for d = 33 (not a multiple of 32)."""
    import exact_tiled_attention_12_gb300 as fa

    g = torch.Generator().manual_seed(4)
    oa, ob = torch.randn((1, 1, 5, 33), generator=g).cuda(), torch.randn((1, 1, 5, 33), generator=g).cuda()
    la, lb = torch.randn((1, 1, 5), generator=g).cuda(), torch.randn((1, 1, 5), generator=g).cuda()
    o, lse = fa.merge([oa, ob], [la, lb])
    wa = torch.exp(la) / (torch.exp(la) + torch.exp(lb))
    want = wa[..., None] * oa + (1 - wa[..., None]) * ob
    assert float((o - want).abs().max()) <= 1e-6
    assert float((lse - torch.logaddexp(la, lb)).abs().max()) <= 1e-6


def test_autograd_with_fewer_queries_than_keys():
    import exact_tiled_attention_12_gb300 as fa

    B, H, Nq, Nk, d = 1, 2, 100, 356, 64
    q, k, v, do = make_inputs_kv(B, H, Nq, Nk, d, "bf16", "normal", 61, device="cuda")
    q, k, v = (t.clone().requires_grad_(True) for t in (q, k, v))
    o = fa.attention(q, k, v, causal=True)
    o.backward(do)
    ref = run_oracle_heads(q.detach(), k.detach(), v.detach(), do, True, d ** -0.5, _heads(B, H))
    gpu = {"O": to64(o.detach()[0]), "LSE": ref["LSE"], "dQ": to64(q.grad[0]), "dK": to64(k.grad[0]),
           "dV": to64(v.grad[0])}
    compare(gpu, ref, "bf16")


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("causal", [False, True])
def test_d96_kv_and_split(dtype, causal):
    """d = 96 with Nq != Nk, ragged lengths, and a shape whose forward splits."""
    for B, H, Nq, Nk in ((1, 2, 200, 460), (1, 1, 2048, 2048)):
        q, k, v, do = make_inputs_kv(B, H, Nq, Nk, 96, dtype, "normal", 400 + Nq, device="cuda")
        gpu = _run(q, k, v, do, causal)
        ref = run_oracle_heads(q, k, v, do, causal, 96 ** -0.5, _heads(B, H))
        compare({key: val.reshape((-1,) + val.shape[2:]) for key, val in gpu.items()}, ref, dtype)


# ------------------------------------------------------------------ few queries over many keys
#
# With 2 to 128 queries per head and fewer units than SMs, every unit of the
# forward is split over ranges of its K/V tiles (with and without the mask;
# d = 256 only without) and merged on the device; each part keeps one
# partial row per query.

SHORT_SHAPES = [
    # B, H, Nq, Nk, d
    (2, 4, 16, 4096, 128),
    (1, 3, 2, 2000, 64),     # two queries, ragged keys
    (1, 2, 128, 2048, 128),  # a full 128-query tile (16 K/V tiles: two parts of 8)
    (1, 2, 100, 2100, 96),   # d = 96, ragged
    (4, 8, 7, 3000, 128),    # more heads, ragged
    (1, 2, 16, 2048, 256),   # d = 256 (split without the mask only)
]


@pytest.mark.parametrize("B,H,Nq,Nk,d", SHORT_SHAPES)
@pytest.mark.parametrize("causal", [False, True])
def test_few_queries_split_over_keys(B, H, Nq, Nk, d, causal):
    import exact_tiled_attention_12_gb300 as fa

    splits = fa.fwd_workspace_size(B, H, Nq, d, causal, torch.bfloat16, Nk=Nk) > 0
    assert splits == (not (causal and d == 256))   # every shape here has fewer units than SMs
    q, k, v, do = make_inputs_kv(B, H, Nq, Nk, d, "bf16", "normal", 300 + Nq + Nk + d, device="cuda")
    gpu = _run(q, k, v, do, causal)
    ref = run_oracle_heads(q, k, v, do, causal, d ** -0.5, _heads(B, H))
    compare({key: val.reshape((-1,) + val.shape[2:]) for key, val in gpu.items()}, ref, "bf16")


def test_few_queries_split_equals_unsplit_forward():
    """The split forward (workspace given) and the whole-unit forward (no
    workspace) agree on O within bf16 rounding and on LSE within 1e-5."""
    import exact_tiled_attention_12_gb300 as fa

    q, k, v, _ = make_inputs_kv(2, 8, 16, 8192, 128, "bf16", "normal", 77, device="cuda")
    for causal in (False, True):
        o1, l1 = fa.fwd(q, k, v, causal=causal)
        o2, l2 = fa.fwd(q, k, v, causal=causal, workspace=False)
        assert fa.sync_status() == 0
        assert float((o1.float() - o2.float()).abs().max()) <= 2 ** -8
        assert float((l1 - l2).abs().max()) <= 1e-5
