"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Shapes span several tiles, an odd number of 128-row tiles (a half-empty
two-tile CTA), single-tile heads, ragged N (a last tile partly past N) and
both masks; the fp32 dtype also covers ragged d.  Tolerances are in
tests/_helpers.py.
"""

import numpy as np
import pytest
import torch

from exact_tiled_attention_12_gb300.synthetic import WORKLOADS, make_inputs, make_workload_inputs

from ._helpers import BF16_GRAD_RTOL_FRO, BF16_LSE_ATOL, compare, rel_fro, run_library, run_oracle_heads, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()


def _all_heads(B, H):
    return [(b, h) for b in range(B) for h in range(H)]


def _check(B, H, N, d, causal, dtype, dist="normal", seed=7):
    q, k, v, do = make_inputs(B, H, N, d, dtype, dist, seed, device="cuda")
    scale = d ** -0.5
    gpu = run_library(q, k, v, do, causal, scale)
    heads = _all_heads(B, H)
    ref = run_oracle_heads(q, k, v, do, causal, scale, heads)
    flat = {key: val.reshape((-1,) + val.shape[2:]) for key, val in gpu.items()}
    return compare(flat, ref, dtype)


# ------------------------------------------------------------------ fp32 dtype


def test_tiny_fp32_workload():
    """The tiny fp32 workload (1 x 1 x 256 x 64, non-causal) within 1e-5."""
    w = WORKLOADS["tiny_fp32"]
    q, k, v, do = make_workload_inputs(w, device="cuda")
    gpu = run_library(q, k, v, do, w.causal, w.scale)
    ref = run_oracle_heads(q, k, v, do, w.causal, w.scale, [(0, 0)])
    compare({key: val[0:1, 0] for key, val in gpu.items()}, ref, "fp32")


@pytest.mark.parametrize("B,H,N,d", [(1, 1, 256, 64), (2, 3, 77, 40), (1, 2, 200, 128), (1, 1, 1, 1), (1, 1, 33, 127)])
@pytest.mark.parametrize("causal", [False, True])
def test_fp32_parity(B, H, N, d, causal):
    _check(B, H, N, d, causal, "fp32", seed=B * 1000 + N + d)


# ------------------------------------------------------------------ bf16 dtype (tensor cores)

BF16_SHAPES = [
    (1, 2, 256, 128),   # one two-tile CTA per head
    (2, 3, 384, 64),    # three tiles: the second CTA's upper tile is past N
    (1, 1, 128, 128),   # a single tile
    (1, 1, 128, 64),
    (1, 2, 1024, 128),  # several K/V stages and ring wrap-around
    (3, 2, 640, 64),
    (1, 2, 200, 128),   # ragged: one two-tile CTA, the second tile holds 72 rows
    (2, 1, 333, 64),    # ragged: three tiles, 77 rows in the last
    (1, 1, 1, 128),     # a single row
    (1, 1, 127, 64),
    (2, 2, 1000, 128),  # ragged with several K/V stages
    (1, 2, 256, 96),    # d = 96: tiles padded to 128 columns
    (2, 1, 333, 96),
    (2, 1, 256, 64),    # d = 64, two query tiles: both score buffers, nothing issued two tiles ahead
    (1, 1, 896, 64),    # d = 64, seven query tiles: each score buffer reused, the Q/dO ring wraps twice
]


@pytest.mark.parametrize("B,H,N,d", BF16_SHAPES)
@pytest.mark.parametrize("causal", [False, True])
def test_bf16_parity(B, H, N, d, causal):
    _check(B, H, N, d, causal, "bf16", seed=B * 1000 + N + d + int(causal))


@pytest.mark.parametrize("B,H,N,d", [(1, 1, 2048, 128), (1, 2, 4096, 64), (2, 1, 2176, 128), (1, 1, 2100, 128)])
def test_bf16_split_forward(B, H, N, d):
    """The load-balanced forward (last-wave units split over K/V ranges and
    merged on the device) against the oracle and against the unsplit run."""
    import exact_tiled_attention_12_gb300 as fa

    assert fa.fwd_workspace_size(B, H, N, d) > 0      # these shapes leave a partial last wave
    q, k, v, _ = make_inputs(B, H, N, d, "bf16", "normal", 31 + N + d, device="cuda")
    o_split, l_split = fa.fwd(q, k, v)
    o_whole, l_whole = fa.fwd(q, k, v, workspace=False)
    assert fa.sync_status() == 0
    assert float((o_split.float() - o_whole.float()).abs().max()) <= 1e-2
    assert float((l_split - l_whole).abs().max()) <= 1e-4
    import oracle

    for b in range(B):
        for h in range(H):
            ref_o, ref_l = oracle.attention_forward_head(to64(q[b, h]), to64(k[b, h]), to64(v[b, h]), d ** -0.5)
            assert np.max(np.abs(to64(o_split[b, h]) - ref_o)) <= 1e-2
            assert np.max(np.abs(to64(l_split[b, h]) - ref_l)) <= 1e-3


@pytest.mark.parametrize("B,H,N,d", [(8, 32, 1000, 64), (4, 40, 2048, 128), (2, 96, 777, 96), (1, 200, 256, 128)])
def test_bf16_persistent_forward(B, H, N, d):
    """More two-tile units than SMs and at most 16 K/V tiles each, without
    the mask: the forward runs as one persistent CTA per SM walking the
    units (ragged N, d = 64, 96, 128; units of 2 to 16 K/V tiles).  Forward
    and backward of the first and last heads against the oracle."""
    q, k, v, do = make_inputs(B, H, N, d, "bf16", "normal", 50 + N + d, device="cuda")
    scale = d ** -0.5
    gpu = run_library(q, k, v, do, False, scale)
    heads = [(0, 0), (B - 1, H - 1)]
    ref = run_oracle_heads(q, k, v, do, False, scale, heads)
    compare({key: np.stack([val[b, h] for b, h in heads]) for key, val in gpu.items()}, ref, "bf16")


@pytest.mark.parametrize("dtype,B,H,N", [("bf16", 1, 200, 128), ("bf16", 2, 96, 256), ("bf16", 8, 24, 1024),
                                          ("bf16", 3, 40, 700), ("fp16", 2, 64, 384)])
def test_persistent_backward_d64(dtype, B, H, N):
    """d = 64 without the mask, more K/V tiles than SMs and at most 8 query
    tiles per head: the backward runs as one persistent CTA per SM walking
    the K/V tiles (1, 2, 8 and ragged query tiles per unit; fp16 too).
    First and last heads against the oracle, every head for inf/NaN and the
    gradient invariants."""
    q, k, v, do = make_inputs(B, H, N, 64, dtype, "normal", 60 + N + H, device="cuda")
    scale = 64 ** -0.5
    gpu = run_library(q, k, v, do, False, scale)
    for key in ("O", "LSE", "dQ", "dK", "dV"):
        assert np.all(np.isfinite(gpu[key])), key
    dk, dv, dov = gpu["dK"], gpu["dV"], to64(do)
    assert np.linalg.norm(dk.sum(axis=2)) <= 2e-2 * np.linalg.norm(dk)
    assert np.linalg.norm(dv.sum(axis=2) - dov.sum(axis=2)) <= 2e-2 * np.linalg.norm(dv)
    heads = [(0, 0), (B - 1, H - 1)]
    ref = run_oracle_heads(q, k, v, do, False, scale, heads)
    compare({key: np.stack([val[b, h] for b, h in heads]) for key, val in gpu.items()}, ref, "bf16")


def test_bf16_stress_small():
    """Scores scaled to magnitudes in the hundreds (Q, K drawn ×8, d = 64)."""
    errs = _check(2, 2, 512, 64, False, "bf16", dist="stress", seed=5)
    assert errs["O"] <= 1e-2


@pytest.mark.parametrize("causal", [False, True])
def test_bf16_stress_ragged(causal):
    """Large scores with a ragged last tile: the zero-filled keys past N score
    0, far above rows whose scores are all very negative; they must neither
    enter the softmax nor turn dQ into inf · 0."""
    _check(2, 1, 300, 64, causal, "bf16", dist="stress", seed=6)


@pytest.mark.parametrize("dtype,d,scale", [(dt, d, sc) for dt, d in (("bf16", 64), ("bf16", 128)) for sc in (1e-3, 0.3, 1.0)]
                         + [("fp32", 64, 1e-3), ("fp32", 64, 0.3)])
@pytest.mark.parametrize("causal", [False, True])
def test_scales(dtype, d, scale, causal):
    """Scales other than 1/sqrt(d) (the softmax of the scaled scores, "Flash
    Attention" tutorial 1.FlashAttention 整体结构 一): nearly uniform rows
    (10⁻³) up to sharp ones (1.0: scores with a standard deviation of 8-11,
    so a row's weight sits on a few keys).

    The O bound for bf16 is derived, not the workloads' 1e-2: P is rounded to
    bf16 (8 significant bits, relative error ≤ 2⁻⁸) before P V while ℓ sums
    the unrounded values, so the weights on V are off by at most 2⁻⁸ in all,
    and O itself is stored in bf16; hence |O − O_ref| ≤ 2⁻⁸·(max|V| + |O_ref|)
    (+10⁻³ for the fp32 sums).  A sharp row puts O near a single V_j, where
    these roundings no longer average out: at scale 1.0 they reach ~0.017
    for |V_j| ≈ 4.  LSE, the gradients (relative Frobenius) and fp32 keep the
    workloads' tolerances; fp32 stays at scores of the default's size, its
    1e-5 bar being absolute."""
    q, k, v, do = make_inputs(1, 2, 384, d, dtype, "normal", 40 + d + int(causal), device="cuda")
    gpu = run_library(q, k, v, do, causal, scale)
    ref = run_oracle_heads(q, k, v, do, causal, scale, _all_heads(1, 2))
    flat = {key: val.reshape((-1,) + val.shape[2:]) for key, val in gpu.items()}
    if dtype == "fp32":
        compare(flat, ref, dtype)
        return
    for key in ("O", "LSE", "dQ", "dK", "dV"):
        assert np.all(np.isfinite(flat[key])), key
    vmax = np.abs(to64(v).reshape(2, -1)).max(axis=1).reshape(2, 1, 1)
    bound = 2.0 ** -8 * (vmax + np.abs(ref["O"])) + 1e-3
    assert np.all(np.abs(flat["O"] - ref["O"]) <= bound), float(np.max(np.abs(flat["O"] - ref["O"]) - bound))
    assert np.max(np.abs(flat["LSE"] - ref["LSE"])) <= BF16_LSE_ATOL
    for key in ("dQ", "dK", "dV"):
        assert rel_fro(flat[key], ref[key]) <= BF16_GRAD_RTOL_FRO, (key, rel_fro(flat[key], ref[key]))


# ------------------------------------------------------------------ closed forms on the GPU


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_bf16_constant_v(d, causal):
    """Rows of P sum to one: V_j = c gives O_i = c to within one bf16 ulp of |c|."""
    import exact_tiled_attention_12_gb300 as fa

    q, k, _, _ = make_inputs(1, 2, 512, d, "bf16", "normal", 11, device="cuda")
    c = torch.linspace(-3, 3, d, dtype=torch.float32).to(torch.bfloat16)
    v = c.view(1, 1, 1, d).expand(1, 2, 512, d).contiguous().cuda()
    o, _ = fa.fwd(q, k, v, causal=causal)
    cf = c.double().abs()
    ulp = torch.where(cf > 0, torch.exp2(torch.floor(torch.log2(cf.clamp_min(1e-30))) - 7), torch.zeros_like(cf))
    err = (o.double().cpu() - c.double().view(1, 1, 1, d)).abs()
    assert bool((err <= ulp.view(1, 1, 1, d) + 1e-12).all()), float(err.max())


@pytest.mark.parametrize("causal", [False, True])
def test_bf16_identical_keys(causal):
    """K_j = k for all j: P is uniform over visible keys, O_i = mean of visible V_j."""
    import exact_tiled_attention_12_gb300 as fa

    q, _, v, _ = make_inputs(1, 1, 384, 128, "bf16", "normal", 12, device="cuda")
    k = make_inputs(1, 1, 1, 128, "bf16", "normal", 13, device="cuda")[0].expand(1, 1, 384, 128).contiguous()
    o, lse = fa.fwd(q, k, v, causal=causal)
    vv = to64(v[0, 0])
    want = np.cumsum(vv, axis=0) / np.arange(1, 385)[:, None] if causal else np.tile(vv.mean(axis=0), (384, 1))
    assert np.max(np.abs(to64(o[0, 0]) - want)) <= 1e-2


def test_bf16_gradient_invariants():
    """Σ_j dK_j = 0 and Σ_j dV_j = Σ_i dO_i, relative to the gradients' size."""
    q, k, v, do = make_inputs(2, 2, 512, 128, "bf16", "normal", 14, device="cuda")
    for causal in (False, True):
        g = run_library(q, k, v, do, causal)
        for b in range(2):
            for h in range(2):
                dk, dv, dov = g["dK"][b, h], g["dV"][b, h], to64(do[b, h])
                assert np.linalg.norm(dk.sum(axis=0)) <= 2e-2 * np.linalg.norm(dk)
                assert np.linalg.norm(dv.sum(axis=0) - dov.sum(axis=0)) <= 2e-2 * np.linalg.norm(dv)


# ------------------------------------------------------------------ API behaviour


def test_bf16_forward_and_dkdv_are_deterministic():
    import exact_tiled_attention_12_gb300 as fa

    q, k, v, do = make_inputs(1, 2, 512, 128, "bf16", "normal", 15, device="cuda")
    o1, l1 = fa.fwd(q, k, v)
    o2, l2 = fa.fwd(q, k, v)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    g1 = fa.bwd(q, k, v, o1, do, l1)
    g2 = fa.bwd(q, k, v, o1, do, l1)
    assert torch.equal(g1[1], g2[1]) and torch.equal(g1[2], g2[2])
    assert float((g1[0].float() - g2[0].float()).abs().max()) <= 1e-2


def test_stage_api_matches_fa_bwd():
    import exact_tiled_attention_12_gb300 as fa

    q, k, v, do = make_inputs(1, 2, 512, 64, "bf16", "normal", 16, device="cuda")
    o, lse = fa.fwd(q, k, v, causal=True)
    dq, dk, dv = fa.bwd(q, k, v, o, do, lse, causal=True)
    ws = torch.empty(fa.bwd_workspace_size(1, 2, 512, 64), dtype=torch.uint8, device="cuda")
    dq2, dk2, dv2 = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    fa.bwd_stages(q, k, v, o, do, lse, dq2, dk2, dv2, ws, causal=True)
    assert fa.sync_status() == 0
    assert torch.equal(dk, dk2) and torch.equal(dv, dv2)
    assert float((dq.float() - dq2.float()).abs().max()) <= 1e-2


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_empty_problems(dtype):
    import exact_tiled_attention_12_gb300 as fa

    for shape in [(1, 1, 0, 64), (0, 2, 128, 64), (1, 0, 128, 64)]:
        q, k, v, do = make_inputs(*shape, dtype, "normal", 1, device="cuda")
        o, lse = fa.fwd(q, k, v)
        dq, dk, dv = fa.bwd(q, k, v, o, do, lse)
        assert o.shape == q.shape and lse.shape == shape[:3] and dq.shape == q.shape
    assert fa.sync_status() == 0


def test_unsupported_shapes_raise():
    import exact_tiled_attention_12_gb300 as fa

    for shape in [(1, 1, 256, 80), (1, 1, 200, 32)]:
        q, k, v, _ = make_inputs(*shape, "bf16", "normal", 1, device="cuda")
        with pytest.raises(fa.FaError) as e:
            fa.fwd(q, k, v)
        assert e.value.code == 2


@pytest.mark.parametrize("dtype,causal", [("bf16", False), ("bf16", True), ("fp32", True)])
def test_autograd_attention_matches_oracle(dtype, causal):
    """attention() under torch.autograd: O from forward, dQ/dK/dV from .backward()."""
    import exact_tiled_attention_12_gb300 as fa

    B, H, N, d = 1, 2, 256, 64
    q, k, v, do = make_inputs(B, H, N, d, dtype, "normal", 41, device="cuda")
    q, k, v = (t.clone().requires_grad_(True) for t in (q, k, v))
    o = fa.attention(q, k, v, causal=causal)
    o.backward(do)
    ref = run_oracle_heads(q.detach(), k.detach(), v.detach(), do, causal, d ** -0.5, [(0, 0), (0, 1)])
    gpu = {"O": to64(o.detach()[0]), "LSE": ref["LSE"], "dQ": to64(q.grad[0]), "dK": to64(k.grad[0]),
           "dV": to64(v.grad[0])}
    compare(gpu, ref, dtype)


# ------------------------------------------------------------------ the square entry points, called directly

_DT = {"bf16": 0, "fp32": 1, "fp16": 2}


@pytest.mark.parametrize("dtype,B,H,N,d,causal", [
    ("bf16", 1, 2, 512, 128, False),
    ("bf16", 2, 1, 384, 64, True),
    ("bf16", 1, 2, 300, 128, True),     # ragged N through the square symbols
    ("fp16", 1, 1, 256, 128, False),
    ("fp32", 1, 2, 96, 64, True),
])
def test_square_entry_points_fa_fwd_fa_bwd(dtype, B, H, N, d, causal):
    """fa_fwd and fa_bwd (the square C-ABI symbols, not the Nq/Nk ones the
    binding uses) called through ctypes with caller-owned outputs and
    workspaces, compared with the oracle on every head."""
    import ctypes

    import exact_tiled_attention_12_gb300 as fa

    L = fa.lib()
    q, k, v, do = make_inputs(B, H, N, d, dtype, "normal", 70 + N, device="cuda")
    scale = d ** -0.5
    code = _DT[dtype]
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    sp = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    fws_n = L.fa_fwd_workspace_size(B, H, N, d, int(causal), code)
    fws = torch.empty(max(fws_n, 1), dtype=torch.uint8, device="cuda")
    st = L.fa_fwd(P(q), P(k), P(v), P(o), P(lse), B, H, N, d, scale, int(causal), code,
                  P(fws) if fws_n else None, fws_n, sp)
    assert st == 0, fa.status_string(st)
    bws_n = L.fa_bwd_workspace_size(B, H, N, d, code)
    bws = torch.empty(max(bws_n, 1), dtype=torch.uint8, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    st = L.fa_bwd(P(q), P(k), P(v), P(o), P(do), P(lse), P(dq), P(dk), P(dv), B, H, N, d, scale, int(causal), code,
                  P(bws), bws_n, sp)
    assert st == 0, fa.status_string(st)
    assert L.fa_sync_status(sp) == 0
    gpu = {"O": to64(o), "LSE": to64(lse), "dQ": to64(dq), "dK": to64(dk), "dV": to64(dv)}
    heads = _all_heads(B, H)
    ref = run_oracle_heads(q, k, v, do, causal, scale, heads)
    flat = {key: val.reshape((-1,) + val.shape[2:]) for key, val in gpu.items()}
    compare(flat, ref, "fp32" if dtype == "fp32" else "bf16")
