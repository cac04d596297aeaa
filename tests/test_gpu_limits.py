"""The largest shapes the boundary accepts, run on the GPU.

The C ABI refuses more than 65,535 heads and more than 65,535 K/V tiles of
128 keys per head: the backward's grid puts heads (or, under the causal
mask, K/V tiles) in its second dimension.  These tests run exactly at those
limits: every head and every key range is launched, every output is checked
for inf/NaN and for the gradient invariants Σ_j dK_j = 0 and
Σ_j dV_j = Σ_i dO_i ("Flash Attention" tutorial, 4.附录A 反向传播的公式推导:
the rows of P sum to 1 and those of dS to 0), and sampled heads and rows
are recomputed by the fp64 oracle from the exact values the GPU saw.
"""

import numpy as np
import pytest
import torch

import oracle

from ._helpers import BF16_GRAD_RTOL_FRO, BF16_LSE_ATOL, BF16_O_ATOL, compare, rel_fro, run_oracle_heads, to64

pytestmark = pytest.mark.gpu

MAX_HEADS = 65535
MAX_KEYS = 65535 * 128


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()


def _invariants(dk, dv, do):
    dks = dk.float().sum(dim=2)
    assert float(dks.norm()) <= 2e-2 * float(dk.float().norm())
    dvs = dv.float().sum(dim=2) - do.float().sum(dim=2)
    assert float(dvs.norm()) <= 2e-2 * float(dv.float().norm())


def _many_heads(n_heads, n, d, seed):
    """[n_heads, 1, n, d] bf16 tensors built on the GPU from 11 drawn heads:
    Q and K repeat with period 11, V and dO also get a head-dependent offset
    (head mod 97, in steps of 2⁻⁶), so no two nearby heads are equal."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    base = [torch.randn((11, 1, n, d), generator=g, dtype=torch.float32).cuda() for _ in range(4)]
    heads = torch.arange(n_heads, device="cuda")
    shift = ((heads % 97).float() * 2.0 ** -6).view(n_heads, 1, 1, 1)
    out = []
    for i, t in enumerate(base):
        full = t[heads % 11]
        if i >= 2:
            full = full + shift
        out.append(full.to(torch.bfloat16).contiguous())
        del full
    torch.cuda.empty_cache()
    return out


@pytest.mark.parametrize("causal", [False, True])
def test_most_heads(causal):
    """65,535 heads (B = 65535, H = 1) of 128 queries and keys, d = 64."""
    import exact_tiled_attention_12_gb300 as fa

    q, k, v, do = _many_heads(MAX_HEADS, 128, 64, seed=71 + int(causal))
    scale = 64 ** -0.5
    o, lse = fa.fwd(q, k, v, causal=causal)
    dq, dk, dv = fa.bwd(q, k, v, o, do, lse, causal=causal)
    assert fa.sync_status() == 0
    for t in (o, lse, dq, dk, dv):
        assert bool(torch.isfinite(t).all())
    _invariants(dk, dv, do)
    heads = [(0, 0), (MAX_HEADS // 2, 0), (MAX_HEADS - 1, 0)]
    ref = run_oracle_heads(q, k, v, do, causal, scale, heads)
    gpu = {key: np.stack([to64(t[b, h]) for b, h in heads]) for key, t in
           (("O", o), ("LSE", lse), ("dQ", dq), ("dK", dk), ("dV", dv))}
    compare(gpu, ref, "bf16")
    del q, k, v, do, o, lse, dq, dk, dv
    torch.cuda.empty_cache()


def _host_bytes_available():
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 0


def _long_keys(nq, nk, d, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    q = torch.randn((1, 1, nq, d), generator=g, device="cuda").to(torch.bfloat16)
    k = torch.randn((1, 1, nk, d), generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn((1, 1, nk, d), generator=g, device="cuda").to(torch.bfloat16)
    do = torch.randn((1, 1, nq, d), generator=g, device="cuda").to(torch.bfloat16)
    return q, k, v, do


@pytest.mark.parametrize("nq,causal,d,nk", [(1, False, 64, MAX_KEYS), (300, False, 64, MAX_KEYS),
                                           (300, True, 64, MAX_KEYS), (300, True, 256, 65535 * 64)])
def test_most_keys(nq, causal, d, nk):
    """One head over 65,535 K/V tiles (8,388,480 keys), d = 64: the decoding
    step (one query), a ragged query block without the mask, and the same
    block as the last 300 positions under the causal mask; and d = 256 under
    the mask at its own limit, 65,535 tiles of 64 keys.  Forward rows and dQ
    rows are recomputed by the oracle; dK and dV are held to the invariants
    (their rows would need every query's softmax)."""
    import exact_tiled_attention_12_gb300 as fa

    # The oracle holds K, V and the backward's per-row dK, dV shares in fp64
    # on the host (4 × nk × d × 8 bytes): skip rather than exhaust the host.
    need = 4 * nk * d * 8
    if _host_bytes_available() < 3 * need:
        pytest.skip(f"needs about {need >> 30} GiB of free host memory for the oracle")
    scale = d ** -0.5
    q, k, v, do = _long_keys(nq, nk, d, seed=83 + nq + int(causal) + d)
    o, lse = fa.fwd(q, k, v, causal=causal)
    assert fa.sync_status() == 0
    assert bool(torch.isfinite(o).all()) and bool(torch.isfinite(lse).all())
    rows = [0, nq - 1] if nq > 1 else [0]
    qh, kh, vh = to64(q[0, 0]), to64(k[0, 0]), to64(v[0, 0])
    ref_o, ref_l = oracle.attention_forward_rows(qh, kh, vh, rows, scale, causal)
    assert np.max(np.abs(to64(o[0, 0])[rows] - ref_o)) <= BF16_O_ATOL
    assert np.max(np.abs(to64(lse[0, 0])[rows] - ref_l)) <= BF16_LSE_ATOL
    if nq > 1:
        dq, dk, dv = fa.bwd(q, k, v, o, do, lse, causal=causal)
        assert fa.sync_status() == 0
        for t in (dq, dk, dv):
            assert bool(torch.isfinite(t).all())
        _invariants(dk, dv, do)
        ref_dq, _, _ = oracle.attention_backward_rows(qh, kh, vh, to64(do[0, 0]), rows, scale, causal)
        assert rel_fro(to64(dq[0, 0])[rows], ref_dq) <= BF16_GRAD_RTOL_FRO
        del dq, dk, dv
    del q, k, v, do, o, lse, kh, vh
    torch.cuda.empty_cache()
