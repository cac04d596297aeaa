"""Layer-level check of attention() inside a small multi-head attention layer.

x [B, N, C] -> Q, K, V projections -> H heads of width d -> attention ->
output projection -> a scalar loss.  The weight gradients that autograd gets
through the library are compared with the same layer run on the CPU in fp64
with the oracle's forward and backward in place of the library.  A second
test wraps the layer in torch.utils.checkpoint (the forward is recomputed in
the backward, as in activation checkpointing) and expects the same
gradients.  Both run with the fp32 dtype (SIMT kernels) and with the bf16
tensor-core path (q, k, v cast to bf16 for attention, the rest of the layer
in fp32: mixed precision as a training step would use it).
"""

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()


class _OracleAttention(torch.autograd.Function):
    """The oracle's forward and backward as an autograd op (CPU, fp64)."""

    @staticmethod
    def forward(ctx, q, k, v, causal):
        import oracle

        scale = q.shape[-1] ** -0.5
        o, _ = oracle.attention_forward(q.numpy(), k.numpy(), v.numpy(), scale, causal)
        ctx.save_for_backward(q, k, v)
        ctx.causal = causal
        return torch.from_numpy(o)

    @staticmethod
    def backward(ctx, do):
        import oracle

        q, k, v = ctx.saved_tensors
        scale = q.shape[-1] ** -0.5
        dq, dk, dv = oracle.attention_backward(q.numpy(), k.numpy(), v.numpy(), do.numpy(), scale, ctx.causal)
        return torch.from_numpy(dq), torch.from_numpy(dk), torch.from_numpy(dv), None


def _layer(x, w, H, attn, causal):
    B, N, C = x.shape
    d = C // H

    def heads(t):
        return t.view(B, N, H, d).transpose(1, 2).contiguous()

    q, k, v = heads(x @ w["q"]), heads(x @ w["k"]), heads(x @ w["v"])
    o = attn(q, k, v, causal)
    y = o.transpose(1, 2).reshape(B, N, C) @ w["o"]
    return (y * y).mean()


def _weights(C, seed, device, dtype):
    g = torch.Generator().manual_seed(seed)
    return {n: (torch.randn((C, C), generator=g) * C ** -0.5).to(device=device, dtype=dtype).requires_grad_(True)
            for n in ("q", "k", "v", "o")}


@pytest.mark.parametrize("causal", [False, True])
def test_layer_gradients_match_oracle_layer(causal):
    import exact_tiled_attention_12_gb300 as fa

    B, N, H, d = 2, 300, 4, 32
    C = H * d
    g = torch.Generator().manual_seed(11)
    x = torch.randn((B, N, C), generator=g)
    w_gpu = _weights(C, 12, "cuda", torch.float32)
    loss = _layer(x.cuda(), w_gpu, H, lambda q, k, v, c: fa.attention(q, k, v, causal=c), causal)
    loss.backward()
    w_ref = _weights(C, 12, "cpu", torch.float64)
    loss_ref = _layer(x.double(), w_ref, H, lambda q, k, v, c: _OracleAttention.apply(q, k, v, c), causal)
    loss_ref.backward()
    assert abs(loss.item() - loss_ref.item()) <= 1e-5 * abs(loss_ref.item())
    for n in w_gpu:
        a, b = w_gpu[n].grad.double().cpu().numpy(), w_ref[n].grad.numpy()
        assert np.linalg.norm(a - b) <= 1e-4 * np.linalg.norm(b), n


def test_layer_under_activation_checkpointing():
    import torch.utils.checkpoint as cp

    import exact_tiled_attention_12_gb300 as fa

    B, N, H, d = 1, 256, 2, 64
    C = H * d
    g = torch.Generator().manual_seed(13)
    x = torch.randn((B, N, C), generator=g).cuda()
    grads = []
    for use_cp in (False, True):
        w = _weights(C, 14, "cuda", torch.float32)

        def run(xx):
            return _layer(xx, w, H, lambda q, k, v, c: fa.attention(q, k, v, causal=c), True)

        loss = cp.checkpoint(run, x, use_reentrant=False) if use_cp else run(x)
        loss.backward()
        grads.append({n: t.grad.clone() for n, t in w.items()})
    for n in grads[0]:
        assert torch.allclose(grads[0][n], grads[1][n], rtol=0, atol=1e-6), n


# ------------------------------------------------------------------ bf16 tensor-core path inside the layer
#
# Tolerances, derived: the attention's own bf16 bounds are O max abs 1e-2 and
# dQ, dK, dV relative Frobenius 2e-2 against the oracle on the same inputs.
# The layer adds four bf16 roundings around the attention (q, k, v in; O and
# the gradient of O out), each at most 2^-9 relative, which moves a weight
# gradient by well under 1e-2 relative.  So the weight gradients must agree
# with the fp64 oracle layer within 3e-2 relative Frobenius and the loss
# within 1e-2 relative.


def _bf16_attention(fa):
    def attn(q, k, v, causal):
        return fa.attention(q.bfloat16(), k.bfloat16(), v.bfloat16(), causal=causal).float()

    return attn


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_layer_gradients_match_oracle_layer_bf16(causal, d):
    import exact_tiled_attention_12_gb300 as fa

    B, N, H = 2, 300, 2
    C = H * d
    g = torch.Generator().manual_seed(15 + d)
    x = torch.randn((B, N, C), generator=g)
    w_gpu = _weights(C, 16, "cuda", torch.float32)
    loss = _layer(x.cuda(), w_gpu, H, _bf16_attention(fa), causal)
    loss.backward()
    w_ref = _weights(C, 16, "cpu", torch.float64)
    loss_ref = _layer(x.double(), w_ref, H, lambda q, k, v, c: _OracleAttention.apply(q, k, v, c), causal)
    loss_ref.backward()
    assert abs(loss.item() - loss_ref.item()) <= 1e-2 * abs(loss_ref.item())
    for n in w_gpu:
        a, b = w_gpu[n].grad.double().cpu().numpy(), w_ref[n].grad.numpy()
        assert np.all(np.isfinite(a)), n
        assert np.linalg.norm(a - b) <= 3e-2 * np.linalg.norm(b), (n, np.linalg.norm(a - b) / np.linalg.norm(b))


def test_layer_under_activation_checkpointing_bf16():
    """Recomputing the bf16 forward inside the backward gives the same weight
    gradients: O, LSE, dK and dV are reproducible bit for bit; dQ sums fp32
    partials in a varying order, which can move a bf16 rounding of dQ by one
    unit (2^-8 relative), so the gradients are compared within 5e-3 relative
    Frobenius."""
    import torch.utils.checkpoint as cp

    import exact_tiled_attention_12_gb300 as fa

    B, N, H, d = 1, 384, 2, 128
    C = H * d
    g = torch.Generator().manual_seed(17)
    x = torch.randn((B, N, C), generator=g).cuda()
    grads = []
    for use_cp in (False, True):
        w = _weights(C, 18, "cuda", torch.float32)

        def run(xx):
            return _layer(xx, w, H, _bf16_attention(fa), True)

        loss = cp.checkpoint(run, x, use_reentrant=False) if use_cp else run(x)
        loss.backward()
        grads.append({n: t.grad.clone() for n, t in w.items()})
    for n in grads[0]:
        a, b = grads[1][n], grads[0][n]
        assert float(torch.linalg.norm(a - b)) <= 5e-3 * float(torch.linalg.norm(b)), n
