"""torch.autograd integration: ``attention(q, k, v, scale=None, causal=False)``.

Forward saves only what the backward of the "Flash Attention" tutorial's
3.Recomputation needs — q, k, v, O and the per-row LSE — and the backward
calls the library's tiled backward, which recomputes P tile by tile.  Both
directions run in libfa.so; this module only wires them into autograd.
Gradients are returned for q, k and v (in their dtype); scale and causal are
not differentiable.
"""

from __future__ import annotations

import torch

from . import binding


class _Attention(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, scale, causal):
        q, k, v = (t.contiguous() for t in (q, k, v))
        o, lse = binding.fwd(q, k, v, scale=scale, causal=causal)
        ctx.save_for_backward(q, k, v, o, lse)
        ctx.scale = scale
        ctx.causal = causal
        return o

    @staticmethod
    def backward(ctx, do):
        q, k, v, o, lse = ctx.saved_tensors
        dq, dk, dv = binding.bwd(q, k, v, o, do.contiguous(), lse, scale=ctx.scale, causal=ctx.causal)
        return dq, dk, dv, None, None


def attention(q, k, v, scale=None, causal=False):
    """softmax(scale · Q Kᵀ) V, differentiable: q [B, H, Nq, d], k and v
    [B, H, Nk, d] CUDA tensors (bf16, fp16 or fp32).  Under ``causal`` the queries
    are the last Nq positions (query i sees keys j <= i + Nk - Nq)."""
    return _Attention.apply(q, k, v, scale, causal)
