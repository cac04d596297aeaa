"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module only draws random numbers.  It holds none of the attention
arithmetic, so both the CUDA path and the fp64 oracle can take their inputs
from it without sharing any of the method.

Recipe: a CPU ``torch.Generator`` seeded with ``seed`` draws Q, K, V, dO in
that order as float32, then each is rounded to the working dtype (bf16 with
round-to-nearest-even, fp16 likewise, or kept fp32).  Both sides read the same rounded bits;
bf16 -> fp64 is exact, so the oracle sees exactly what the kernels see.

Distributions:
  * ``normal``: Q, K, V, dO iid N(0, 1);
  * ``stress``: Q, K iid 8·N(0, 1) (a power-of-two factor, exact in bf16, so
    scaled scores reach magnitudes of a few hundred), V iid U(-1, 1)
    (``2·rand - 1``), dO iid N(0, 1).
"""

from __future__ import annotations

from dataclasses import dataclass

import torch

BASE_SEED = 20261202


@dataclass(frozen=True)
class Workload:
    """One named attention workload: shape, mask, dtype and input distribution."""

    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool
    dtype: str          # "bf16" or "fp32"
    dist: str           # "normal" or "stress"
    seed: int

    @property
    def scale(self) -> float:
        return self.d ** -0.5

    def flops_fwd(self) -> float:
        """4·N²·d per head (two N×N×d products); half of it under the causal mask."""
        f = 4.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2 if self.causal else f

    def flops_bwd(self) -> float:
        """10·N²·d per head (four products plus the recomputed S); half if causal."""
        f = 10.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2 if self.causal else f

    def describe(self) -> str:
        return (f"B={self.B},H={self.H},N={self.N},d={self.d},"
                f"{'causal' if self.causal else 'non-causal'},{self.dtype},{self.dist}")


# The workloads the library is measured and checked on.  Shapes follow the
# pages' workloads: a tiny fp32 case with the cnnetsun.cn self-test's shape
# (1 x 256 x 64, scale 64^-0.5), 32 heads of width 128 as in a 7B decoder
# layer, a long 8192-token sequence, and a d=64 stress case with large scores.
WORKLOADS = {
    "tiny_fp32": Workload("tiny_fp32", 1, 1, 256, 64, False, "fp32", "normal", BASE_SEED + 1),
    "bf16_n2048": Workload("bf16_n2048", 4, 32, 2048, 128, False, "bf16", "normal", BASE_SEED + 2),
    "bf16_causal_n4096": Workload("bf16_causal_n4096", 2, 32, 4096, 128, True, "bf16", "normal", BASE_SEED + 3),
    "bf16_n8192": Workload("bf16_n8192", 1, 16, 8192, 128, False, "bf16", "normal", BASE_SEED + 4),
    "bf16_causal_n8192": Workload("bf16_causal_n8192", 1, 16, 8192, 128, True, "bf16", "normal", BASE_SEED + 4),
    "bf16_stress_n1024": Workload("bf16_stress_n1024", 8, 16, 1024, 64, False, "bf16", "stress", BASE_SEED + 5),
}


def torch_dtype(name: str) -> torch.dtype:
    return {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}[name]


def make_inputs(B, H, N, d, dtype="bf16", dist="normal", seed=BASE_SEED, device="cpu"):
    """Draw (q, k, v, do) of shape [B, H, N, d] on the CPU, then move to ``device``."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    shape = (B, H, N, d)
    if dist == "normal":
        q = torch.randn(shape, generator=g, dtype=torch.float32)
        k = torch.randn(shape, generator=g, dtype=torch.float32)
        v = torch.randn(shape, generator=g, dtype=torch.float32)
    elif dist == "stress":
        q = torch.randn(shape, generator=g, dtype=torch.float32) * 8.0
        k = torch.randn(shape, generator=g, dtype=torch.float32) * 8.0
        v = torch.rand(shape, generator=g, dtype=torch.float32) * 2.0 - 1.0
    else:
        raise ValueError(f"unknown distribution {dist!r}")
    do = torch.randn(shape, generator=g, dtype=torch.float32)
    td = torch_dtype(dtype)
    out = [t.to(td).contiguous() for t in (q, k, v, do)]
    if device != "cpu":
        out = [t.to(device) for t in out]
    return tuple(out)


def make_inputs_kv(B, H, Nq, Nk, d, dtype="bf16", dist="normal", seed=BASE_SEED, device="cpu"):
    """Draw q [B, H, Nq, d], k and v [B, H, Nk, d], do [B, H, Nq, d] (in that
    order, same distributions and rounding as ``make_inputs``)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    qs, ks = (B, H, Nq, d), (B, H, Nk, d)
    if dist == "normal":
        q = torch.randn(qs, generator=g, dtype=torch.float32)
        k = torch.randn(ks, generator=g, dtype=torch.float32)
        v = torch.randn(ks, generator=g, dtype=torch.float32)
    elif dist == "stress":
        q = torch.randn(qs, generator=g, dtype=torch.float32) * 8.0
        k = torch.randn(ks, generator=g, dtype=torch.float32) * 8.0
        v = torch.rand(ks, generator=g, dtype=torch.float32) * 2.0 - 1.0
    else:
        raise ValueError(f"unknown distribution {dist!r}")
    do = torch.randn(qs, generator=g, dtype=torch.float32)
    td = torch_dtype(dtype)
    out = [t.to(td).contiguous() for t in (q, k, v, do)]
    if device != "cpu":
        out = [t.to(device) for t in out]
    return tuple(out)


def make_workload_inputs(w: Workload, device="cpu", heads=None):
    """Inputs of a named workload; ``heads`` optionally overrides H (same seed)."""
    return make_inputs(w.B, w.H if heads is None else heads, w.N, w.d, w.dtype, w.dist, w.seed, device)
