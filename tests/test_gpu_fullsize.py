"""Parity at the full sizes of every bf16 workload, in the launch configuration
the bench times.

The whole workload runs on the GPU; the fp64 oracle then recomputes sampled
heads completely (every row of O and LSE, and all of dQ, dK, dV for those
heads), and every head is checked for inf/NaN and for the gradient
invariants Σ_j dK_j = 0 and Σ_j dV_j = Σ_i dO_i.
"""

import numpy as np
import pytest
import torch

from exact_tiled_attention_12_gb300.synthetic import WORKLOADS, make_workload_inputs

from ._helpers import compare, run_oracle_heads, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()


@pytest.mark.parametrize("name", [n for n, w in WORKLOADS.items() if w.dtype == "bf16"])
def test_fullsize_workload(name):
    import exact_tiled_attention_12_gb300 as fa

    w = WORKLOADS[name]
    q, k, v, do = make_workload_inputs(w, device="cuda")
    o, lse = fa.fwd(q, k, v, scale=w.scale, causal=w.causal)
    dq, dk, dv = fa.bwd(q, k, v, o, do, lse, scale=w.scale, causal=w.causal)
    assert fa.sync_status() == 0
    for t in (o, lse, dq, dk, dv):
        assert bool(torch.isfinite(t).all())
    # invariants on every head, computed on the GPU in fp32
    dks = dk.float().sum(dim=2)
    assert float(dks.norm()) <= 2e-2 * float(dk.float().norm())
    dvs = dv.float().sum(dim=2) - do.float().sum(dim=2)
    assert float(dvs.norm()) <= 2e-2 * float(dv.float().norm())
    # sampled heads, recomputed in full by the oracle
    heads = [(0, 0), (w.B - 1, w.H - 1)]
    ref = run_oracle_heads(q, k, v, do, w.causal, w.scale, heads)
    gpu = {key: np.stack([to64(t[b, h]) for b, h in heads]) for key, t in
           (("O", o), ("LSE", lse), ("dQ", dq), ("dK", dk), ("dV", dv))}
    compare(gpu, ref, "bf16")
