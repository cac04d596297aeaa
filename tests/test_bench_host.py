"""The bench's host-side bookkeeping, without a GPU: the per-configuration
summary (rates, fractions, the dominant kernel), the oracle's forward and
backward timing on a bounded row block, and the nvidia-smi fallback's
parsing of clock samples and throttle reasons."""

import math

import pytest


def test_summarise_rates_and_fractions():
    import bench
    from exact_tiled_attention_12_gb300.synthetic import WORKLOADS

    w = WORKLOADS["bf16_n8192"]
    t = {"steps": 4, "wall_s": 0.01, "clocks": {"sm_mhz": 2070.0, "samples": 5},
         "fwd": [0.43] * 4, "bwd": [1.23] * 4, "tiles": [1.19] * 4, "step": [1.66] * 4}
    s = bench.summarise(w, t, 1918.6)
    assert math.isclose(s["fwd"]["tflops"], w.flops_fwd() / 0.43e-3 / 1e12, rel_tol=1e-3)
    assert math.isclose(s["bwd"]["frac_of_peak"], w.flops_bwd() / 1.23e-3 / 1e12 / 1918.6, rel_tol=1e-3)
    assert math.isclose(s["dominant_kernel"]["tflops"], w.flops_bwd() / 1.19e-3 / 1e12, rel_tol=1e-3)
    assert s["dominant_kernel"]["name"].startswith("fa_bwd_bf16_kernel<d=128")
    assert math.isclose(s["step_tflops"], (w.flops_fwd() + w.flops_bwd()) / 1.66e-3 / 1e12, rel_tol=1e-3)
    assert s["clocks"]["samples"] == 5


@pytest.mark.parametrize("name", ["tiny_fp32", "bf16_causal_n4096"])
def test_oracle_timing_legs(name):
    """Forward and backward are timed separately on the same row block, with
    FLOPs counted per visible (query, key) pair as on the GPU."""
    import bench
    from exact_tiled_attention_12_gb300.synthetic import WORKLOADS, make_workload_inputs

    w = WORKLOADS[name]
    q, k, v, do = make_workload_inputs(w, device="cpu", heads=1)
    arrays = [t[0, 0].double().numpy() for t in (q, k, v, do)]
    r = bench.cpu_baseline_split(w, arrays, budget_s=0.3)
    assert r["kind"] == "oracle" and r["cores"] >= 1
    for leg in ("fwd", "bwd"):
        assert r[leg]["tflops"] > 0 and r[leg]["seconds"] > 0 and r[leg]["reps"] >= 1
    rows = list(range(w.N - 5, w.N))
    pairs = bench._visible_pairs(w, rows)
    assert pairs == (sum(i + 1 for i in rows) if w.causal else 5 * w.N)
    assert bench._rows_flops(w, rows) == 14.0 * pairs * w.d


def test_smi_fallback_parses_reasons():
    import os
    import types

    import bench

    sampler = bench.SmiClockSampler(types.SimpleNamespace(index=0))   # only the sample file, no nvidia-smi
    with open(sampler.path, "w") as f:
        f.write("2026/12/02 10:00:00.000, 0, 2070, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Not Active\n")
        f.write("2026/12/02 10:00:00.100, 0, 1980, 2070, 1400.0, 0x4, Not Active, Not Active, Not Active, Active\n")
        f.write("garbage line\n")
    out = sampler._summary()
    os.unlink(sampler.path)
    assert out["samples"] == 2 and out["sm_max_mhz"] == 2070.0
    assert out["sm_mhz"] == (2070 + 1980) / 2
    assert out["reasons"] == ["sw_power_cap"]


def test_dominant_kernel_names_the_persistent_backward():
    """The d = 64 unmasked stress workload (8 query tiles a head, 1024 K/V
    tiles) runs the persistent backward on a 152-SM GPU; with more SMs than
    K/V tiles, or at d = 128, the one-tile-per-CTA kernel."""
    import bench
    from exact_tiled_attention_12_gb300.synthetic import WORKLOADS

    assert bench.dominant_kernel(WORKLOADS["bf16_stress_n1024"], 152).startswith("fa_bwd_bf16_persist64_kernel")
    assert bench.dominant_kernel(WORKLOADS["bf16_stress_n1024"], 2048).startswith("fa_bwd_bf16_kernel<d=64")
    assert bench.dominant_kernel(WORKLOADS["bf16_n2048"], 152).startswith("fa_bwd_bf16_kernel<d=128")
