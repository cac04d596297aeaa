"""Benchmark: exact attention forward + backward TFLOP/s on one GB300.

One step = one pass of the whole hot path over one batch of synthetic input:
fa_fwd (O, LSE) then fa_bwd as its three stages (D pre-pass, tiled dQ/dK/dV
loop, dQ finish).  Inputs are resident in HBM before the timed region; L2 is
flushed (a 256 MiB write) before every timed step, outside the step's events.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--impl ours|reference] [--no-cpu-baseline]

Prints one JSON line (rank 0).  ``--impl reference`` times the fp64 CPU oracle
on this machine's host cores on a bounded sample of the same workload.
"""

from __future__ import annotations

import os

# The CPU oracle's BLAS threads: every core this process may run on.  Set
# before numpy is imported anywhere.
_CORES = len(os.sched_getaffinity(0))
for _var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_var, str(_CORES))

import argparse  # noqa: E402
import json  # noqa: E402
import statistics  # noqa: E402
import subprocess  # noqa: E402
import sys  # noqa: E402
import time  # noqa: E402

import torch  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from exact_tiled_attention_12_gb300.synthetic import WORKLOADS, make_workload_inputs  # noqa: E402

METRIC = "attention fwd/bwd TFLOPS (bf16, 1 GB300) and % of dense BF16 tensor peak"
DEFAULT_WORKLOAD = "bf16_n8192"          # B=1, H=16, N=8192, d=128: where the target is stated
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}


def measured_traffic(kernel, d, causal, workload):
    """DRAM bytes per launch recorded from an ncu capture in profiles/dram_traffic.txt,
    or None when there is none or the kernel's sources changed since it was taken."""
    import hashlib

    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    csrc = os.path.join(ROOT, "exact_tiled_attention_12_gb300", "csrc")
    src = {"fa_bwd_bf16_kernel": "fa_bwd_bf16.cu", "fa_fwd_bf16_kernel": "fa_fwd_bf16.cu"}[kernel]
    h = hashlib.sha256()
    for f in (src, "sm103_ptx.cuh", "fa_kernels.h"):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    digest = h.hexdigest()[:16]
    with open(path) as fh:
        for line in fh:
            parts = line.split()
            if len(parts) == 6 and not line.startswith("#"):
                if parts[0] == kernel and int(parts[1]) == d and int(parts[2]) == int(causal) and parts[3] == workload:
                    return int(parts[4]) if parts[5] == digest else None
    return None


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ clocks


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        self.path = os.path.join(ROOT, "gpurun_out", f"clocks_gpu{device_index}.csv")

    def start(self):
        os.makedirs(os.path.dirname(self.path), exist_ok=True)
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu=timestamp,{self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        self.t0 = time.time()

    def stop(self):
        self.t1 = time.time()
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    sm.append(float(parts[2]))
                    mx.append(float(parts[3]))
                except ValueError:
                    continue
                for name, val in zip(names, parts[6:10]):
                    if val.lower() in ("active", "0x1", "1"):
                        reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ ranks


def max_over_ranks(ms, device, world):
    """The slowest rank's timed region (every rank returns the same value)."""
    if world <= 1:
        return ms
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_step_per_rank, steps, slowest_ms, world):
    """Whole-job throughput: every rank runs its own batch (weak scaling), so
    the job does world × steps × flops in the slowest rank's time."""
    return world * flops_per_step_per_rank * steps / (slowest_ms * 1e-3) / 1e12


# ------------------------------------------------------------------ GPU arm


def run_ours(args, w, rank, world):
    import exact_tiled_attention_12_gb300 as fa
    from exact_tiled_attention_12_gb300.build import build

    build()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    peaks, peak_kind = load_peaks()
    q, k, v, do = make_workload_inputs(w, device=dev)
    B, H, N, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    ws = torch.empty(fa.bwd_workspace_size(B, H, N, d, q.dtype), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    L = fa.lib()
    stream = torch.cuda.current_stream(dev)
    import ctypes

    sp = ctypes.c_void_p(stream.cuda_stream)
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731

    fws_n = fa.fwd_workspace_size(B, H, N, d, w.causal, q.dtype)
    fws = torch.empty(max(fws_n, 1), dtype=torch.uint8, device=dev)

    def fwd():
        st = L.fa_fwd(P(q), P(k), P(v), P(o), P(lse), B, H, N, d, w.scale, int(w.causal), 0,
                      P(fws) if fws_n else None, fws_n, sp)
        assert st == 0, fa.status_string(st)

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]

    def step(i=None):
        if i is not None:
            ev[i][0].record(stream)
        fwd()
        if i is not None:
            ev[i][1].record(stream)
        fa.bwd_stages(q, k, v, o, do, lse, dq, dk, dv, ws, scale=w.scale, causal=w.causal,
                      between=None if i is None else (lambda: ev[i][2].record(stream), lambda: ev[i][3].record(stream)))
        if i is not None:
            ev[i][4].record(stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    assert fa.sync_status(dev) == 0
    clocks = ClockSampler(dev.index)
    clocks.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()
        step(i)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    status = fa.sync_status(dev)
    assert status == 0, fa.status_string(status)

    t_step = [ev[i][0].elapsed_time(ev[i][4]) for i in range(args.steps)]          # ms
    t_fwd = [ev[i][0].elapsed_time(ev[i][1]) for i in range(args.steps)]
    t_bwd = [ev[i][1].elapsed_time(ev[i][4]) for i in range(args.steps)]
    t_tiles = [ev[i][2].elapsed_time(ev[i][3]) for i in range(args.steps)]
    total_ms = sum(t_step)
    total_ms = max_over_ranks(total_ms, dev, world)
    ms_per_step = total_ms / args.steps
    flops_fwd, flops_bwd = w.flops_fwd(), w.flops_bwd()
    value = job_tflops(flops_fwd + flops_bwd, args.steps, total_ms, world)
    fwd_tflops = flops_fwd / (statistics.mean(t_fwd) * 1e-3) / 1e12
    bwd_tflops = flops_bwd / (statistics.mean(t_bwd) * 1e-3) / 1e12
    tiles_tflops = flops_bwd / (statistics.mean(t_tiles) * 1e-3) / 1e12
    peak = float(peaks["bf16_tflops"])
    peak_sus = float(peaks.get("bf16_tflops_sustained", peak))
    # Clock-derived dense bf16 rate: SMs × 8192 FLOP per SM clock (2·4096 MACs,
    # the nominal 2.25 PFLOP/s over SMs and boost clock) × the maximum SM clock.
    n_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    sm_max = float(peaks.get("sm_max_mhz", 2070.0))
    peak_theory = n_sms * 8192 * sm_max * 1e6 / 1e12

    # End to end through the public API: every step copies its inputs in from
    # pinned host memory and reads all of its results (O, LSE, dQ, dK, dV)
    # back.  Pipelined the way a caller would: two sets of device buffers, and
    # the uploads, the attention calls and the downloads on three streams, so
    # step i's compute overlaps step i+1's upload and step i-1's download.
    # The timed region runs from the first upload to the last download.
    # 30 steps (fewer if --steps is smaller): the first upload and the last
    # download, which nothing overlaps, then weigh 1/30 of the region.
    n_e2e = 0 if args.no_e2e else max(3, min(args.steps, 30))
    elem_bytes = q.numel() * q.element_size()
    e2e = None
    if n_e2e:
        hin = [tuple(t.to("cpu").pin_memory() for t in (q, k, v, do))]
        hin.append(tuple(t.clone().pin_memory() for t in hin[0]))
        hout = [tuple(torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (q, lse, q, k, v)) for _ in range(2)]
        dev_in = [(q, k, v, do), tuple(torch.empty_like(t) for t in (q, k, v, do))]
        ws2 = [ws, torch.empty_like(ws)]
        s_up, s_comp, s_down = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_in = [torch.cuda.Event() for _ in range(2)]       # inputs of set b uploaded
        ev_used = [torch.cuda.Event() for _ in range(2)]     # compute on set b done
        ev_read = [torch.cuda.Event() for _ in range(2)]     # results of set b downloaded
        outs = [None, None]

        def e2e_step(i):
            b = i % 2
            with torch.cuda.stream(s_up):
                s_up.wait_event(ev_used[b])                  # step i-2 has finished with these buffers
                for d_, h_ in zip(dev_in[b], hin[b]):
                    d_.copy_(h_, non_blocking=True)
                ev_in[b].record(s_up)
            with torch.cuda.stream(s_comp):
                s_comp.wait_event(ev_in[b])
                s_comp.wait_event(ev_read[b])                # step i-2's results are on the host
                qq, kk, vv, dd = dev_in[b]
                o_, lse_ = fa.fwd(qq, kk, vv, scale=w.scale, causal=w.causal)
                g = fa.bwd(qq, kk, vv, o_, dd, lse_, scale=w.scale, causal=w.causal, workspace=ws2[b])
                outs[b] = (o_, lse_) + tuple(g)
                ev_used[b].record(s_comp)
            with torch.cuda.stream(s_down):
                s_down.wait_event(ev_used[b])
                for h_, t_ in zip(hout[b], outs[b]):
                    h_.copy_(t_, non_blocking=True)
                    t_.record_stream(s_down)
                ev_read[b].record(s_down)

        for i in range(2):                                    # warm-up (both buffer sets)
            e2e_step(i)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s_up)
        for i in range(n_e2e):
            e2e_step(i)
        e1.record(s_down)
        torch.cuda.synchronize(dev)
        e2e_ms = e0.elapsed_time(e1) / n_e2e
        e2e = {"value": round(world * (flops_fwd + flops_bwd) / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
               "h2d_bytes_per_step": 4 * elem_bytes, "d2h_bytes_per_step": 4 * elem_bytes + lse.numel() * 4,
               "ms_per_step": round(e2e_ms, 3), "steps": n_e2e,
               "pipelining": "two buffer sets; uploads, compute and downloads on three streams"}

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{w.name}: {w.describe()}", "B": B, "H": H, "N": N, "d": d, "causal": w.causal,
                   "flops_per_step": flops_fwd + flops_bwd, "flop_convention": "fwd 4N^2d, bwd 10N^2d per head, causal /2",
                   "l2": "flushed before every timed step (256 MiB write, outside the step's events)",
                   "parallelism": f"replicas x{world}"},
        "fwd": {"tflops": round(fwd_tflops, 2), "ms": round(statistics.mean(t_fwd), 4),
                "ms_median": round(statistics.median(t_fwd), 4), "ms_min": round(min(t_fwd), 4),
                "ms_max": round(max(t_fwd), 4), "frac_of_peak": round(fwd_tflops / peak, 4)},
        "bwd": {"tflops": round(bwd_tflops, 2), "ms": round(statistics.mean(t_bwd), 4),
                "ms_median": round(statistics.median(t_bwd), 4), "ms_min": round(min(t_bwd), 4),
                "ms_max": round(max(t_bwd), 4), "frac_of_peak": round(bwd_tflops / peak, 4)},
        "roofline": {"bound": "tensor", "kernel": f"fa_bwd_bf16_kernel<d={d},causal={int(w.causal)}> (fa_bwd_tiles)",
                     "achieved": round(tiles_tflops, 2), "peak": peak, "peak_kind": f"{peak_kind} bf16 burst",
                     "unit": "TFLOP/s", "frac": round(tiles_tflops / peak, 4),
                     "frac_of_sustained": round(tiles_tflops / peak_sus, 4),
                     "peak_theoretical": round(peak_theory, 1),
                     "frac_of_theoretical": round(tiles_tflops / peak_theory, 4),
                     "peak_theoretical_note": f"{n_sms} SMs x 8192 FLOP/clk x {sm_max:.0f} MHz (clock-derived estimate)",
                     "ms_per_launch": round(statistics.mean(t_tiles), 4),
                     "algorithmic_flops_per_launch": flops_bwd,
                     "traffic": measured_traffic("fa_bwd_bf16_kernel", d, w.causal, w.name),
                     "traffic_unit": "bytes per launch (ncu dram read + write)"},
        "e2e": e2e,
        "softmax": {
            # exponentials of the forward (one per visible score) per SM clock at
            # the sampled median SM clock: the MUFU-side rate of the softmax
            "exp_per_clk_per_sm": (round(w.B * w.H * N * N / (2 if w.causal else 1)
                                         / (statistics.mean(t_fwd) * 1e-3) / (clk["sm_mhz"] * 1e6) / n_sms, 2)
                                   if clk.get("sm_mhz") else None),
        },
        # per step: forward (+ the split-merge kernel when the forward splits),
        # D pre-pass, tiled backward, dQ finish
        "gpu_launches": (3 + (2 if fws_n else 1)) * args.steps,
        "clocks": clk,
        "wall_s_timed": round(wall, 4),
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, q, k, v, do, budget_s=15.0)
    return line


# ------------------------------------------------------------------ CPU oracle


def _oracle_rows_step(w, qh, kh, vh, doh, rows):
    """fwd + bwd of the fp64 oracle restricted to a block of query rows."""
    import oracle

    oracle.attention_forward_rows(qh, kh, vh, rows, w.scale, w.causal)
    oracle.attention_backward_rows(qh, kh, vh, doh, rows, w.scale, w.causal)


def _rows_flops(w, rows):
    """Algorithmic FLOPs of the sampled rows under the bench's convention (per-row share)."""
    n_vis = sum((r + 1) if w.causal else w.N for r in rows)
    return 14.0 * n_vis * w.d


def _pick_rows(w, qh, kh, vh, doh, budget_s):
    """Largest contiguous block of query rows whose fwd+bwd fits the time budget."""
    import numpy as np

    n = 256
    t0 = time.perf_counter()
    _oracle_rows_step(w, qh, kh, vh, doh, np.arange(w.N - n, w.N))
    per_row = (time.perf_counter() - t0) / n
    m = int(max(64, min(w.N, budget_s / max(per_row, 1e-9))))
    return np.arange(w.N - m, w.N)


def _head_arrays(q, k, v, do):
    return [t[0, 0].to("cpu", torch.float64).numpy() for t in (q, k, v, do)]


def cpu_baseline(w, q, k, v, do, budget_s):
    """The oracle on whole heads of the workload (fwd + bwd), head after head
    until about `budget_s` seconds have been spent (at least one row block)."""
    import numpy as np

    qh, kh, vh, doh = _head_arrays(q, k, v, do)
    rows = _pick_rows(w, qh, kh, vh, doh, budget_s)
    heads = [(b, h) for b in range(w.B) for h in range(w.H)]
    flops, dt, done = 0.0, 0.0, 0
    if len(rows) < w.N:                      # one head is over budget: a block of its rows
        t0 = time.perf_counter()
        _oracle_rows_step(w, qh, kh, vh, doh, rows)
        dt = time.perf_counter() - t0
        flops = _rows_flops(w, rows)
        sample = f"fp64 numpy oracle fwd+bwd for the last {len(rows)} query rows of head (0,0)"
    else:
        all_rows = np.arange(w.N)
        for b, h in heads:
            arrs = [t[b, h].to("cpu", torch.float64).numpy() for t in (q, k, v, do)]
            t0 = time.perf_counter()
            _oracle_rows_step(w, *arrs, all_rows)
            dt += time.perf_counter() - t0
            flops += _rows_flops(w, all_rows)
            done += 1
            if dt >= budget_s:
                break
        sample = f"fp64 numpy oracle fwd+bwd on {done} of {len(heads)} heads (whole heads, all {w.N} rows)"
    return {"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": _CORES, "kind": "oracle",
            "sample": f"{sample}, {dt:.1f} s; FLOPs by the same convention as the GPU",
            "threads": os.environ.get("OPENBLAS_NUM_THREADS")}


def run_reference(args, w, rank, world):
    """The oracle as the reference arm: K timed steps of a bounded sample on host cores."""
    q, k, v, do = make_workload_inputs(w, device="cpu", heads=1)
    qh, kh, vh, doh = _head_arrays(q, k, v, do)
    per_step_budget = max(0.5, 150.0 / max(1, args.steps + args.warmup))
    rows = _pick_rows(w, qh, kh, vh, doh, per_step_budget)
    for _ in range(args.warmup):
        _oracle_rows_step(w, qh, kh, vh, doh, rows)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_rows_step(w, qh, kh, vh, doh, rows)
    dt = time.perf_counter() - t0
    value = _rows_flops(w, rows) * args.steps / dt / 1e12
    sample = (f"fp64 numpy oracle fwd+bwd, last {len(rows)} query rows of one head of {w.name} against all "
              f"{w.N} keys, per step")
    return {
        "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
        "config": {"workload": f"{w.name}: {w.describe()}", "B": w.B, "H": w.H, "N": w.N, "d": w.d,
                   "causal": w.causal},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": _CORES, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ------------------------------------------------------------------ main


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=600)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg (profiling runs)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    w = WORKLOADS[args.workload]
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, w, rank, world)), flush=True)
        return
    if world > 1:
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        torch.distributed.init_process_group("nccl")
    line = run_ours(args, w, rank, world)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
