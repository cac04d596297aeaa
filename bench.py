"""Benchmark: exact attention forward + backward TFLOP/s on one GB300.

One step = one pass of the whole hot path over one batch of synthetic input:
fa_fwd (O, LSE) then fa_bwd as its three stages (D pre-pass, tiled dQ/dK/dV
loop, dQ finish).  Inputs are resident in HBM before the timed region; L2 is
flushed (a 256 MiB write) before every timed step, outside the step's events.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--impl ours|reference] [--no-cpu-baseline] [--no-e2e]
                  [--no-workloads]

Prints one JSON line (rank 0).  Its headline (value, fwd, bwd, roofline,
e2e, cpu_baseline, clocks) is exactly K timed steps of --workload.  On one
GPU the same line also carries ``workloads``: every configuration (the
long-sequence case with and without the mask, the batched 2048 and causal
4096 cases, the d = 64 stress case and the tiny fp32 case), each timed for
at least half a second with its own clock record, its forward, backward and
dominant-kernel rates, and the oracle's forward and backward timed
separately on the host cores.  ``--impl reference`` times the fp64 CPU
oracle on this machine's host cores on a bounded sample of the workload.
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
import tempfile  # noqa: E402
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

# NVML clock-event reason bits (nvml.h) and the names nvidia-smi gives them.
_REASON_BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
                0x80: "hw_power_brake_slowdown"}


class NvmlClockSampler:
    """Polls the SM clock and the clock-event (throttle) reasons through NVML
    every `period_s` from a background thread while the timed work runs, so
    that even a region of a few tens of milliseconds gets a clock record."""

    def __init__(self, device, period_s=0.002):
        import ctypes
        import threading

        self._ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        uuid = str(getattr(torch.cuda.get_device_properties(device), "uuid", "") or "")
        found = False
        if uuid:
            tag = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
            found = self.lib.nvmlDeviceGetHandleByUUID(tag.encode(), ctypes.byref(self.h)) == 0
        if not found and self.lib.nvmlDeviceGetHandleByIndex_v2(device.index, ctypes.byref(self.h)) != 0:
            self.lib.nvmlShutdown()
            raise OSError("no NVML handle for the device")
        self._reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        self.period = period_s
        self.samples = []
        self._stop = threading.Event()
        self._thread = threading.Thread(target=self._run, daemon=True)
        c = ctypes.c_uint()
        self.max_mhz = float(c.value) if self.lib.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(c)) == 0 else None

    def _read(self):
        c, r = self._ct.c_uint(), self._ct.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.h, 1, self._ct.byref(c)) != 0:   # 1 = NVML_CLOCK_SM
            return None
        if self._reasons_fn(self.h, self._ct.byref(r)) != 0:
            return None
        return float(c.value), int(r.value)

    def _run(self):
        while not self._stop.is_set():
            x = self._read()
            if x is not None:
                self.samples.append(x)
            time.sleep(self.period)

    def start(self):
        self._thread.start()

    def stop(self):
        self._stop.set()
        self._thread.join()
        self.lib.nvmlShutdown()
        sm = [m for m, _ in self.samples]
        reasons = sorted({name for _, bits in self.samples for b, name in _REASON_BITS.items() if bits & b})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_min_mhz": min(sm) if sm else None,
                "sm_max_mhz": self.max_mhz, "reasons": reasons, "samples": len(sm),
                "source": f"NVML every {self.period * 1e3:.0f} ms during the timed region"}


class SmiClockSampler:
    """Fallback: nvidia-smi sampling of SM clocks and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.idx = device.index
        self.proc = None
        fd, self.path = tempfile.mkstemp(prefix=f"fa_clocks_gpu{self.idx}_", suffix=".csv")
        os.close(fd)

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu=timestamp,{self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            os.unlink(self.path)
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        try:
            return self._summary()
        finally:
            os.unlink(self.path)

    def _summary(self):
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
                "reasons": sorted(reasons), "samples": len(sm), "source": "nvidia-smi every 100 ms"}


def clock_sampler(device):
    try:
        return NvmlClockSampler(device)
    except (OSError, AttributeError):
        return SmiClockSampler(device)


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


class Harness:
    """Device buffers for one workload and one timed step of the whole hot
    path through the C ABI: fa_fwd, then fa_bwd as its three stages (D
    pre-pass, tiled dQ/dK/dV loop, dQ finish), with CUDA events around the
    forward, the backward and the tiled launch on the launching stream."""

    def __init__(self, fa, w, dev):
        import ctypes

        self.fa, self.w, self.dev = fa, w, dev
        self.q, self.k, self.v, self.do = make_workload_inputs(w, device=dev)
        q = self.q
        self.B, self.H, self.N, self.d = q.shape
        self.o = torch.empty_like(q)
        self.lse = torch.empty((self.B, self.H, self.N), dtype=torch.float32, device=dev)
        self.dq, self.dk, self.dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
        self.ws = torch.empty(max(fa.bwd_workspace_size(self.B, self.H, self.N, self.d, q.dtype), 1),
                              dtype=torch.uint8, device=dev)
        self.L = fa.lib()
        self.stream = torch.cuda.current_stream(dev)
        self.sp = ctypes.c_void_p(self.stream.cuda_stream)
        self.code = {torch.bfloat16: 0, torch.float32: 1, torch.float16: 2}[q.dtype]
        self.fws_n = fa.fwd_workspace_size(self.B, self.H, self.N, self.d, w.causal, q.dtype)
        self.fws = torch.empty(max(self.fws_n, 1), dtype=torch.uint8, device=dev)
        self._P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
        # Kernels one step launches: the forward (+ the merge of its split
        # last wave when it splits), then pre-pass, tiled loop, finish (the
        # fp32 path: pre-pass and its two backward kernels).
        self.launches_per_step = (2 if self.fws_n else 1) + 3

    def fwd(self):
        P = self._P
        st = self.L.fa_fwd(P(self.q), P(self.k), P(self.v), P(self.o), P(self.lse), self.B, self.H, self.N, self.d,
                           self.w.scale, int(self.w.causal), self.code, P(self.fws) if self.fws_n else None,
                           self.fws_n, self.sp)
        assert st == 0, self.fa.status_string(st)

    def step(self, ev=None):
        s = self.stream
        if ev is not None:
            ev[0].record(s)
        self.fwd()
        if ev is not None:
            ev[1].record(s)
        self.fa.bwd_stages(self.q, self.k, self.v, self.o, self.do, self.lse, self.dq, self.dk, self.dv, self.ws,
                           scale=self.w.scale, causal=self.w.causal,
                           between=None if ev is None else (lambda: ev[2].record(s), lambda: ev[3].record(s)))
        if ev is not None:
            ev[4].record(s)

    def head_arrays(self):
        """Head (0, 0) of the inputs in fp64 on the host (for the oracle)."""
        return [t[0, 0].to("cpu", torch.float64).numpy() for t in (self.q, self.k, self.v, self.do)]


def _stats(xs):
    return {"ms": round(statistics.mean(xs), 4), "ms_median": round(statistics.median(xs), 4),
            "ms_min": round(min(xs), 4), "ms_max": round(max(xs), 4)}


def time_steps(h, flush, warmup, steps=None, min_seconds=0.0, world=1):
    """Warm-up, then timed steps (exactly `steps`, or as many as fill
    `min_seconds`) with the L2 flushed before each, outside its events.
    Returns per-step times (ms) of the step, forward, backward and tiled
    launch, the clock record of the timed region and its wall time."""
    dev = h.dev
    for _ in range(warmup):
        flush.zero_()
        h.step()
    assert h.fa.sync_status(dev) == 0
    if steps is None:
        probe = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(3)]
        t0 = time.perf_counter()
        for e in probe:
            flush.zero_()
            h.step(e)
        torch.cuda.synchronize(dev)
        per_step = (time.perf_counter() - t0) / len(probe)
        steps = max(20, int(min_seconds / max(per_step, 1e-6)) + 1)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(steps)]
    clocks = clock_sampler(dev)
    clocks.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    wall0 = time.perf_counter()
    for i in range(steps):
        flush.zero_()
        h.step(ev[i])
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    status = h.fa.sync_status(dev)
    assert status == 0, h.fa.status_string(status)
    return {
        "steps": steps, "wall_s": wall, "clocks": clk,
        "step": [e[0].elapsed_time(e[4]) for e in ev], "fwd": [e[0].elapsed_time(e[1]) for e in ev],
        "bwd": [e[1].elapsed_time(e[4]) for e in ev], "tiles": [e[2].elapsed_time(e[3]) for e in ev],
    }


# The library's choice of backward kernel at d = 64 without the mask
# (kBwdPersistMaxTiles in csrc/fa_kernels.h): the persistent form when a head
# has at most this many 128-row query tiles and there are more K/V tiles than SMs.
BWD_PERSIST_MAX_TILES = 8


def dominant_kernel(w, n_sms=0):
    if n_sms <= 0 and torch.cuda.is_available():
        n_sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    if w.dtype == "fp32":
        return "dkv_f32_kernel + dq_f32_kernel (fa_bwd_tiles, fp32 SIMT)"
    if w.d == 256:
        return f"fa_bwd_d256 dkv + dq kernels<causal={int(w.causal)}> (fa_bwd_tiles)"
    tiles = -(-w.N // 128)
    if w.d == 64 and not w.causal and tiles <= BWD_PERSIST_MAX_TILES and w.B * w.H * tiles > n_sms > 0:
        return "fa_bwd_bf16_persist64_kernel (fa_bwd_tiles)"
    return f"fa_bwd_bf16_kernel<d={w.d},causal={int(w.causal)}> (fa_bwd_tiles)"


def summarise(w, t, peak):
    """Forward / backward / dominant-kernel rates of one workload's timed steps."""
    ff, fb = w.flops_fwd(), w.flops_bwd()
    f_ms, b_ms, k_ms = statistics.mean(t["fwd"]), statistics.mean(t["bwd"]), statistics.mean(t["tiles"])
    f_tf, b_tf, k_tf = ff / (f_ms * 1e-3) / 1e12, fb / (b_ms * 1e-3) / 1e12, fb / (k_ms * 1e-3) / 1e12
    return {
        "config": w.describe(), "dtype": w.dtype, "steps": t["steps"], "wall_s_timed": round(t["wall_s"], 3),
        "fwd": dict(tflops=round(f_tf, 2), frac_of_peak=round(f_tf / peak, 4), **_stats(t["fwd"])),
        "bwd": dict(tflops=round(b_tf, 2), frac_of_peak=round(b_tf / peak, 4), **_stats(t["bwd"])),
        "step_tflops": round((ff + fb) / (statistics.mean(t["step"]) * 1e-3) / 1e12, 2),
        "dominant_kernel": {"name": dominant_kernel(w), "tflops": round(k_tf, 2),
                            "frac_of_peak": round(k_tf / peak, 4), **_stats(t["tiles"])},
        "clocks": t["clocks"],
    }


def e2e_leg(fa, h, w, n_e2e, world):
    """End to end through the public API: every step copies its inputs in from
    pinned host memory and reads all of its results (O, LSE, dQ, dK, dV)
    back.  Pipelined the way a caller would: two sets of device buffers, and
    the uploads, the attention calls and the downloads on three streams, so
    step i's compute overlaps step i+1's upload and step i-1's download.
    The timed region runs from the first upload to the last download."""
    dev = h.dev
    q, k, v, do, lse, ws = h.q, h.k, h.v, h.do, h.lse, h.ws
    elem_bytes = q.numel() * q.element_size()
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
    flops = w.flops_fwd() + w.flops_bwd()
    return {"value": round(world * flops / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
            "h2d_bytes_per_step": 4 * elem_bytes, "d2h_bytes_per_step": 4 * elem_bytes + lse.numel() * 4,
            "ms_per_step": round(e2e_ms, 3), "steps": n_e2e,
            "pipelining": "two buffer sets; uploads, compute and downloads on three streams"}


# Every configuration the bench records besides the headline's K steps, each
# timed for at least this long (enough for a clock record of many samples).
TABLE_WORKLOADS = ("bf16_n8192", "bf16_causal_n8192", "bf16_n2048", "bf16_causal_n4096", "bf16_stress_n1024",
                   "tiny_fp32")
TABLE_MIN_SECONDS = 0.5


def run_ours(args, w, rank, world):
    import exact_tiled_attention_12_gb300 as fa
    from exact_tiled_attention_12_gb300.build import build

    build()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    peaks, peak_kind = load_peaks()
    peak = float(peaks["bf16_tflops"])
    peak_sus = float(peaks.get("bf16_tflops_sustained", peak))
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    # ---- the headline: exactly K timed steps of the workload
    h = Harness(fa, w, dev)
    t = time_steps(h, flush, args.warmup, steps=args.steps, world=world)
    B, H, N, d = h.q.shape
    total_ms = max_over_ranks(sum(t["step"]), dev, world)
    ms_per_step = total_ms / args.steps
    flops_fwd, flops_bwd = w.flops_fwd(), w.flops_bwd()
    value = job_tflops(flops_fwd + flops_bwd, args.steps, total_ms, world)
    head = summarise(w, t, peak)
    tiles_tflops = head["dominant_kernel"]["tflops"]
    clk = t["clocks"]
    # Clock-derived dense bf16 rate: SMs × 8192 FLOP per SM clock (2·4096 MACs,
    # the nominal 2.25 PFLOP/s over SMs and boost clock) × the maximum SM clock.
    n_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    sm_max = float(peaks.get("sm_max_mhz", 2070.0))
    peak_theory = n_sms * 8192 * sm_max * 1e6 / 1e12

    # 30 end-to-end steps (fewer if --steps is smaller): the first upload and
    # the last download, which nothing overlaps, then weigh 1/30 of the region.
    n_e2e = 0 if args.no_e2e else max(3, min(args.steps, 30))
    e2e = e2e_leg(fa, h, w, n_e2e, world) if n_e2e else None
    head_arrays = h.head_arrays() if rank == 0 and not args.no_cpu_baseline else None
    launches = h.launches_per_step * args.steps
    del h
    torch.cuda.empty_cache()

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": f"{w.name}: {w.describe()}", "B": B, "H": H, "N": N, "d": d, "causal": w.causal,
                   "flops_per_step": flops_fwd + flops_bwd, "flop_convention": "fwd 4N^2d, bwd 10N^2d per head, causal /2",
                   "l2": "flushed before every timed step (256 MiB write, outside the step's events)",
                   "parallelism": f"replicas x{world}"},
        "fwd": head["fwd"], "bwd": head["bwd"],
        "roofline": {"bound": "tensor", "kernel": dominant_kernel(w),
                     "achieved": tiles_tflops, "peak": peak, "peak_kind": f"{peak_kind} bf16 burst",
                     "unit": "TFLOP/s", "frac": round(tiles_tflops / peak, 4),
                     "frac_of_sustained": round(tiles_tflops / peak_sus, 4),
                     "peak_theoretical": round(peak_theory, 1),
                     "frac_of_theoretical": round(tiles_tflops / peak_theory, 4),
                     "peak_theoretical_note": f"{n_sms} SMs x 8192 FLOP/clk x {sm_max:.0f} MHz (clock-derived estimate)",
                     "ms_per_launch": head["dominant_kernel"]["ms"],
                     "algorithmic_flops_per_launch": flops_bwd,
                     "traffic": measured_traffic("fa_bwd_bf16_kernel", d, w.causal, w.name),
                     "traffic_unit": "bytes per launch (ncu dram read + write)"},
        "e2e": e2e,
        "softmax": {
            # exponentials of the forward (one per visible score) per SM clock at
            # the sampled median SM clock: the MUFU-side rate of the softmax
            "exp_per_clk_per_sm": (round(w.B * w.H * N * N / (2 if w.causal else 1)
                                         / (head["fwd"]["ms"] * 1e-3) / (clk["sm_mhz"] * 1e6) / n_sms, 2)
                                   if clk.get("sm_mhz") else None),
        },
        "gpu_launches": launches,
        "clocks": clk,
        "wall_s_timed": round(t["wall_s"], 4),
    }

    # ---- every configuration, each for at least TABLE_MIN_SECONDS (one GPU only)
    tables, oracle_inputs = {}, {}
    if world == 1 and not args.no_workloads:
        for name in TABLE_WORKLOADS:
            wl = WORKLOADS[name]
            hh = Harness(fa, wl, dev)
            tt = time_steps(hh, flush, args.warmup, min_seconds=TABLE_MIN_SECONDS)
            tables[name] = summarise(wl, tt, peak)
            tables[name]["gpu_launches"] = hh.launches_per_step * tt["steps"]
            if not args.no_cpu_baseline:
                oracle_inputs[name] = hh.head_arrays()
            del hh
            torch.cuda.empty_cache()
        line["workloads"] = tables

    # ---- the oracle on the host cores, after every GPU timing
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, head_arrays, budget_s=15.0)
        for name, arrs in oracle_inputs.items():
            tables[name]["cpu_baseline"] = cpu_baseline_split(WORKLOADS[name], arrs, budget_s=8.0)
    return line


# ------------------------------------------------------------------ CPU oracle


def _oracle_fwd_rows(w, qh, kh, vh, rows):
    import oracle

    oracle.attention_forward_rows(qh, kh, vh, rows, w.scale, w.causal)


def _oracle_bwd_rows(w, qh, kh, vh, doh, rows):
    import oracle

    oracle.attention_backward_rows(qh, kh, vh, doh, rows, w.scale, w.causal)


def _oracle_rows_step(w, qh, kh, vh, doh, rows):
    """fwd + bwd of the fp64 oracle restricted to a block of query rows."""
    _oracle_fwd_rows(w, qh, kh, vh, rows)
    _oracle_bwd_rows(w, qh, kh, vh, doh, rows)


def _visible_pairs(w, rows):
    return sum((r + 1) if w.causal else w.N for r in rows)


def _rows_flops(w, rows):
    """Algorithmic FLOPs (fwd + bwd) of the sampled rows under the bench's convention (per-row share)."""
    return 14.0 * _visible_pairs(w, rows) * w.d


def _pick_rows(w, qh, kh, vh, doh, budget_s):
    """Largest contiguous block of the last query rows whose fwd+bwd fits the time budget."""
    import numpy as np

    n = min(256, w.N)
    t0 = time.perf_counter()
    _oracle_rows_step(w, qh, kh, vh, doh, np.arange(w.N - n, w.N))
    per_row = (time.perf_counter() - t0) / n
    m = int(max(min(64, w.N), min(w.N, budget_s / max(per_row, 1e-9))))
    return np.arange(w.N - m, w.N)


def cpu_baseline(w, arrays, budget_s):
    """The oracle (fwd + bwd) on head (0, 0) of the workload: the whole head
    when it fits the budget, repeated for the other heads' worth of work up
    to the budget, else the largest block of its last rows that fits."""
    import numpy as np

    qh, kh, vh, doh = arrays
    rows = _pick_rows(w, qh, kh, vh, doh, budget_s)
    flops, dt, reps = 0.0, 0.0, 0
    while True:
        t0 = time.perf_counter()
        _oracle_rows_step(w, qh, kh, vh, doh, rows)
        dt += time.perf_counter() - t0
        flops += _rows_flops(w, rows)
        reps += 1
        if len(rows) < w.N or dt >= budget_s or reps >= w.B * w.H:
            break
    if len(rows) < w.N:
        sample = f"fp64 numpy oracle fwd+bwd for the last {len(rows)} query rows of head (0,0) against all {w.N} keys"
    else:
        sample = f"fp64 numpy oracle fwd+bwd on head (0,0), all {w.N} rows, {reps} time(s)"
    return {"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": _CORES, "kind": "oracle",
            "sample": f"{sample}, {dt:.1f} s; FLOPs by the same convention as the GPU",
            "threads": os.environ.get("OPENBLAS_NUM_THREADS")}


def cpu_baseline_split(w, arrays, budget_s):
    """The oracle's forward and backward timed separately on the same block of
    the last query rows of head (0, 0), sized so that one forward and one
    backward take about `budget_s`; a block that is quicker than that (a
    whole small head) is repeated until each leg has run for its share."""
    qh, kh, vh, doh = arrays
    rows = _pick_rows(w, qh, kh, vh, doh, budget_s)

    def timed(fn, share):
        n, dt = 0, 0.0
        while n == 0 or dt < share * budget_s:
            t0 = time.perf_counter()
            fn()
            dt += time.perf_counter() - t0
            n += 1
        return n, dt

    n_f, t_f = timed(lambda: _oracle_fwd_rows(w, qh, kh, vh, rows), 0.3)
    n_b, t_b = timed(lambda: _oracle_bwd_rows(w, qh, kh, vh, doh, rows), 0.6)
    pairs = _visible_pairs(w, rows)
    return {"fwd": {"tflops": round(4.0 * pairs * w.d * n_f / t_f / 1e12, 6), "seconds": round(t_f, 3), "reps": n_f},
            "bwd": {"tflops": round(10.0 * pairs * w.d * n_b / t_b / 1e12, 6), "seconds": round(t_b, 3), "reps": n_b},
            "unit": "TFLOP/s", "cores": _CORES, "kind": "oracle",
            "sample": f"fp64 numpy oracle, the last {len(rows)} query rows of head (0,0) against all {w.N} keys "
                      f"(the backward recomputes P for its rows); FLOPs by the same convention as the GPU",
            "threads": os.environ.get("OPENBLAS_NUM_THREADS")}


def run_reference(args, w, rank, world):
    """The oracle as the reference arm: K timed steps of a bounded sample on host cores."""
    q, k, v, do = make_workload_inputs(w, device="cpu", heads=1)
    qh, kh, vh, doh = [t[0, 0].to("cpu", torch.float64).numpy() for t in (q, k, v, do)]
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
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the per-configuration table (profiling runs)")
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
