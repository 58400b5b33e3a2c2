#!/usr/bin/env python
"""Benchmark of the fused MoE dispatch + expert GEMM on GB300.

One step = one pass of the whole path (router top-k, histogram + scan,
gather into expert-contiguous tiles, expert GEMM) over one batch of the
seeded synthetic workload, through the C ABI.  The headline workload is the
Mixtral-like layer (T=4096, H=4096, F=14336, E=8, top-2, seed 1); at one GPU
the same JSON line also carries a ``per_config`` block that measures all
five seeded workloads (tiny, Mixtral-like, fine-grained skewed, decode,
imbalanced large batch) the same way: fused and unfused launches, the
dispatch role alone, the roofline of the workload's bound, the clocks seen
during its timed region, and the CPU oracle on a bounded sample of it.

Timing: W warm-up steps, then exactly K timed steps; every step is bracketed
by CUDA events on the launching stream, with a 256 MiB write (larger than
L2) between steps outside the events; the timed region is bracketed by a
barrier and a device synchronise; the max over ranks is taken.  Clocks and
throttle reasons are sampled in-process through NVML queries every 0.5 ms
while the timed region runs.  Under torchrun every rank runs its own batch
(weak scaling, no data-path collective).

``--impl reference`` times the CPU oracle instead (rank 0 only), each step a
bounded sample of the same workload.  Prints ONE JSON line on rank 0.
"""
from __future__ import annotations

import argparse
import ctypes
import datetime
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from moe_token_dispatch_persistent_gb300 import synth  # noqa: E402

METRIC = "fused dispatch+grouped-GEMM TFLOP/s (% bf16 peak) and dispatch GB/s (% HBM)"
UNIT = "TFLOP/s"
FLUSH_BYTES = 256 << 20
L2_NOTE = "flushed between timed GPU steps (256 MiB write, outside the events)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=2, choices=sorted(synth.WORKLOADS),
                    help="headline workload (the line's value)")
    ap.add_argument("--configs", default="1,2,3,4,5",
                    help="workloads of the per_config block at one GPU (comma list, or 'none')")
    ap.add_argument("--dispatch-ctas", type=int, default=0)
    ap.add_argument("--n-group", type=int, default=0)
    ap.add_argument("--no-extras", action="store_true",
                    help="headline only: no per_config block and no unfused / dispatch-only / e2e / cpu legs")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="budget of the headline CPU-baseline sample")
    ap.add_argument("--cpu-seconds-per-config", type=float, default=4.0,
                    help="budget of each per_config CPU-baseline sample")
    ap.add_argument("--dispatch-only", action="store_true",
                    help="time the dispatch role alone (routing, scan, gather; no GEMM) as the main loop, in GB/s")
    ap.add_argument("--experts-div", type=int, default=1,
                    help="small case for profiler captures: E/D experts and T/D tokens, H, F, k and the value "
                         "recipe unchanged (not a bench workload)")
    ap.add_argument("--trace", action="store_true",
                    help="instead of the bench line: per-phase times of the fused launch (trace stamps, median of "
                         "5 traced launches after 3 warm-ups) for each workload of --configs, one JSON line")
    ap.add_argument("--h-div", type=int, default=1,
                    help="small case for profiler captures: H/D, everything else unchanged, so routing and the "
                         "rows of every expert stay those of the full layer (not a bench workload)")
    return ap.parse_args(argv)


# --------------------------------------------------------------- helpers --

def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_code_digest(paths) -> str:
    """sha256 of the sources' code: comments and whitespace removed, so an
    edit of a comment does not invalidate a capture (nothing else changes
    the compiled kernel)."""
    import hashlib
    import re

    h = hashlib.sha256()
    for src in paths:
        with open(os.path.join(ROOT, src), encoding="utf-8") as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()


def ncu_traffic(workload_name: str):
    """DRAM bytes (read + write) per launch of the fused kernel from the
    committed ncu capture of this workload (profiles/ncu_traffic.json), or
    None when there is none or the kernel code changed since it was taken.
    Returns (bytes, source) or (None, reason)."""
    try:
        with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
            rec = json.load(f).get(workload_name)
    except (OSError, ValueError):
        return None, "no committed capture"
    if not rec:
        return None, "no committed capture of this workload"
    try:
        digest = kernel_code_digest(rec["kernel_sources"])
    except OSError:
        return None, "kernel sources missing"
    if digest != rec["kernel_code_sha256"]:
        return None, "kernel code changed since the committed capture"
    src = f"committed ncu capture ({rec.get('source', 'profiles/')}), kernel code digest matches"
    if rec.get("scaled_from"):
        src += f"; {rec['scaled_from']}"
    return rec["bytes_per_launch"], src


def reduced_workload(w: synth.Workload, d: int) -> synth.Workload:
    """The same layer with E/d experts and T/d tokens: H, F, k, the seed and
    the value recipe stay, so the rows per expert stay about the same while
    the weights shrink d-fold.  A small case of the same kernel for profiler
    captures of workloads whose full size holds many GB on the device."""
    if d == 1:
        return w
    if d < 1 or w.E % d or w.T % d or w.E // d < 32:
        raise SystemExit(f"--experts-div {d}: needs a divisor of E={w.E} and T={w.T} leaving at least 32 experts")
    return synth.Workload(f"{w.name}_experts_div_{d}", w.T // d, w.H, w.F, w.E // d, w.k, w.seed, w.kind)


def reduced_hidden(w: synth.Workload, d: int) -> synth.Workload:
    """The same layer with H/d: T, E, k, F, the seed and the logits recipe
    stay, so routing, the active experts and every expert's rows are those
    of the full layer while the weights shrink d-fold.  A small case of the
    same kernel for profiler captures of a skewed or decode layer whose full
    weights hold many GB on the device."""
    if d == 1:
        return w
    if d < 1 or w.H % (64 * d):
        raise SystemExit(f"--h-div {d}: H={w.H} / {d} must stay a multiple of 64")
    return synth.Workload(f"{w.name}_h_div_{d}", w.T, w.H // d, w.F, w.E, w.k, w.seed, w.kind)


def compulsory_bytes(w: synth.Workload, active_experts: int) -> int:
    """x + logits + active experts' W + y_sorted (bf16) + src_index + gate_w + offsets."""
    return (w.T * w.H * 2 + w.T * w.E * 4 + active_experts * w.H * w.F * 2 + w.rows * w.F * 2 + w.rows * 8
            + (w.E + 1) * 4)


def dispatch_bytes(w: synth.Workload) -> int:
    """Algorithmic bytes of the dispatch role: logits read, token rows read and
    written to the staging tiles, src_index / gate_w written, offsets."""
    return w.T * w.E * 4 + 2 * w.rows * w.H * 2 + w.rows * 8 + (w.E + 1) * 4


def roofline_bound(w: synth.Workload, active_experts: int, peaks) -> str:
    """The bound of the fused launch: the larger of the time its FLOPs take
    at the bf16 peak and the time its compulsory bytes take at the HBM peak."""
    t_tensor = w.flop / (float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])) * 1e12)
    t_hbm = compulsory_bytes(w, active_experts) / (float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])) * 1e9)
    return "tensor" if t_tensor >= t_hbm else "hbm"


def bench_config(w: synth.Workload):
    """The line's ``config``: the workload and how L2 is handled.  Both arms
    print exactly this dict, so the two lines name the same workload."""
    return {"workload": w.describe(), "T": w.T, "H": w.H, "F": w.F, "E": w.E, "k": w.k, "seed": w.seed,
            "l2": L2_NOTE}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(value: float, world: int) -> float:
    """Max of a float over ranks (identity at world 1)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flop_per_rank: float, world: int, seconds_max: float) -> float:
    return flop_per_rank * world / seconds_max / 1e12


# ---------------------------------------------------------------- clocks --

# NVML clocks-event reason bits (nvml.h): the four the timing rules name.
_REASON_BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
                "hw_thermal_slowdown": 0x40}
_NVML_CLOCK_SM = 1


class NvmlClocks:
    """SM clock and throttle reasons of one GPU, sampled in-process every
    ``period_s`` by a thread doing NVML queries (read only) while a timed
    region runs, so that short regions still hold samples.  ``start_region``
    starts the thread, ``end_region`` stops it; ``region()`` summarises the
    samples of the last region (with the one the caller takes from the main
    thread by ``sample_now`` while the GPU still runs the enqueued steps)."""

    def __init__(self, nvml_index: int, period_s: float = 0.0005):
        self.ok = False
        self.period = period_s
        self.samples = []  # (t, sm_mhz, reasons_bits)
        self.lock = threading.Lock()
        self.t0 = self.t1 = None
        self._stop = threading.Event()
        self._th = None
        try:
            lib = None
            for name in ("libnvidia-ml.so.1", "libnvidia-ml.so"):
                try:
                    lib = ctypes.CDLL(name)
                    break
                except OSError:
                    continue
            if lib is None or lib.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(nvml_index), ctypes.byref(h)) != 0:
                return
            self.lib, self.h = lib, h
            mx = ctypes.c_uint()
            self.max_mhz = (float(mx.value) if lib.nvmlDeviceGetMaxClockInfo(h, _NVML_CLOCK_SM, ctypes.byref(mx)) == 0
                            else None)
            self._reasons_fn = (getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None)
                                or getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons", None))
            self.ok = self.read() is not None
        except (OSError, AttributeError):
            self.ok = False

    def read(self):
        mhz = ctypes.c_uint()
        if self.lib.nvmlDeviceGetClockInfo(self.h, _NVML_CLOCK_SM, ctypes.byref(mhz)) != 0:
            return None
        bits = ctypes.c_ulonglong(0)
        if self._reasons_fn is not None:
            self._reasons_fn(self.h, ctypes.byref(bits))
        return (time.perf_counter(), float(mhz.value), int(bits.value))

    def _loop(self):
        while not self._stop.is_set():
            s = self.read()
            if s is not None:
                with self.lock:
                    self.samples.append(s)
            time.sleep(self.period)

    def sample_now(self):
        if self.ok:
            s = self.read()
            if s is not None:
                with self.lock:
                    self.samples.append(s)

    def start_region(self):
        with self.lock:
            self.samples = []
        self.t0 = time.perf_counter()
        if self.ok:
            self._stop.clear()
            self._th = threading.Thread(target=self._loop, daemon=True)
            self._th.start()

    def end_region(self):
        self.t1 = time.perf_counter()
        if self._th is not None:
            self._stop.set()
            self._th.join(timeout=2)
            self._th = None

    def stop(self):
        pass

    def region(self):
        if not self.ok:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvml unavailable"], "samples": 0,
                    "samples_in_timed_region": 0, "source": "none"}
        with self.lock:
            inside = [s for s in self.samples if self.t0 <= s[0] <= self.t1]
        reasons = sorted({nm for s in inside for nm, b in _REASON_BITS.items() if s[2] & b})
        mhz = [s[1] for s in inside]
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_mhz_min": min(mhz) if mhz else None,
                "sm_max_mhz": self.max_mhz, "reasons": reasons, "samples": len(inside),
                "samples_in_timed_region": len(inside), "period_ms": self.period * 1e3,
                "timed_region_ms": (self.t1 - self.t0) * 1e3, "source": "nvml queries in-process"}


class SmiClocks:
    """Fallback when NVML cannot be loaded: nvidia-smi sampling every 50 ms
    for the whole run (queries only); a region keeps the rows inside it."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu, self.proc = gpu_index, None
        self.t0 = self.t1 = None
        self.ok = True
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(self.gpu), "-lms", "50"], stdout=self.fh,
                                         stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def sample_now(self):
        pass

    def start_region(self):
        self.t0 = time.time()

    def end_region(self):
        self.t1 = time.time()
        time.sleep(0.06)  # the sample after the region is written

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        os.unlink(self.path)
        self.proc = None

    def region(self):
        rows = []
        if self.proc is not None:
            self.fh.flush()
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) < 10:
                        continue
                    try:
                        ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                        rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10]))
                    except ValueError:
                        continue
        inside = [r for r in rows if self.t0 is not None and self.t0 <= r[0] <= self.t1]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({nm for r in inside for nm, v in zip(names, r[3]) if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[1] for r in inside) if inside else None,
                "sm_max_mhz": max(r[2] for r in inside) if inside else None, "reasons": reasons,
                "samples": len(inside), "samples_in_timed_region": len(inside), "period_ms": 50,
                "source": "nvidia-smi"}


def make_clock_sampler(local: int):
    try:
        import torch

        idx = torch.cuda._get_nvml_device_index(local)
    except Exception:  # noqa: BLE001 -- any failure: the plain index
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        idx = int(vis.split(",")[local]) if vis and vis.split(",")[local].strip().isdigit() else local
    s = NvmlClocks(idx)
    if s.ok:
        return s
    return SmiClocks(idx)


# ------------------------------------------------------------ reference --

_WE_CACHE = {}


def oracle_sample(w: synth.Workload, budget_s: float, inputs=None):
    """Time the CPU oracle on a bounded sample of workload ``w``.

    One sample = the routing + dispatch of all T tokens plus the fp64 expert
    product of n sorted rows of the most loaded expert, n sized so the
    product takes about ``budget_s``.  The value is the sample's product
    FLOPs (2*n*H*F; routing counts no FLOPs) over the sample's wall time, a
    measured rate; the time the whole workload would take at that rate is
    reported beside it, marked as an estimate.
    """
    from oracle.oracle import Oracle

    orc = Oracle()
    if inputs is None:
        ch = synth._streams(w)
        logits = synth.make_logits(w, ch)
        x = synth.make_x(w, ch)
    else:
        x, logits = inputs
    t0 = time.perf_counter()
    idx, gate = orc.route(logits, w.k)
    offsets, src, gw = orc.dispatch(idx, gate, w.E)
    t_route = time.perf_counter() - t0
    # rows of the most loaded expert: one weight matrix for the whole sample
    e = int(np.argmax(np.diff(offsets)))
    key = (w.seed, w.E, w.H, w.F, e)
    if key not in _WE_CACHE:
        _WE_CACHE.clear()
        _WE_CACHE[key] = synth.make_w_expert(w, e)
    We = _WE_CACHE[key]
    off1 = np.array([0, offsets[e + 1] - offsets[e]], dtype=np.int32)
    src1 = src[offsets[e]:offsets[e + 1]]
    n = max(1, min(off1[1], orc.num_threads()))
    t0 = time.perf_counter()
    orc.expert_rows(x, We[None], w.k, off1, src1, np.arange(n))
    t_cal = (time.perf_counter() - t0) / n
    n = int(max(1, min(off1[1], budget_s / max(t_cal, 1e-9))))
    t0 = time.perf_counter()
    orc.expert_rows(x, We[None], w.k, off1, src1, np.arange(n))
    t_rows = time.perf_counter() - t0
    t_step = t_route + t_rows
    flop = 2.0 * n * w.H * w.F
    rate = flop / t_step
    return {
        "value": rate / 1e12,
        "unit": UNIT,
        "cores": orc.num_threads(),
        "kind": "oracle",
        "sample": (f"routing+dispatch of all {w.T} tokens ({t_route:.3f} s) + fp64 product of {n} of {w.rows} "
                   f"sorted rows ({t_rows:.2f} s); value = the sample's product FLOPs / its time"),
        "sample_seconds": t_step,
        "full_workload_seconds_estimated": w.flop / rate,
        "estimated": True,
    }


def run_reference(args, w):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    # each step a bounded sample: the whole run ends within a few minutes
    per_step_budget = max(0.05, min(4.0, 100.0 / max(1, args.steps + args.warmup)))
    times, rates, cb = [], [], None
    ch = synth._streams(w)
    inputs = (synth.make_x(w, ch), synth.make_logits(w, ch))
    for i in range(args.warmup + args.steps):
        r = oracle_sample(w, per_step_budget, inputs)
        if i >= args.warmup:
            times.append(r["sample_seconds"])
            rates.append(r["value"])
            cb = r
    value = statistics.mean(rates)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": statistics.mean(times) * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
        "config": bench_config(w),
        "step": "one bounded sample of the workload on the host cores (see cpu_baseline.sample)",
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cb["cores"], "kind": "oracle", "sample": cb["sample"],
                         "full_workload_seconds_estimated": cb["full_workload_seconds_estimated"],
                         "estimated": True},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ ours --

TILE_NAMES = {1: "128-row", 2: "256-row on SM pairs", 3: "256-row (two accumulators per SM)"}
GATHER_NAMES = {1: "staged rows", 2: "rows straight from x (cp.async)", 3: "rows straight from x (TMA gather4)"}


class Gpu:
    """Device state of one rank: the library, the stream, the L2 flush buffer."""

    def __init__(self, local: int):
        import torch

        import moe_token_dispatch_persistent_gb300 as mk
        from moe_token_dispatch_persistent_gb300 import build

        self.torch, self.mk = torch, mk
        build.build()
        self.dev = torch.device("cuda", torch.cuda.current_device())
        self.stream = torch.cuda.current_stream(self.dev)
        self.flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=self.dev)

    def upload(self, x_np, l_np, W_np):
        torch = self.torch
        x = torch.from_numpy(x_np.view(np.int16)).view(torch.bfloat16).to(self.dev)
        logits = torch.from_numpy(l_np).to(self.dev)
        W = torch.from_numpy(W_np.view(np.int16)).view(torch.bfloat16).to(self.dev)
        return x, logits, W

    def timed(self, call, steps, warmup, clocks=None):
        """Per-step CUDA-event times (ms) of ``call``; with ``clocks`` the
        timed region is marked on the sampler."""
        torch, mk = self.torch, self.mk
        for _ in range(warmup):
            self.flush.fill_(1)
            call()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        if clocks is not None:
            clocks.start_region()
        for a, b in evs:
            self.flush.fill_(1)
            a.record(self.stream)
            call()
            b.record(self.stream)
        if clocks is not None:
            clocks.sample_now()  # the GPU is still running the enqueued steps
        torch.cuda.synchronize()
        if clocks is not None:
            clocks.end_region()
        st = mk.mk_get_status(self.stream)
        if st != mk.MK_OK:
            raise mk.MkError(st, "device status")
        return [a.elapsed_time(b) for a, b in evs]


def roofline(w, active, ms_mean, peaks, peaks_src):
    """Roofline of the fused launch on workload ``w`` (its bound chosen by
    roofline_bound), from the mean CUDA-event time of a launch."""
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    traffic, tsrc = ncu_traffic(w.name)
    cb = compulsory_bytes(w, active)
    if roofline_bound(w, active, peaks) == "hbm":
        achieved = cb / (ms_mean / 1e3) / 1e9
        r = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
             "peak_source": f"hbm_gbs (copy: read+write bytes), {peaks_src}",
             "note": "mostly reads: a read stream can exceed the copy bandwidth, so frac can pass 1",
             "tflops": w.flop / (ms_mean / 1e3) / 1e12}
    else:
        achieved = w.flop / (ms_mean / 1e3) / 1e12
        r = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
             "peak_source": f"bf16_tflops (burst), {peaks_src}"}
    r.update({"kernel": "mk_fused_kernel", "traffic": traffic, "traffic_source": tsrc, "compulsory_bytes": cb,
              "algorithmic_per_launch": w.flop if r["bound"] == "tensor" else cb})
    return r


def measure_workload(g: Gpu, w: synth.Workload, args, peaks, peaks_src, clocks, inputs=None, cpu_budget=4.0,
                     headline_ms=None):
    """One workload of the per_config block: fused launch (K steps), the same
    steps as four launches, the dispatch role alone, roofline, clocks and the
    CPU oracle on a bounded sample."""
    mk, torch = g.mk, g.torch
    ch = synth._streams(w)
    if inputs is None:
        x_np, l_np = synth.make_x(w, ch), synth.make_logits(w, ch)
        W_np = synth.make_w(w)
        x, logits, W = g.upload(x_np, l_np, W_np)
        del W_np
    else:
        x_np, l_np, x, logits, W = inputs
    out = mk.alloc_outputs(w.T, w.F, w.E, w.k, device=g.dev)

    def call(c):
        st = mk.mk_moe_dispatch_gemm_ex(x, logits, w.T, w.H, w.E, w.k, W, w.F, out["y_sorted"], out["src_index"],
                                        out["expert_offsets"], out["gate_w"], g.stream, c)
        if st != mk.MK_OK:
            raise mk.MkError(st, "mk_moe_dispatch_gemm_ex")

    cfg = mk.make_config()
    if headline_ms is None:
        ms = g.timed(lambda: call(cfg), args.steps, args.warmup, clocks)
        clk = clocks.region()
    else:
        ms, clk = headline_ms
    info = mk.mk_last_launch_info() if headline_ms is None else None
    if info is None:
        call(cfg)
        torch.cuda.synchronize()
        info = mk.mk_last_launch_info()
    active = int((np.diff(out["expert_offsets"].cpu().numpy()) > 0).sum())
    ms_mean = statistics.mean(ms)
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    ucfg = mk.make_config(mode=mk.MK_MODE_UNFUSED)
    ums = statistics.mean(g.timed(lambda: call(ucfg), args.steps, 3))
    dcfg = mk.make_config(mode=mk.MK_MODE_DISPATCH_ONLY)
    dms = statistics.mean(g.timed(lambda: call(dcfg), args.steps, 3))
    db = dispatch_bytes(w)
    # the three ways token rows reach the GEMM, on the default tiles
    forms = {}
    for name, gv in (("staged", mk.MK_GATHER_STAGED), ("cp_async", mk.MK_GATHER_DIRECT),
                     ("tma_gather4", mk.MK_GATHER_GATHER4)):
        fc = mk.make_config(gather=gv)
        forms[name] = statistics.mean(g.timed(lambda: call(fc), args.steps, 3))
    rec = {
        "workload": w.describe(),
        "ms_mean": ms_mean, "ms_median": statistics.median(ms), "ms_min": min(ms), "steps": len(ms),
        "tflops": w.flop / (ms_mean / 1e3) / 1e12,
        "roofline": roofline(w, active, ms_mean, peaks, peaks_src),
        "clocks": clk,
        "fused_ms": ms_mean, "unfused_ms": ums, "fused_speedup": ums / ms_mean, "unfused_launches_per_step": 4,
        "dispatch": {"gbs": db / (dms / 1e3) / 1e9, "frac_hbm": db / (dms / 1e3) / 1e9 / hbm, "ms": dms,
                     "bytes": db, "peak_gbs": hbm, "peak_source": f"hbm_gbs, {peaks_src}"},
        "active_experts": active,
        "row_forms_ms": forms,
        "launch": {"grid_ctas": info["grid_ctas"], "dispatch_ctas": info["dispatch_ctas"],
                   "n_group": info["n_group"], "tiles": TILE_NAMES.get(info["mma_pair"], str(info["mma_pair"])),
                   "rows": GATHER_NAMES.get(info["gather"], str(info["gather"])),
                   "route_lanes": info["route_lanes"]},
    }
    if cpu_budget > 0:
        rec["cpu_baseline"] = {k: v for k, v in oracle_sample(w, cpu_budget, (x_np, l_np)).items()
                               if k != "sample_seconds"}
    del out
    return rec


def run_ours(args, w):
    import torch

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    g = Gpu(local)
    mk = g.mk
    peaks, peaks_src = load_peaks()
    clocks = make_clock_sampler(local)

    # inputs: each rank its own batch of tokens (seed offset), same expert weights
    wr = synth.Workload(w.name, w.T, w.H, w.F, w.E, w.k, w.seed + 1000 * rank, w.kind) if rank else w
    ch = synth._streams(wr)
    x_np, l_np = synth.make_x(wr, ch), synth.make_logits(wr, ch)
    W_np = synth.make_w(w)
    x, logits, W = g.upload(x_np, l_np, W_np)
    del W_np
    out = mk.alloc_outputs(w.T, w.F, w.E, w.k, device=g.dev)
    stream = g.stream
    cfg = mk.make_config(dispatch_ctas=args.dispatch_ctas, n_group=args.n_group,
                         mode=mk.MK_MODE_DISPATCH_ONLY if args.dispatch_only else mk.MK_MODE_FUSED)
    combined = torch.empty((w.T, w.F), dtype=torch.bfloat16, device=g.dev)

    def call(c, combine=False):
        if combine:
            st = mk.mk_moe_dispatch_gemm_combine(x, logits, w.T, w.H, w.E, w.k, W, w.F, out["y_sorted"],
                                                 out["src_index"], out["expert_offsets"], out["gate_w"], combined,
                                                 stream, c)
        else:
            st = mk.mk_moe_dispatch_gemm_ex(x, logits, w.T, w.H, w.E, w.k, W, w.F, out["y_sorted"],
                                            out["src_index"], out["expert_offsets"], out["gate_w"], stream, c)
        if st != mk.MK_OK:
            raise mk.MkError(st, "mk_moe_dispatch_gemm_ex")

    # headline: the fused path, exactly K timed steps
    for _ in range(args.warmup):
        g.flush.fill_(1)
        call(cfg)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    ms = g.timed(lambda: call(cfg), args.steps, 0, clocks)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.region()
    info = mk.mk_last_launch_info()
    gpu_launches = args.steps * info["launches"]
    ms_mean = statistics.mean(ms)
    ms_max = reduce_max(ms_mean, world)
    value = whole_job_tflops(w.flop, world, ms_max / 1e3)
    active = int((np.diff(out["expert_offsets"].cpu().numpy()) > 0).sum())

    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    unit = UNIT
    if args.dispatch_only:
        # the dispatch role alone: its algorithmic bytes against HBM
        db = dispatch_bytes(w)
        achieved = db / (ms_mean / 1e3) / 1e9
        value = db * world / (ms_max / 1e3) / 1e9
        unit = "GB/s"
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                "peak_source": f"hbm_gbs, {peaks_src}", "kernel": "mk_fused_kernel (dispatch only)",
                "traffic": None, "traffic_source": "not captured for this mode", "algorithmic_bytes": db}
    else:
        roof = roofline(w, active, ms_mean, peaks, peaks_src)
    line = {
        "metric": METRIC, "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": bench_config(w),
        "launch": {"mode": "dispatch only" if args.dispatch_only else "fused persistent",
                   "grid_ctas": info["grid_ctas"], "dispatch_ctas": info["dispatch_ctas"],
                   "n_group": info["n_group"], "tiles": TILE_NAMES.get(info["mma_pair"], str(info["mma_pair"])),
                   "rows": GATHER_NAMES.get(info["gather"], str(info["gather"])), "active_experts": active},
        "roofline": roof,
        "gpu_launches": gpu_launches,
        "clocks": clk,
        "ms_per_step_min": min(ms), "ms_per_step_median": statistics.median(ms),
    }

    if not (args.no_extras or args.dispatch_only):
        steps_x = min(args.steps, 50)
        # dispatch role alone (routing + gather), GB/s against HBM
        dcfg = mk.make_config(mode=mk.MK_MODE_DISPATCH_ONLY)
        dms = statistics.mean(g.timed(lambda: call(dcfg), steps_x, 3))
        db = dispatch_bytes(w)
        line["dispatch"] = {"gbs": db / (dms / 1e3) / 1e9, "frac_hbm": db / (dms / 1e3) / 1e9 / hbm,
                            "ms": dms, "bytes": db, "peak_gbs": hbm}
        # the same steps as four launches (host-driven baseline)
        ucfg = mk.make_config(mode=mk.MK_MODE_UNFUSED)
        ums = statistics.mean(g.timed(lambda: call(ucfg), steps_x, 3))
        line["unfused"] = {"ms_per_step": ums, "tflops": w.flop / (ums / 1e3) / 1e12,
                           "fused_speedup": ums / ms_mean, "launches_per_step": 4}
        # the MoE layer's combine (gated sum of each token's expert rows)
        cms = statistics.mean(g.timed(lambda: call(cfg, True), steps_x, 3))
        cums = statistics.mean(g.timed(lambda: call(ucfg, True), steps_x, 3))
        cbytes = w.rows * w.F * 2 + w.T * w.F * 2 + w.rows * 8  # y_sorted read, out written, rows + gates
        line["combine"] = {"fused_ms": cms, "unfused_ms": cums, "fused_speedup": cums / cms,
                           "added_ms": cms - ms_mean, "bytes": cbytes,
                           "added_gbs": cbytes / max(cms - ms_mean, 1e-6) * 1e3 / 1e9}
        # the gated (SwiGLU) expert FFN: two projections, one tensor-core pass per item
        w3 = synth.Workload(w.name, w.T, w.H, w.F, w.E, w.k, w.seed + 7, w.kind)
        W3 = torch.from_numpy(synth.make_w(w3).view(np.int16)).view(torch.bfloat16).to(g.dev)

        def gated_once():
            st = mk.mk_moe_dispatch_gated(x, logits, w.T, w.H, w.E, w.k, W, W3, w.F, out["y_sorted"],
                                          out["src_index"], out["expert_offsets"], out["gate_w"], stream, cfg)
            if st != mk.MK_OK:
                raise mk.MkError(st, "mk_moe_dispatch_gated")

        gms = statistics.mean(g.timed(gated_once, steps_x, 3))
        line["gated"] = {"ms": gms, "tflops": 2 * w.flop / (gms / 1e3) / 1e12,
                         "frac_bf16": 2 * w.flop / (gms / 1e3) / 1e12 / peak}
        del W3
        # token rows straight from x (no staging rows): the same product
        dgcfg = mk.make_config(dispatch_ctas=args.dispatch_ctas, n_group=args.n_group, gather=mk.MK_GATHER_DIRECT)
        dgms = statistics.mean(g.timed(lambda: call(dgcfg), steps_x, 3))
        line["direct_gather"] = {
            "ms": dgms, "tflops": w.flop / (dgms / 1e3) / 1e12, "frac_bf16": w.flop / (dgms / 1e3) / 1e12 / peak,
            "vs_staged": ms_mean / dgms,
            "workspace_bytes": mk.mk_workspace_size(w.T, w.H, w.F, w.E, w.k, dgcfg),
            "staged_workspace_bytes": mk.mk_workspace_size(w.T, w.H, w.F, w.E, w.k, cfg)}
        # expert parallelism simulated on this GPU: the most ranks (<= 8) that divide E
        ranks = max(r for r in (1, 2, 4, 8) if w.E % r == 0)

        def ep_once():
            st = mk.mk_moe_ep_sim(x, logits, w.T, w.H, w.E, w.k, W, w.F, ranks, out["y_sorted"], out["src_index"],
                                  out["expert_offsets"], out["gate_w"], combined, stream, cfg)
            if st != mk.MK_OK:
                raise mk.MkError(st, "mk_moe_ep_sim")

        ems = statistics.mean(g.timed(ep_once, steps_x, 3))
        line["ep_sim"] = {"ranks": ranks, "ms": ems, "tflops": w.flop / (ems / 1e3) / 1e12,
                          "vs_single_device_with_combine": cms / ems,
                          "workspace_bytes": mk.mk_ep_workspace_size(w.T, w.H, w.F, w.E, w.k, ranks)}
        mk.mk_release_workspace()
        # end to end through the host-buffer entry point
        xh = torch.from_numpy(x_np.view(np.int16)).pin_memory()
        lh = torch.from_numpy(l_np).pin_memory()
        yh = torch.empty((w.rows, w.F), dtype=torch.int16).pin_memory()
        sh = torch.empty(w.rows, dtype=torch.int32).pin_memory()
        oh = torch.empty(w.E + 1, dtype=torch.int32).pin_memory()
        gh = torch.empty(w.rows, dtype=torch.float32).pin_memory()
        e2e_steps = max(3, min(args.steps, 30))
        et = []
        for i in range(args.warmup + e2e_steps):
            g.flush.fill_(1)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            st = mk.mk_moe_dispatch_gemm_host(xh, lh, w.T, w.H, w.E, w.k, W, w.F, yh, sh, oh, gh, stream, cfg)
            t1 = time.perf_counter()
            if st != mk.MK_OK:
                raise mk.MkError(st, "mk_moe_dispatch_gemm_host")
            if i >= args.warmup:
                et.append(t1 - t0)
        e2e_s = reduce_max(statistics.mean(et), world)
        line["e2e"] = {"value": whole_job_tflops(w.flop, world, e2e_s), "unit": UNIT,
                       "h2d_bytes_per_step": x_np.nbytes + l_np.nbytes,
                       "d2h_bytes_per_step": yh.numel() * 2 + sh.numel() * 4 + oh.numel() * 4 + gh.numel() * 4,
                       "ms_per_step": e2e_s * 1e3, "api": "mk_moe_dispatch_gemm_host (pinned host buffers)"}
        del xh, lh, yh, sh, oh, gh
        if rank == 0 and world == 1:
            line["cpu_baseline"] = {k: v for k, v in oracle_sample(w, args.cpu_seconds, (x_np, l_np)).items()
                                    if k != "sample_seconds"}
        # every workload, one at a time (one GPU only: under torchrun each rank
        # would repeat the whole set)
        wanted = [] if args.configs.strip().lower() == "none" else [int(c) for c in args.configs.split(",") if c]
        if world == 1 and args.experts_div == 1 and args.h_div == 1 and wanted:
            per = {}
            for cid in wanted:
                wc = synth.WORKLOADS[cid]
                if cid == args.config:
                    rec = measure_workload(g, wc, args, peaks, peaks_src, clocks, (x_np, l_np, x, logits, W),
                                           cpu_budget=0.0, headline_ms=(ms, clk))
                    rec["cpu_baseline"] = line["cpu_baseline"]
                    rec["headline"] = True
                else:
                    rec = measure_workload(g, wc, args, peaks, peaks_src, clocks,
                                           cpu_budget=args.cpu_seconds_per_config)
                    mk.mk_release_workspace()
                    torch.cuda.empty_cache()
                per[wc.describe()] = rec
            line["per_config"] = per
    clocks.stop()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


TRACE_PHASES = {0: "cta_start", 1: "routing_done", 2: "routing_barrier", 3: "scatter_done", 4: "scatter_barrier",
                5: "gather_done", 6: "gemm_start", 7: "gemm_end", 8: "combine_barrier", 9: "combine_done",
                10: "first_mma", 11: "last_mma", 15: "cta_exit"}


def run_trace(args):
    """Phase timeline of the fused launch per workload: for each traced
    stamp, the earliest, median and latest CTA in µs after the first CTA
    started (medians over 5 traced launches), and the CTAs that reached it."""
    g = Gpu(0)
    mk, torch = g.mk, g.torch
    wanted = [int(c) for c in args.configs.split(",") if c] if args.configs.strip().lower() != "none" else []
    out_all = {}
    for wid in wanted:
        w = synth.WORKLOADS[wid]
        ch = synth._streams(w)
        x, logits, W = g.upload(synth.make_x(w, ch), synth.make_logits(w, ch), synth.make_w(w))
        out = mk.alloc_outputs(w.T, w.F, w.E, w.k, device=g.dev)
        mode = mk.MK_MODE_DISPATCH_ONLY if args.dispatch_only else mk.MK_MODE_FUSED
        cfg = mk.make_config(mode=mode, trace=1)
        runs = []
        for rep in range(8):
            g.flush.fill_(1)
            st = mk.mk_moe_dispatch_gemm_ex(x, logits, w.T, w.H, w.E, w.k, W, w.F, out["y_sorted"], out["src_index"],
                                            out["expert_offsets"], out["gate_w"], g.stream, cfg)
            if st != mk.MK_OK:
                raise mk.MkError(st, "mk_moe_dispatch_gemm_ex")
            torch.cuda.synchronize()
            info = mk.mk_last_launch_info()
            tr = mk.mk_read_trace(w.T, w.H, w.E, w.k, info["grid_ctas"], stream=g.stream).astype(np.int64)
            if rep < 3:
                continue
            t0 = tr[:, 0][tr[:, 0] > 0].min()
            row = {}
            for slot, name in TRACE_PHASES.items():
                v = tr[:, slot]
                v = (v[v > 0] - t0) / 1e3
                if len(v):
                    row[name] = [float(v.min()), float(np.median(v)), float(v.max()), int(len(v))]
            runs.append(row)
        st = mk.mk_get_status(g.stream)
        if st != mk.MK_OK:
            raise mk.MkError(st, "device status")
        summary = {}
        for name in TRACE_PHASES.values():
            vals = [r[name] for r in runs if name in r]
            if vals:
                summary[name] = [round(float(np.median([v[i] for v in vals])), 1) for i in range(3)] + [vals[0][3]]
        out_all[w.describe()] = {"dispatch_ctas": info["dispatch_ctas"], "grid_ctas": info["grid_ctas"],
                                 "mode": "dispatch only" if args.dispatch_only else "fused", "phases_us": summary}
        del x, logits, W, out
        mk.mk_release_workspace()
        torch.cuda.empty_cache()
    print(json.dumps({"trace": out_all, "unit": "µs after the first CTA started: [earliest, median, latest CTA, CTAs]"}),
          flush=True)
    return 0


def main(argv=None):
    args = parse_args(argv)
    w = reduced_hidden(reduced_workload(synth.WORKLOADS[args.config], args.experts_div), args.h_div)
    if args.impl == "reference":
        return run_reference(args, w)
    if args.trace:
        return run_trace(args)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
