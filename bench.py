#!/usr/bin/env python
"""Benchmark of the fused MoE dispatch + expert GEMM on GB300.

One step = one pass of the whole path (router top-k, histogram + scan,
gather into expert-contiguous tiles, expert GEMM) over one batch of the
seeded synthetic workload, through the C ABI.  Default workload: the
Mixtral-like layer (T=4096, H=4096, F=14336, E=8, top-2, seed 1).

Timing: W warm-up steps, then K timed steps; every step is bracketed by CUDA
events on the launching stream, with a 256 MiB write (larger than L2)
between steps outside the events; the timed region is bracketed by a
barrier and a device synchronise; the max over ranks is taken.  Under
torchrun every rank runs its own batch (weak scaling, no data-path
collective).

``--impl reference`` times the CPU oracle instead (rank 0 only).
Prints ONE JSON line on rank 0.
"""
from __future__ import annotations

import argparse
import datetime
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from moe_token_dispatch_persistent_gb300 import synth  # noqa: E402

METRIC = "fused dispatch+grouped-GEMM TFLOP/s (% bf16 peak) and dispatch GB/s (% HBM)"
UNIT = "TFLOP/s"
FLUSH_BYTES = 256 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=2, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--dispatch-ctas", type=int, default=0)
    ap.add_argument("--n-group", type=int, default=0)
    ap.add_argument("--no-extras", action="store_true", help="skip unfused / dispatch-only / e2e / cpu legs")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="budget of the CPU-baseline sample")
    ap.add_argument("--dispatch-only", action="store_true",
                    help="time the dispatch role alone (routing, scan, gather; no GEMM) as the main loop, in GB/s")
    ap.add_argument("--experts-div", type=int, default=1,
                    help="small case for profiler captures: E/D experts and T/D tokens, H, F, k and the value "
                         "recipe unchanged (not a bench workload)")
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
    committed ncu capture of this workload, or None when there is none or the
    kernel code changed since it was taken."""
    try:
        with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
            rec = json.load(f).get(workload_name)
    except (OSError, ValueError):
        return None
    if not rec:
        return None
    try:
        digest = kernel_code_digest(rec["kernel_sources"])
    except OSError:
        return None
    return rec["bytes_per_launch"] if digest == rec["kernel_code_sha256"] else None


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


def roofline_bound(w: synth.Workload, active_experts: int, peaks) -> str:
    """The bound of the fused launch: the larger of the time its FLOPs take
    at the bf16 peak and the time its compulsory bytes take at the HBM peak."""
    t_tensor = w.flop / (float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])) * 1e12)
    t_hbm = compulsory_bytes(w, active_experts) / (float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])) * 1e9)
    return "tensor" if t_tensor >= t_hbm else "hbm"


def workload_config(w: synth.Workload, extra=None):
    c = {"workload": w.describe(), "T": w.T, "H": w.H, "F": w.F, "E": w.E, "k": w.k, "seed": w.seed,
         "l2": "flushed between timed steps (256 MiB write, outside the events)"}
    if extra:
        c.update(extra)
    return c


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


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 50

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None
        self.t0 = self.t1 = None

    def start(self):
        """Start sampling; returns once the first sample is written (or after 5 s)."""
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(self.gpu), "-lms", str(self.PERIOD_MS)], stdout=self.fh,
                                         stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
            return
        deadline = time.time() + 5.0
        while time.time() < deadline and os.path.getsize(self.path) == 0 and self.proc.poll() is None:
            time.sleep(0.02)

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def stop(self):
        """Median SM clock and the throttle reasons of the samples taken between
        mark_start and mark_end (all samples if none fell inside)."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
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
        os.unlink(self.path)
        inside = [r for r in rows if self.t0 is not None and self.t1 is not None and self.t0 <= r[0] <= self.t1]
        use = inside or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({nm for r in use for nm, v in zip(names, r[3]) if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[1] for r in use) if use else None,
                "sm_max_mhz": max(r[2] for r in use) if use else None, "reasons": reasons,
                "samples": len(use), "samples_in_timed_region": len(inside), "period_ms": self.PERIOD_MS}


# ------------------------------------------------------------ reference --

_WE_CACHE = {}


def oracle_sample(w: synth.Workload, budget_s: float, inputs=None):
    """Time the CPU oracle on a bounded sample of workload ``w``.

    The full routing + dispatch of all T tokens is timed once; the fp64
    expert product is timed on a sample of sorted rows sized to the budget.
    The full-workload time is estimated as t_routing + t_row * T*k, and the
    value is the workload's FLOPs over that estimate.
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
    t_row = t_rows / n
    est = t_route + t_row * w.rows
    return {
        "value": w.flop / est / 1e12,
        "unit": UNIT,
        "cores": orc.num_threads(),
        "kind": "oracle",
        "sample": (f"routing+dispatch of all {w.T} tokens ({t_route:.3f} s) + fp64 product of {n} sorted rows "
                   f"({t_rows:.2f} s); full-workload time estimated as t_route + t_row*{w.rows} = {est:.1f} s"),
        "seconds_estimated_full": est,
    }


def run_reference(args, w):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    per_step_budget = max(0.05, min(2.0, 120.0 / max(1, args.steps + args.warmup)))
    times, cb = [], None
    ch = synth._streams(w)
    inputs = (synth.make_x(w, ch), synth.make_logits(w, ch))
    for i in range(args.warmup + args.steps):
        r = oracle_sample(w, per_step_budget, inputs)
        if i >= args.warmup:
            times.append(r["seconds_estimated_full"])
            cb = r
    est = statistics.mean(times)
    value = w.flop / est / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": est * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
        "config": workload_config(w, {"l2": "n/a (CPU)"}),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cb["cores"], "kind": "oracle", "sample": cb["sample"]},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ ours --

def dispatch_bytes(w: synth.Workload) -> int:
    """Algorithmic bytes of the dispatch role: logits read, token rows read and
    written to the staging tiles, src_index / gate_w written, offsets."""
    return w.T * w.E * 4 + 2 * w.rows * w.H * 2 + w.rows * 8 + (w.E + 1) * 4


TILE_NAMES = {1: "128-row", 2: "256-row on SM pairs", 3: "256-row (two accumulators per SM)"}


def compulsory_bytes(w: synth.Workload, active_experts: int) -> int:
    """x + logits + active experts' W + y_sorted (bf16) + src_index + gate_w + offsets."""
    return (w.T * w.H * 2 + w.T * w.E * 4 + active_experts * w.H * w.F * 2 + w.rows * w.F * 2 + w.rows * 8
            + (w.E + 1) * 4)


def run_ours(args, w):
    import torch

    import moe_token_dispatch_persistent_gb300 as mk
    from moe_token_dispatch_persistent_gb300 import build

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    build.build()
    dev = torch.device("cuda", torch.cuda.current_device())
    peaks, peaks_src = load_peaks()

    # inputs: each rank its own batch of tokens (seed offset), same expert weights
    wr = synth.Workload(w.name, w.T, w.H, w.F, w.E, w.k, w.seed + 1000 * rank, w.kind) if rank else w
    ch = synth._streams(wr)
    x_np, l_np = synth.make_x(wr, ch), synth.make_logits(wr, ch)
    W_np = synth.make_w(w)
    x = torch.from_numpy(x_np.view(np.int16)).view(torch.bfloat16).to(dev)
    logits = torch.from_numpy(l_np).to(dev)
    W = torch.from_numpy(W_np.view(np.int16)).view(torch.bfloat16).to(dev)
    del W_np
    out = mk.alloc_outputs(w.T, w.F, w.E, w.k, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    cfg = mk.make_config(dispatch_ctas=args.dispatch_ctas, n_group=args.n_group,
                         mode=mk.MK_MODE_DISPATCH_ONLY if args.dispatch_only else mk.MK_MODE_FUSED)

    combined = torch.empty((w.T, w.F), dtype=torch.bfloat16, device=dev)

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

    def timed(c, steps, warmup, combine=False):
        for _ in range(warmup):
            flush.fill_(1)
            call(c, combine)
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for a, b in evs:
            flush.fill_(1)
            a.record(stream)
            call(c, combine)
            b.record(stream)
        torch.cuda.synchronize()
        st = mk.mk_get_status(stream)
        if st != mk.MK_OK:
            raise mk.MkError(st, "device status")
        return [a.elapsed_time(b) for a, b in evs]

    # headline: fused path
    sampler = ClockSampler(int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[local])
                           if os.environ.get("CUDA_VISIBLE_DEVICES") else local)
    for _ in range(args.warmup):
        flush.fill_(1)
        call(cfg)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler.start()
    launches_before = 0
    sampler.mark_start()
    ms = timed(cfg, args.steps, 0)
    torch.cuda.synchronize()
    sampler.mark_end()
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    info = mk.mk_last_launch_info()
    gpu_launches = args.steps * info["launches"] + launches_before
    ms_mean = statistics.mean(ms)
    ms_max = reduce_max(ms_mean, world)
    value = whole_job_tflops(w.flop, world, ms_max / 1e3)
    offs = out["expert_offsets"].cpu().numpy()
    active = int((np.diff(offs) > 0).sum())

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
                "traffic": None, "algorithmic_bytes": db}
    elif roofline_bound(w, active, peaks) == "hbm":
        # weight streaming (few rows per expert): compulsory bytes against HBM
        cb = compulsory_bytes(w, active)
        achieved = cb / (ms_mean / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                "peak_source": f"hbm_gbs, {peaks_src}", "kernel": "mk_fused_kernel",
                "traffic": ncu_traffic(w.name), "compulsory_bytes": cb,
                "tflops": w.flop / (ms_mean / 1e3) / 1e12}
    else:
        achieved = w.flop / (ms_mean / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "peak_source": f"bf16_tflops (burst), {peaks_src}",
                "kernel": "mk_fused_kernel", "traffic": ncu_traffic(w.name),
                "compulsory_bytes": compulsory_bytes(w, active)}
    line = {
        "metric": METRIC, "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(w, {"mode": "dispatch only" if args.dispatch_only else "fused persistent",
                                      "grid_ctas": info["grid_ctas"],
                                      "dispatch_ctas": info["dispatch_ctas"], "n_group": info["n_group"],
                                      "tiles": TILE_NAMES.get(info["mma_pair"], str(info["mma_pair"])),
                                      "active_experts": active}),
        "roofline": roof,
        "gpu_launches": gpu_launches,
        "clocks": clocks,
        "ms_per_step_min": min(ms), "ms_per_step_median": statistics.median(ms),
    }

    if not (args.no_extras or args.dispatch_only):
        # dispatch role alone (routing + gather), GB/s against HBM
        dcfg = mk.make_config(mode=mk.MK_MODE_DISPATCH_ONLY)
        dms = statistics.mean(timed(dcfg, min(args.steps, 50), 3))
        db = dispatch_bytes(w)
        line["dispatch"] = {"gbs": db / (dms / 1e3) / 1e9, "frac_hbm": db / (dms / 1e3) / 1e9 / hbm,
                            "ms": dms, "bytes": db, "peak_gbs": hbm}
        # the same steps as four launches (host-driven baseline)
        ucfg = mk.make_config(mode=mk.MK_MODE_UNFUSED)
        ums = statistics.mean(timed(ucfg, min(args.steps, 50), 3))
        line["unfused"] = {"ms_per_step": ums, "tflops": w.flop / (ums / 1e3) / 1e12,
                           "fused_speedup": ums / ms_mean, "launches_per_step": 4}
        # the MoE layer's combine (gated sum of each token's expert rows)
        cms = statistics.mean(timed(cfg, min(args.steps, 50), 3, combine=True))
        cums = statistics.mean(timed(ucfg, min(args.steps, 50), 3, combine=True))
        cbytes = w.rows * w.F * 2 + w.T * w.F * 2 + w.rows * 8  # y_sorted read, out written, rows + gates
        line["combine"] = {"fused_ms": cms, "unfused_ms": cums, "fused_speedup": cums / cms,
                           "added_ms": cms - ms_mean, "bytes": cbytes,
                           "added_gbs": cbytes / max(cms - ms_mean, 1e-6) * 1e3 / 1e9}
        # the gated (SwiGLU) expert FFN: two projections, one tensor-core pass per item
        w3 = synth.Workload(w.name, w.T, w.H, w.F, w.E, w.k, w.seed + 7, w.kind)
        W3 = torch.from_numpy(synth.make_w(w3).view(np.int16)).view(torch.bfloat16).to(dev)

        def gated_once():
            st = mk.mk_moe_dispatch_gated(x, logits, w.T, w.H, w.E, w.k, W, W3, w.F, out["y_sorted"],
                                          out["src_index"], out["expert_offsets"], out["gate_w"], stream, cfg)
            if st != mk.MK_OK:
                raise mk.MkError(st, "mk_moe_dispatch_gated")

        for _ in range(3):
            flush.fill_(1)
            gated_once()
        gms_list = []
        for _ in range(min(args.steps, 50)):
            flush.fill_(1)
            a_ev, b_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a_ev.record(stream)
            gated_once()
            b_ev.record(stream)
            gms_list.append((a_ev, b_ev))
        torch.cuda.synchronize()
        if mk.mk_get_status(stream) != mk.MK_OK:
            raise RuntimeError("gated path: device error")
        gms = statistics.mean(a.elapsed_time(b) for a, b in gms_list)
        line["gated"] = {"ms": gms, "tflops": 2 * w.flop / (gms / 1e3) / 1e12,
                         "frac_bf16": 2 * w.flop / (gms / 1e3) / 1e12 / peak}
        del W3
        # token rows straight from x (no staging rows): the same product
        dgcfg = mk.make_config(dispatch_ctas=args.dispatch_ctas, n_group=args.n_group, gather=mk.MK_GATHER_DIRECT)
        dgms = statistics.mean(timed(dgcfg, min(args.steps, 50), 3))
        line["direct_gather"] = {
            "ms": dgms, "tflops": w.flop / (dgms / 1e3) / 1e12, "frac_bf16": w.flop / (dgms / 1e3) / 1e12 / peak,
            "vs_staged": ms_mean / dgms,
            "workspace_bytes": mk.mk_workspace_size(w.T, w.H, w.F, w.E, w.k, dgcfg),
            "staged_workspace_bytes": mk.mk_workspace_size(w.T, w.H, w.F, w.E, w.k, cfg)}
        # expert parallelism simulated on this GPU: the most ranks (<= 8) that divide E
        ranks = max(r for r in (1, 2, 4, 8) if w.E % r == 0)
        ep_once = lambda c: mk.mk_moe_ep_sim(x, logits, w.T, w.H, w.E, w.k, W, w.F, ranks, out["y_sorted"],  # noqa: E731
                                             out["src_index"], out["expert_offsets"], out["gate_w"], combined,
                                             stream, c)
        for _ in range(3):
            flush.fill_(1)
            if ep_once(cfg) != mk.MK_OK:
                raise RuntimeError("mk_moe_ep_sim refused the configuration")
        ep_evs = []
        for _ in range(min(args.steps, 50)):
            flush.fill_(1)
            a_ev, b_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a_ev.record(stream)
            ep_once(cfg)
            b_ev.record(stream)
            ep_evs.append((a_ev, b_ev))
        torch.cuda.synchronize()
        if mk.mk_get_status(stream) != mk.MK_OK:
            raise RuntimeError("expert-parallel path: device error")
        ems = statistics.mean(a.elapsed_time(b) for a, b in ep_evs)
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
            flush.fill_(1)
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
        if rank == 0 and world == 1:
            line["cpu_baseline"] = {k: v for k, v in oracle_sample(w, args.cpu_seconds, (x_np, l_np)).items()
                                    if k != "seconds_estimated_full"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def main(argv=None):
    args = parse_args(argv)
    w = reduced_workload(synth.WORKLOADS[args.config], args.experts_div)
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
