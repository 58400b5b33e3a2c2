"""Host logic of bench.py that needs no GPU: the clock samplers keep only the
samples taken inside the timed region, the reference arm prints the contract's
line with the same config as ours, and the roofline picks the workload's bound."""
import datetime
import os
import subprocess
import sys
import tempfile

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _line(ts, sm, reasons=("Not Active",) * 4):
    stamp = datetime.datetime.fromtimestamp(ts).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    return ", ".join([stamp, "0", str(sm), "2070", "900.00", "0x0", *reasons]) + "\n"


def _smi_with(lines, t0, t1):
    """An nvidia-smi sampler whose output file already holds ``lines``."""
    s = bench.SmiClocks.__new__(bench.SmiClocks)
    fd, s.path = tempfile.mkstemp(suffix=".csv")
    os.close(fd)
    with open(s.path, "w") as f:
        f.writelines(lines)
    s.fh = open(os.devnull, "w")
    s.proc = object()  # stands for the running nvidia-smi
    s.t0, s.t1, s.ok = t0, t1, True
    return s


def test_smi_samples_outside_the_timed_region_are_dropped():
    t0 = 1_800_000_000.0
    lines = [_line(t0 - 1.0, 345, ("Not Active", "Not Active", "Not Active", "Active")),  # idle, before
             _line(t0 + 0.1, 2070), _line(t0 + 0.2, 2055),
             _line(t0 + 0.3, 2040, ("Not Active", "Not Active", "Not Active", "Active")),
             _line(t0 + 5.0, 600, ("Active", "Not Active", "Not Active", "Not Active"))]  # after
    c = _smi_with(lines, t0, t0 + 1.0).region()
    assert c["samples_in_timed_region"] == 3 and c["samples"] == 3
    assert c["sm_mhz"] == 2055 and c["sm_max_mhz"] == 2070
    assert c["reasons"] == ["sw_power_cap"]  # the hw_slowdown after the region is not counted


def test_smi_region_without_samples_reports_none():
    t0 = 1_800_000_000.0
    c = _smi_with([_line(t0 - 2.0, 1900), _line(t0 - 1.0, 2000)], t0, t0 + 0.001).region()
    assert c["samples_in_timed_region"] == 0 and c["sm_mhz"] is None


def test_smi_malformed_lines_are_skipped():
    t0 = 1_800_000_000.0
    c = _smi_with(["garbage\n", "[N/A], 0\n", _line(t0 + 0.5, 2070)], t0, t0 + 1.0).region()
    assert c["samples"] == 1 and c["sm_mhz"] == 2070


def _nvml_with(samples, t0, t1):
    import threading

    s = bench.NvmlClocks.__new__(bench.NvmlClocks)
    s.ok, s.lock, s.samples, s.t0, s.t1, s.max_mhz, s.period = True, threading.Lock(), samples, t0, t1, 2070.0, 5e-4
    return s


def test_nvml_region_keeps_its_samples_and_decodes_reasons():
    """Reason bits follow nvml.h: 0x4 sw power cap, 0x8 hw slowdown, 0x20 sw
    thermal, 0x40 hw thermal; other bits (idle 0x1) are not throttling."""
    t0 = 100.0
    smp = [(99.0, 400.0, 0x1), (100.001, 2070.0, 0x0), (100.002, 1980.0, 0x4), (100.003, 2040.0, 0x0),
           (100.5, 900.0, 0x8 | 0x40)]
    c = _nvml_with(smp, t0, t0 + 0.01).region()
    assert c["samples_in_timed_region"] == 3 and c["sm_mhz"] == 2040.0 and c["sm_mhz_min"] == 1980.0
    assert c["reasons"] == ["sw_power_cap"] and c["sm_max_mhz"] == 2070.0
    c = _nvml_with(smp, 100.4, 100.6).region()
    assert c["reasons"] == ["hw_slowdown", "hw_thermal_slowdown"]


def test_nvml_unavailable_is_reported():
    s = bench.NvmlClocks.__new__(bench.NvmlClocks)
    s.ok = False
    c = s.region()
    assert c["samples_in_timed_region"] == 0 and c["reasons"] == ["nvml unavailable"]


def test_both_arms_print_the_same_config():
    """The reference arm and ours build ``config`` with the same function, so
    the two lines carry the same keys and values for the same workload."""
    w = bench.synth.WORKLOADS[2]
    c = bench.bench_config(w)
    assert set(c) == {"workload", "T", "H", "F", "E", "k", "seed", "l2"}
    assert c["workload"] == w.describe() and "flush" in c["l2"]


def test_reference_arm_prints_one_json_line():
    """`bench.py --impl reference` times the CPU oracle (no GPU needed) and
    prints the contract's line with impl, cpu_baseline and e2e."""
    import json

    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "1",
                          "--steps", "2", "--warmup", "1"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 1 and d["n_gpus"] == 1
    assert d["value"] > 0 and d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"] and d["e2e"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"] == bench.bench_config(bench.synth.WORKLOADS[1])
    # ms_per_step is the measured time of a step (a bounded sample), not an extrapolation
    assert 0 < d["ms_per_step"] < 600e3
    assert d["cpu_baseline"]["estimated"] is True and d["cpu_baseline"]["full_workload_seconds_estimated"] > 0


def test_kernel_code_digest_ignores_comments_only(tmp_path, monkeypatch):
    a = tmp_path / "a.cu"
    a.write_text("int f(int x) {  // doubles\n    return 2 * x; /* twice */\n}\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    d0 = bench.kernel_code_digest(["a.cu"])
    a.write_text("// a header comment\nint f(int x) {\n  return 2 * x;   // still twice\n}\n")
    assert bench.kernel_code_digest(["a.cu"]) == d0
    a.write_text("int f(int x) {\n  return 3 * x;\n}\n")
    assert bench.kernel_code_digest(["a.cu"]) != d0


def test_roofline_bound_follows_the_workload():
    """The Mixtral-like, skewed and imbalanced layers are bound by the bf16
    peak; the decode layer (a few rows per expert) by streaming its weights."""
    import numpy as np

    peaks = dict(bench.FALLBACK_PEAKS)
    for wid, bound in ((2, "tensor"), (3, "tensor"), (5, "tensor"), (4, "hbm")):
        w = bench.synth.WORKLOADS[wid]
        # experts that receive rows: only their weights are compulsory bytes
        top = np.argsort(-bench.synth.make_logits(w), axis=1, kind="stable")[:, :w.k]
        active = int((np.bincount(top.ravel(), minlength=w.E) > 0).sum())
        assert bench.roofline_bound(w, active, peaks) == bound, w.name
    # all 256 experts of the skewed layer active would make it weight-bound
    assert bench.roofline_bound(bench.synth.WORKLOADS[3], 256, peaks) == "hbm"


def test_reduced_workload_keeps_rows_per_expert():
    w = bench.synth.WORKLOADS[3]
    r = bench.reduced_workload(w, 8)
    assert (r.T, r.E) == (w.T // 8, w.E // 8) and (r.H, r.F, r.k, r.seed, r.kind) == (w.H, w.F, w.k, w.seed, w.kind)
    assert r.rows / r.E == w.rows / w.E and r.name != w.name
    assert bench.reduced_workload(w, 1) is w
    import pytest

    with pytest.raises(SystemExit):
        bench.reduced_workload(bench.synth.WORKLOADS[2], 2)  # 4 experts: too few


def test_reference_arm_on_a_reduced_case():
    """`--experts-div` names the reduced layer in the line's config."""
    import json

    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "3",
                          "--experts-div", "8", "--steps", "1", "--warmup", "0"], capture_output=True, text=True,
                         timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    d = json.loads([ln for ln in out.stdout.splitlines() if ln.strip().startswith("{")][0])
    assert d["config"]["workload"].startswith("fine_grained_skewed_experts_div_8(T=1024,H=7168,F=2048,E=32,k=8")
    assert d["config"]["E"] == 32 and d["config"]["T"] == 1024 and d["value"] > 0


def test_reduced_hidden_keeps_the_routing():
    """`--h-div` shrinks only H: the logits, hence every expert's rows, are
    those of the full layer (the skewed layer keeps its 40 active experts)."""
    import numpy as np
    import pytest

    w = bench.synth.WORKLOADS[3]
    r = bench.reduced_hidden(w, 8)
    assert (r.T, r.E, r.k, r.F, r.seed, r.kind) == (w.T, w.E, w.k, w.F, w.seed, w.kind) and r.H == w.H // 8
    assert np.array_equal(bench.synth.make_logits(r), bench.synth.make_logits(w))
    assert bench.reduced_hidden(w, 1) is w
    with pytest.raises(SystemExit):
        bench.reduced_hidden(bench.synth.WORKLOADS[1], 16)  # 512 / 16 = 32: not a multiple of 64


def test_trace_mode_is_a_separate_output():
    """--trace prints a phase timeline instead of the bench line; the default
    run (what the driver launches) never traces."""
    assert bench.parse_args(["--trace"]).trace is True
    assert bench.parse_args([]).trace is False
    assert bench.TRACE_PHASES[10] == "first_mma" and bench.TRACE_PHASES[15] == "cta_exit"
