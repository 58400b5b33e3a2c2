"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and
compare every output with the CPU oracle on the same seeded inputs."""
from __future__ import annotations

import numpy as np

import moe_token_dispatch_persistent_gb300 as mk
from moe_token_dispatch_persistent_gb300 import synth
from oracle.oracle import Oracle

GATE_TOL = 2e-6          # fp32 expf vs the oracle's fp64 exp (abs)
Y_TOL = {mk.MK_OUT_BF16: 1e-2, mk.MK_OUT_F32: 1e-4}  # ||Y - Yref||_inf / ||Yref||_inf


def to_device(x_bits, logits, W_bits):
    import torch

    x = torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).view(torch.bfloat16).cuda()
    l = torch.from_numpy(np.ascontiguousarray(logits, dtype=np.float32)).cuda()
    W = torch.from_numpy(np.ascontiguousarray(W_bits).view(np.int16)).view(torch.bfloat16).cuda()
    return x, l, W


def run_gpu(x, l, W, k, cfg=None, out=None):
    """Run through the C ABI; returns numpy copies of the outputs."""
    import torch

    o = mk.moe_dispatch_gemm(x, l, W, k, cfg=cfg, out=out)
    torch.cuda.synchronize()
    y = o["y_sorted"]
    y = y.float().cpu().numpy() if y.dtype == torch.bfloat16 else y.cpu().numpy()
    return dict(y=y, src_index=o["src_index"].cpu().numpy(), expert_offsets=o["expert_offsets"].cpu().numpy(),
                gate_w=o["gate_w"].cpu().numpy())


def oracle_reference(x_bits, logits, W_bits, k, rows=None, orc: Oracle | None = None):
    orc = orc or Oracle()
    return orc.full(x_bits, logits, W_bits, k, rows=rows)


def assert_routing_exact(g, ref):
    np.testing.assert_array_equal(g["expert_offsets"], ref["expert_offsets"])
    np.testing.assert_array_equal(g["src_index"], ref["src_index"])


def assert_gates(g, ref):
    d = np.abs(g["gate_w"].astype(np.float64) - ref["gate_w"].astype(np.float64))
    assert d.max(initial=0.0) <= GATE_TOL, f"gate max abs err {d.max()}"


def rel_inf(y, yref):
    den = np.abs(yref).max(initial=0.0)
    num = np.abs(y.astype(np.float64) - yref).max(initial=0.0)
    return num / den if den > 0 else num


def assert_y(g, ref, out_dtype, rows=None):
    y = g["y"] if rows is None else g["y"][rows]
    err = rel_inf(y, ref["y"])
    assert err <= Y_TOL[out_dtype], f"rel-inf error {err:.3e} > {Y_TOL[out_dtype]}"
    return err


def sample_rows(offsets, n_random, rng, rows_total):
    """First and last row of every non-empty expert plus random rows."""
    s = set()
    for e in range(len(offsets) - 1):
        if offsets[e + 1] > offsets[e]:
            s.add(int(offsets[e]))
            s.add(int(offsets[e + 1] - 1))
    s |= set(rng.integers(0, rows_total, size=n_random).tolist())
    return np.array(sorted(s), dtype=np.int64)


def workload_inputs(w: synth.Workload):
    return synth.make_inputs(w)
