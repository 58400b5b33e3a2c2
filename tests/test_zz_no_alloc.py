"""The allocation-free entry point against the allocating one.

mk_moe_dispatch_gemm_noalloc serves callers that may not allocate device
memory while they run this operation (a host framework that owns the
device-memory budget, or a latency-critical decode loop); it works in one
fixed static device array instead of a workspace.  Two calls in a row, on
different problems, must each give what mk_moe_dispatch_gemm gives -- the
second call finds the first call's leftovers in the shared array.  Problems
that do not fit the array are refused without a launch.

This file sorts last so that a run stopping at the first failure has run
every other test first; it also passes alone in a fresh process.
"""
import numpy as np
import pytest

import moe_token_dispatch_persistent_gb300 as mk
from moe_token_dispatch_persistent_gb300 import synth

import gpu_util as gu

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from moe_token_dispatch_persistent_gb300 import build

    build.build()


def _problem(T, H, F, E, k, seed):
    rng = np.random.default_rng(seed)
    x = synth.f32_to_bf16_bits(rng.standard_normal((T, H), dtype=np.float32))
    W = synth.f32_to_bf16_bits(rng.standard_normal((E, H, F), dtype=np.float32) / np.float32(np.sqrt(H)))
    l = rng.standard_normal((T, E), dtype=np.float32)
    return gu.to_device(x, l, W)


def _run(fn, x, l, W, k):
    T, H = x.shape
    E, _, F = W.shape
    out = mk.alloc_outputs(T, F, E, k)
    st = fn(x, l, T, H, E, k, W, F, out["y_sorted"], out["src_index"], out["expert_offsets"], out["gate_w"])
    assert st == mk.MK_OK, mk.mk_status_string(st)
    assert mk.mk_get_status() == mk.MK_OK
    return dict(y=out["y_sorted"].float().cpu().numpy(), src_index=out["src_index"].cpu().numpy(),
                expert_offsets=out["expert_offsets"].cpu().numpy(), gate_w=out["gate_w"].cpu().numpy())


def test_noalloc_matches_allocating_entry_point_on_two_calls_in_a_row():
    w1 = synth.WORKLOADS[1]
    problems = [gu.to_device(*synth.make_inputs(w1)) + (w1.k,), _problem(900, 512, 320, 64, 8, seed=77) + (8,)]
    for x, l, W, k in problems:  # two calls in a row on the shared array
        got = _run(mk.mk_moe_dispatch_gemm_noalloc, x, l, W, k)
        want = _run(mk.mk_moe_dispatch_gemm, x, l, W, k)
        gu.assert_routing_exact(got, want)
        np.testing.assert_array_equal(got["gate_w"], want["gate_w"])
        assert gu.rel_inf(got["y"], want["y"].astype(np.float64)) <= gu.Y_TOL[mk.MK_OUT_BF16]


def test_noalloc_refuses_problems_larger_than_its_array():
    w2 = synth.WORKLOADS[2]  # needs ~67 MB of staged rows plus tables
    assert mk.mk_workspace_size(w2.T, w2.H, w2.F, w2.E, w2.k) > mk.MK_NOALLOC_SCRATCH_BYTES
    st = mk.mk_moe_dispatch_gemm_noalloc(16, 16, w2.T, w2.H, w2.E, w2.k, 16, w2.F, 16, 16, 16, 16)
    assert st == mk.MK_ERR_WORKSPACE
