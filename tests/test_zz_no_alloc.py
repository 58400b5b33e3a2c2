"""The allocation-free entry point against the allocating one and the oracle.

mk_moe_dispatch_gemm_noalloc serves callers that may not allocate device
memory while they run this operation (a host framework that owns the
device-memory budget, or a latency-critical decode loop); it works in one
fixed static device array instead of a workspace.  Calls in a row, on
different problems, must each give exactly what mk_moe_dispatch_gemm gives
(the same kernel on the same inputs: bit for bit), and what the oracle
gives within the usual tolerances; every call after the first finds the
previous call's leftovers in the shared array.  While only these calls run,
the device's free memory does not move.  Problems that do not fit the array
are refused without a launch, and so is tracing.

This file sorts last so that a run stopping at the first failure has run
every other test first; it also passes alone in a fresh process.
"""
import numpy as np
import pytest

import moe_token_dispatch_persistent_gb300 as mk
from moe_token_dispatch_persistent_gb300 import synth
from oracle.oracle import Oracle

import gpu_util as gu

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from moe_token_dispatch_persistent_gb300 import build

    build.build()


def _random_problem(T, H, F, E, k, seed):
    rng = np.random.default_rng(seed)
    x = synth.f32_to_bf16_bits(rng.standard_normal((T, H), dtype=np.float32))
    W = synth.f32_to_bf16_bits(rng.standard_normal((E, H, F), dtype=np.float32) / np.float32(np.sqrt(H)))
    l = rng.standard_normal((T, E), dtype=np.float32)
    return x, l, W, k


def _launch(fn, dev, out):
    x, l, W, k = dev
    T, H = x.shape
    E, _, F = W.shape
    st = fn(x, l, T, H, E, k, W, F, out["y_sorted"], out["src_index"], out["expert_offsets"], out["gate_w"])
    assert st == mk.MK_OK, mk.mk_status_string(st)


def _host(out):
    return {name: t.cpu() for name, t in out.items()}


def test_noalloc_calls_in_a_row_match_the_allocating_path_and_the_oracle():
    problems = [synth.make_inputs(synth.WORKLOADS[1]) + (synth.WORKLOADS[1].k,),
                _random_problem(900, 512, 320, 64, 8, seed=77),
                synth.make_inputs(synth.WORKLOADS[4]) + (synth.WORKLOADS[4].k,)]  # decode: 7168 x 2048, E=256, k=8
    devs = [gu.to_device(x, l, W) + (k,) for x, l, W, k in problems]
    outs = [mk.alloc_outputs(d[0].shape[0], d[2].shape[2], d[2].shape[0], d[3]) for d in devs]
    # no workspace cache entry may serve these calls
    mk.mk_release_workspace()
    # the first call on the device looks the array up (and may load its module)
    _launch(mk.mk_moe_dispatch_gemm_noalloc, devs[0], outs[0])
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    # three problems, then the first again: each call finds the last one's leftovers
    order = [0, 1, 2, 0]
    got = []
    for i in order:
        _launch(mk.mk_moe_dispatch_gemm_noalloc, devs[i], outs[i])
        torch.cuda.synchronize()
        assert mk.mk_get_status() == mk.MK_OK
        got.append(_host(outs[i]))
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"device memory moved during allocation-free calls: {free0 - free1} bytes"

    orc = Oracle()
    for n, i in enumerate(order):
        x, l, W, k = problems[i]
        want_out = mk.alloc_outputs(x.shape[0], W.shape[2], W.shape[0], k)
        _launch(mk.mk_moe_dispatch_gemm, devs[i], want_out)
        torch.cuda.synchronize()
        assert mk.mk_get_status() == mk.MK_OK
        want = _host(want_out)
        # the same kernel on the same inputs: identical bits
        for name in ("y_sorted", "src_index", "expert_offsets", "gate_w"):
            assert torch.equal(got[n][name].view(torch.int16) if name == "y_sorted" else got[n][name],
                               want[name].view(torch.int16) if name == "y_sorted" else want[name]), \
                f"problem {i} (call {n}): {name} differs from the allocating path"
        if n == len(order) - 1:
            continue  # the repeated problem was checked against the oracle on its first call
        ref = orc.full(x, l, W, k)
        g = dict(y=got[n]["y_sorted"].float().numpy(), src_index=got[n]["src_index"].numpy(),
                 expert_offsets=got[n]["expert_offsets"].numpy(), gate_w=got[n]["gate_w"].numpy())
        gu.assert_routing_exact(g, ref)
        gu.assert_gates(g, ref)
        gu.assert_y(g, ref, mk.MK_OUT_BF16)
    mk.mk_release_workspace()


def test_noalloc_refuses_problems_larger_than_its_array():
    w2 = synth.WORKLOADS[2]  # needs ~67 MB of staged rows plus tables
    assert mk.mk_workspace_size(w2.T, w2.H, w2.F, w2.E, w2.k) > mk.MK_NOALLOC_SCRATCH_BYTES
    st = mk.mk_moe_dispatch_gemm_noalloc(16, 16, w2.T, w2.H, w2.E, w2.k, 16, w2.F, 16, 16, 16, 16)
    assert st == mk.MK_ERR_WORKSPACE


def test_noalloc_refuses_tracing():
    """Stamps would land in the array, out of mk_read_trace's reach."""
    w1 = synth.WORKLOADS[1]
    st = mk.mk_moe_dispatch_gemm_noalloc(16, 16, w1.T, w1.H, w1.E, w1.k, 16, w1.F, 16, 16, 16, 16,
                                         cfg=mk.make_config(trace=1))
    assert st == mk.MK_ERR_UNSUPPORTED
