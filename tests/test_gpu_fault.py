"""Failure detection without a GPU fault: the host asks the kernel to withhold
one tile's readiness flag (MK_FAULT_DROP_TILE_FLAG); the compute role's
bounded wait on it runs out after a short spin limit, the kernel records a
timeout and every CTA returns.  The status call reports MK_ERR_TIMEOUT, and
the next call on the same workspace is correct again.  Nothing traps."""
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
    yield
    mk.mk_release_workspace()


def test_withheld_tile_flag_times_out_and_recovers():
    w = synth.WORKLOADS[1]
    x, l, W = synth.make_inputs(w)
    xd, ld, Wd = gu.to_device(x, l, W)
    out = mk.alloc_outputs(w.T, w.F, w.E, w.k)
    cfg = mk.make_config(debug_fault=mk.MK_FAULT_DROP_TILE_FLAG, spin_limit_ns=50_000_000)
    st = mk.mk_moe_dispatch_gemm_ex(xd, ld, w.T, w.H, w.E, w.k, Wd, w.F, out["y_sorted"], out["src_index"],
                                    out["expert_offsets"], out["gate_w"], None, cfg)
    assert st == mk.MK_OK  # the launch itself is fine; the failure is reported by status
    assert mk.mk_get_status() == mk.MK_ERR_TIMEOUT
    assert mk.mk_last_error_detail()["site"] == 4  # waiting on a tile's readiness flag
    assert mk.mk_get_status() == mk.MK_OK  # reading the status cleared it
    # the workspace was left consistent: a normal call now matches the oracle
    ref = gu.oracle_reference(x, l, W, w.k)
    g = gu.run_gpu(xd, ld, Wd, w.k)
    gu.assert_routing_exact(g, ref)
    gu.assert_y(g, ref, mk.MK_OUT_BF16)
