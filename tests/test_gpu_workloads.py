"""The five seeded workloads at full size, in the launch configuration the
benchmark times (fused, default role split).  Routing, offsets, src_index and
gates are compared in full; y_sorted on sampled rows the oracle computes one
by one (first and last row of every active expert plus random rows)."""
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
    yield
    mk.mk_release_workspace()


@pytest.mark.parametrize("wid", [1, 2, 3, 4, 5])
def test_workload_full_size(wid):
    w = synth.WORKLOADS[wid]
    x, l, W = synth.make_inputs(w)
    orc = Oracle()
    idx, gate = orc.route(l, w.k)
    offsets, src, gw = orc.dispatch(idx, gate, w.E)
    xd, ld, Wd = gu.to_device(x, l, W)
    del W
    g = gu.run_gpu(xd, ld, Wd, w.k)
    ref = dict(expert_offsets=offsets, src_index=src, gate_w=gw)
    gu.assert_routing_exact(g, ref)
    gu.assert_gates(g, ref)
    rows = gu.sample_rows(offsets, 48, np.random.default_rng(wid), w.rows)
    # fp64 products of the sampled rows need only the experts they touch
    experts = sorted({int(np.searchsorted(offsets, r, side="right") - 1) for r in rows})
    yref = np.zeros((rows.size, w.F))
    for e in experts:
        sel = np.where((rows >= offsets[e]) & (rows < offsets[e + 1]))[0]
        We = synth.make_w_expert(w, e)
        # a one-expert view keeps the oracle call small: rows of expert e only
        off1 = np.array([0, offsets[e + 1] - offsets[e]], dtype=np.int32)
        src1 = src[offsets[e]:offsets[e + 1]]
        yref[sel] = orc.expert_rows(x, We[None], w.k, off1, src1, rows[sel] - offsets[e])
    err = gu.rel_inf(g["y"][rows], yref)
    assert err <= gu.Y_TOL[mk.MK_OUT_BF16], f"{w.name}: rel-inf {err:.3e}"
