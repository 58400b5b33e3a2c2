"""The direct row gather (the GEMM's producer brings token rows straight
from x; no staging rows) against the oracle, and bit for bit against the
staged path: both feed the same bytes to the same MMA order.  Both forms of
it run every test: 16-byte cp.async by two copy warps (DIRECT) and TMA
tile::gather4, four rows per instruction (GATHER4)."""
import numpy as np
import pytest

import moe_token_dispatch_persistent_gb300 as mk
from moe_token_dispatch_persistent_gb300 import synth

import gpu_util as gu

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

DIRECT = mk.MK_GATHER_DIRECT
ROW_FORMS = pytest.mark.parametrize("rows", [mk.MK_GATHER_DIRECT, mk.MK_GATHER_GATHER4], ids=["cp_async", "gather4"])


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from moe_token_dispatch_persistent_gb300 import build

    build.build()
    yield
    mk.mk_release_workspace()


def _inputs(T, H, F, E, k, seed=0):
    rng = np.random.default_rng(seed)
    x = synth.f32_to_bf16_bits(rng.standard_normal((T, H), dtype=np.float32))
    W = synth.f32_to_bf16_bits(rng.standard_normal((E, H, F), dtype=np.float32) / np.float32(np.sqrt(H)))
    return x, rng.standard_normal((T, E), dtype=np.float32), W


@ROW_FORMS
@pytest.mark.parametrize("mode", [mk.MK_MODE_FUSED, mk.MK_MODE_UNFUSED], ids=["fused", "unfused"])
@pytest.mark.parametrize("out_dtype", [mk.MK_OUT_BF16, mk.MK_OUT_F32], ids=["bf16", "f32"])
def test_direct_tiny(mode, out_dtype, rows):
    w = synth.WORKLOADS[1]
    x, l, W = synth.make_inputs(w)
    ref = gu.oracle_reference(x, l, W, w.k)
    g = gu.run_gpu(*gu.to_device(x, l, W), w.k, cfg=mk.make_config(mode=mode, out_dtype=out_dtype, gather=rows))
    info = mk.mk_last_launch_info()
    assert info["gather"] == rows and info["dispatch_ctas"] == 0
    gu.assert_routing_exact(g, ref)
    gu.assert_gates(g, ref)
    gu.assert_y(g, ref, out_dtype)


@pytest.mark.parametrize("shape", [
    (1, 64, 64, 1, 1),
    (7, 128, 192, 3, 2),
    (129, 256, 320, 5, 3),
    (1000, 512, 256, 64, 8),
    (300, 192, 128, 256, 8),
    (2000, 128, 512, 2, 1),
], ids=lambda s: "x".join(map(str, s)))
@ROW_FORMS
def test_direct_ragged_shapes(shape, rows):
    T, H, F, E, k = shape
    x, l, W = _inputs(T, H, F, E, k, seed=T + E + 3)
    ref = gu.oracle_reference(x, l, W, k)
    g = gu.run_gpu(*gu.to_device(x, l, W), k, cfg=mk.make_config(out_dtype=mk.MK_OUT_F32, gather=rows))
    gu.assert_routing_exact(g, ref)
    gu.assert_y(g, ref, mk.MK_OUT_F32)


@ROW_FORMS
@pytest.mark.parametrize("tiles", [mk.MK_MMA_SINGLE, mk.MK_MMA_WIDE], ids=["128-row", "wide"])
def test_direct_equals_staged_bitwise(rows, tiles):
    x, l, W = gu.to_device(*_inputs(1500, 256, 512, 16, 4, seed=31))
    a = gu.run_gpu(x, l, W, 4, cfg=mk.make_config(gather=mk.MK_GATHER_STAGED, mma_pair=tiles))
    b = gu.run_gpu(x, l, W, 4, cfg=mk.make_config(gather=rows, mma_pair=tiles))
    for key in a:
        np.testing.assert_array_equal(a[key], b[key])


@ROW_FORMS
def test_direct_workspace_has_no_staging_rows(rows):
    T, H, F, E, k = 4096, 4096, 14336, 8, 2
    staged = mk.mk_workspace_size(T, H, F, E, k)
    direct = mk.mk_workspace_size(T, H, F, E, k, mk.make_config(gather=rows))
    assert staged - direct >= T * k * H * 2


@ROW_FORMS
def test_direct_with_combine_and_gated(rows):
    x, l, W = _inputs(700, 256, 256, 8, 2, seed=33)
    _, _, W3 = _inputs(700, 256, 256, 8, 2, seed=34)
    xd, ld, Wd = gu.to_device(x, l, W)
    W3d = gu.to_device(x, l, W3)[2]
    a = mk.moe_layer(xd, ld, Wd, 2, cfg=mk.make_config(gather=mk.MK_GATHER_STAGED))
    b = mk.moe_layer(xd, ld, Wd, 2, cfg=mk.make_config(gather=rows))
    assert torch.equal(a["out"], b["out"]) and torch.equal(a["y_sorted"], b["y_sorted"])
    c = mk.moe_gated(xd, ld, Wd, W3d, 2, cfg=mk.make_config(gather=mk.MK_GATHER_STAGED))
    d = mk.moe_gated(xd, ld, Wd, W3d, 2, cfg=mk.make_config(gather=rows))
    assert torch.equal(c["y_sorted"], d["y_sorted"])


@ROW_FORMS
def test_direct_refuses_sm_pairs(rows):
    T, H, F, E, k = 64, 64, 64, 4, 2
    x, l, W = gu.to_device(*_inputs(T, H, F, E, k))
    o = mk.alloc_outputs(T, F, E, k)
    st = mk.mk_moe_dispatch_gemm_ex(x, l, T, H, E, k, W, F, o["y_sorted"], o["src_index"], o["expert_offsets"],
                                    o["gate_w"], None, mk.make_config(gather=rows, mma_pair=mk.MK_MMA_PAIR))
    assert st == mk.MK_ERR_UNSUPPORTED


@pytest.mark.parametrize("wid", [3, 5])
def test_direct_full_workload_equals_staged(wid):
    """Full-size fine-grained skewed and imbalanced workloads: both direct
    forms and the staged path agree bit for bit."""
    w = synth.WORKLOADS[wid]
    x, l, W = synth.make_inputs(w)
    xd, ld, Wd = gu.to_device(x, l, W)
    del W
    a = gu.run_gpu(xd, ld, Wd, w.k, cfg=mk.make_config(gather=mk.MK_GATHER_STAGED))
    for rows in (mk.MK_GATHER_DIRECT, mk.MK_GATHER_GATHER4):
        b = gu.run_gpu(xd, ld, Wd, w.k, cfg=mk.make_config(gather=rows))
        for key in a:
            np.testing.assert_array_equal(a[key], b[key], err_msg=f"{w.name} rows={rows} {key}")
    mk.mk_release_workspace()


def test_gather_form_is_validated():
    T, H, F, E, k = 64, 64, 64, 4, 2
    x, l, W = gu.to_device(*_inputs(T, H, F, E, k))
    o = mk.alloc_outputs(T, F, E, k)
    st = mk.mk_moe_dispatch_gemm_ex(x, l, T, H, E, k, W, F, o["y_sorted"], o["src_index"], o["expert_offsets"],
                                    o["gate_w"], None, mk.make_config(gather=4))
    assert st == mk.MK_ERR_INVALID_ARG
    ep = mk.mk_moe_ep_sim(x, l, T, H, E, k, W, F, 2, o["y_sorted"], o["src_index"], o["expert_offsets"],
                          o["gate_w"], None, None, mk.make_config(gather=mk.MK_GATHER_GATHER4))
    assert ep == mk.MK_ERR_UNSUPPORTED
