"""Expert parallelism simulated on one GPU (R logical ranks in one launch),
against the CPU oracle's exchange layout and products, and bit for bit
against the single-device path: the same rows meet the same weights in the
same MMA order, only the buffers they travel through differ."""
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


def _inputs(T, H, F, E, k, seed=0):
    rng = np.random.default_rng(seed)
    x = synth.f32_to_bf16_bits(rng.standard_normal((T, H), dtype=np.float32))
    W = synth.f32_to_bf16_bits(rng.standard_normal((E, H, F), dtype=np.float32) / np.float32(np.sqrt(H)))
    return x, rng.standard_normal((T, E), dtype=np.float32), W


def _np(t):
    return t.float().cpu().numpy() if t.dtype == torch.bfloat16 else t.cpu().numpy()


def _run_ep(xd, ld, Wd, k, R, cfg=None, combine=True):
    o = mk.moe_ep_sim(xd, ld, Wd, k, R, cfg=cfg, combine=combine)
    torch.cuda.synchronize()
    return dict(y_tok=_np(o["y_tok"]), out=_np(o["out"]) if combine else None, src_index=o["src_index"].cpu().numpy(),
                expert_offsets=o["expert_offsets"].cpu().numpy(), gate_w=o["gate_w"].cpu().numpy())


def _check_vs_oracle(x, l, W, k, R, out_dtype=mk.MK_OUT_BF16):
    E = W.shape[0]
    orc = Oracle()
    ref = orc.full(x, l, W, k)
    cnt, roff, rsrc = orc.ep_layout(ref["topk_idx"], E, R)
    g = _run_ep(*gu.to_device(x, l, W), k, R, cfg=mk.make_config(out_dtype=out_dtype))
    # receive metadata: the ranks' buffers one after another
    np.testing.assert_array_equal(g["src_index"], rsrc)
    np.testing.assert_array_equal(g["expert_offsets"][::E // R], roff)
    gu.assert_routing_exact(g, ref)
    gu.assert_gates(g, ref)
    # results came back to the sending rank, row t*k + j
    err = gu.rel_inf(g["y_tok"][ref["src_index"]], ref["y"])
    assert err <= gu.Y_TOL[out_dtype], f"y rel-inf {err:.3e}"
    ref_out = orc.combine(ref["y"], ref["src_index"], ref["gate_w"], x.shape[0], k)
    err = gu.rel_inf(g["out"], ref_out)
    assert err <= gu.Y_TOL[out_dtype], f"combine rel-inf {err:.3e}"


@pytest.mark.parametrize("R", [1, 2, 4, 8])
@pytest.mark.parametrize("out_dtype", [mk.MK_OUT_BF16, mk.MK_OUT_F32], ids=["bf16", "f32"])
def test_ep_tiny(R, out_dtype):
    w = synth.WORKLOADS[1]
    _check_vs_oracle(*synth.make_inputs(w), w.k, R, out_dtype)
    assert mk.mk_last_launch_info()["launches"] == 1


@pytest.mark.parametrize("shape", [
    (1, 64, 64, 8, 2, 8),        # one token: seven ranks send nothing
    (7, 128, 192, 4, 2, 4),      # F = 192: last N-block half full
    (129, 256, 320, 6, 3, 3),    # T not divisible by the ranks
    (1000, 512, 256, 64, 8, 8),
    (300, 192, 128, 256, 8, 8),  # 32 experts per rank, most empty
    (2000, 128, 512, 2, 1, 2),   # one expert per rank, k = 1
], ids=lambda s: "x".join(map(str, s)))
def test_ep_ragged_shapes(shape):
    T, H, F, E, k, R = shape
    _check_vs_oracle(*_inputs(T, H, F, E, k, seed=T + 5 * R), k, R, mk.MK_OUT_F32)


@pytest.mark.parametrize("R", [1, 2, 4, 8])
def test_ep_equals_single_device_bitwise(R):
    x, l, W = _inputs(1500, 256, 512, 16, 4, seed=41)
    xd, ld, Wd = gu.to_device(x, l, W)
    single = mk.moe_layer(xd, ld, Wd, 4)
    g = _run_ep(xd, ld, Wd, 4, R)
    src = single["src_index"].cpu().numpy()
    np.testing.assert_array_equal(g["src_index"], src)
    np.testing.assert_array_equal(g["y_tok"][src], _np(single["y_sorted"]))
    np.testing.assert_array_equal(g["out"], _np(single["out"]))


def test_ep_repeated_calls_and_no_combine():
    x, l, W = _inputs(600, 256, 256, 8, 2, seed=43)
    xd, ld, Wd = gu.to_device(x, l, W)
    a = _run_ep(xd, ld, Wd, 2, 4)
    for _ in range(3):
        b = _run_ep(xd, ld, Wd, 2, 4, combine=False)
        np.testing.assert_array_equal(a["y_tok"], b["y_tok"])
    c = _run_ep(xd, ld, Wd, 2, 2)  # another rank count on the same cached workspace
    np.testing.assert_array_equal(a["out"], c["out"])


def test_ep_unsupported_choices():
    T, H, F, E, k = 64, 64, 64, 4, 2
    xd, ld, Wd = gu.to_device(*_inputs(T, H, F, E, k))
    o = mk.alloc_outputs(T, F, E, k)
    for cfg in (mk.make_config(mode=mk.MK_MODE_UNFUSED), mk.make_config(gather=mk.MK_GATHER_DIRECT),
                mk.make_config(mma_pair=mk.MK_MMA_PAIR), mk.make_config(mode=mk.MK_MODE_DISPATCH_ONLY)):
        st = mk.mk_moe_ep_sim(xd, ld, T, H, E, k, Wd, F, 2, o["y_sorted"], o["src_index"], o["expert_offsets"],
                              o["gate_w"], None, None, cfg)
        assert st == mk.MK_ERR_UNSUPPORTED


def test_ep_withheld_rows_time_out_and_recover():
    """A source withholds its arrival count for one tile: the owner's bounded
    wait runs out, the call reports a timeout, and the next call is right."""
    w = synth.WORKLOADS[1]
    x, l, W = synth.make_inputs(w)
    xd, ld, Wd = gu.to_device(x, l, W)
    o = mk.alloc_outputs(w.T, w.F, w.E, w.k)
    cfg = mk.make_config(debug_fault=mk.MK_FAULT_DROP_TILE_FLAG, spin_limit_ns=50_000_000)
    st = mk.mk_moe_ep_sim(xd, ld, w.T, w.H, w.E, w.k, Wd, w.F, 4, o["y_sorted"], o["src_index"],
                          o["expert_offsets"], o["gate_w"], None, None, cfg)
    assert st == mk.MK_OK
    assert mk.mk_get_status() == mk.MK_ERR_TIMEOUT
    assert mk.mk_last_error_detail()["site"] == 4  # the owner's wait on the tile's arrivals
    _check_vs_oracle(x, l, W, w.k, 4)


@pytest.mark.parametrize("wid,R", [(2, 8), (5, 4), (3, 8)], ids=["mixtral_like-R8", "imbalanced-R4", "skewed-R8"])
def test_ep_full_size_equals_single_device(wid, R):
    """Full-size workloads: bit-identical to the single-device path, and
    sampled rows and tokens against the oracle."""
    w = synth.WORKLOADS[wid]
    x, l, W = synth.make_inputs(w)
    xd, ld, Wd = gu.to_device(x, l, W)
    single = mk.moe_layer(xd, ld, Wd, w.k)
    g = _run_ep(xd, ld, Wd, w.k, R)
    src = single["src_index"].cpu().numpy()
    np.testing.assert_array_equal(g["src_index"], src)
    np.testing.assert_array_equal(g["y_tok"][src], _np(single["y_sorted"]))
    np.testing.assert_array_equal(g["out"], _np(single["out"]))
    orc = Oracle()
    idx, gate = orc.route(l, w.k)
    offsets, osrc, _ = orc.dispatch(idx, gate, w.E)
    _, roff, rsrc = orc.ep_layout(idx, w.E, R)
    np.testing.assert_array_equal(g["src_index"], rsrc)
    rows = gu.sample_rows(offsets, 16, np.random.default_rng(wid), w.rows)
    ref = orc.expert_rows(x, W, w.k, offsets, osrc, rows)
    err = gu.rel_inf(g["y_tok"][osrc[rows]], ref)
    assert err <= gu.Y_TOL[mk.MK_OUT_BF16], f"rel-inf {err:.3e}"


@pytest.mark.parametrize("R", [1, 2, 4, 8])
def test_ep_gated_equals_single_device_bitwise(R):
    x, l, W1 = _inputs(1100, 256, 384, 16, 4, seed=61)
    _, _, W3 = _inputs(1100, 256, 384, 16, 4, seed=62)
    xd, ld, W1d = gu.to_device(x, l, W1)
    W3d = gu.to_device(x, l, W3)[2]
    single = mk.moe_gated(xd, ld, W1d, W3d, 4)
    g = mk.moe_ep_sim(xd, ld, W1d, 4, R, W3=W3d)
    torch.cuda.synchronize()
    order = single["src_index"].long()
    assert torch.equal(g["src_index"], single["src_index"])
    assert torch.equal(g["y_tok"][order], single["y_sorted"])


def test_ep_gated_combine_against_oracle():
    T, H, F, E, k = 500, 256, 256, 8, 2
    x, l, W1 = _inputs(T, H, F, E, k, seed=63)
    _, _, W3 = _inputs(T, H, F, E, k, seed=64)
    xd, ld, W1d = gu.to_device(x, l, W1)
    W3d = gu.to_device(x, l, W3)[2]
    g = mk.moe_ep_sim(xd, ld, W1d, k, 4, W3=W3d, cfg=mk.make_config(out_dtype=mk.MK_OUT_F32))
    orc = Oracle()
    ref = orc.gated_full(x, l, W1, W3, k)
    ref_out = orc.combine(ref["y"], ref["src_index"], ref["gate_w"], T, k)
    err = gu.rel_inf(g["out"].cpu().numpy(), ref_out)
    assert err <= gu.Y_TOL[mk.MK_OUT_F32], f"gated EP combine rel-inf {err:.3e}"


def test_ep_gated_full_size_mixtral_like():
    w = synth.WORKLOADS[2]
    x, l, W1 = synth.make_inputs(w)
    W3 = synth.make_w(synth.Workload(w.name, w.T, w.H, w.F, w.E, w.k, w.seed + 7))
    xd, ld, W1d = gu.to_device(x, l, W1)
    W3d = gu.to_device(x, l, W3)[2]
    del W1, W3
    single = mk.moe_gated(xd, ld, W1d, W3d, w.k)
    g = mk.moe_ep_sim(xd, ld, W1d, w.k, 8, W3=W3d)
    torch.cuda.synchronize()
    assert torch.equal(g["y_tok"][single["src_index"].long()], single["y_sorted"])
