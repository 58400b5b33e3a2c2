"""Parity of the combine (out[t] = sum_j gate[t,j] * y[(t,j)]) with the CPU
oracle: fused (one persistent launch) and unfused (five launches), bf16 and
f32 output, small shapes in full and the full-size workloads on sampled
tokens.  The oracle combines its fp64 expert products; the GPU combines the
stored y_sorted (bf16 or f32), so the tolerances are the product's."""
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


def _run(x, l, W, k, cfg):
    o = mk.moe_layer(*gu.to_device(x, l, W), k, cfg=cfg)
    torch.cuda.synchronize()
    f = (lambda t: t.float().cpu().numpy()) if o["out"].dtype == torch.bfloat16 else (lambda t: t.cpu().numpy())
    return dict(out=f(o["out"]), y=f(o["y_sorted"]), src_index=o["src_index"].cpu().numpy(),
                expert_offsets=o["expert_offsets"].cpu().numpy(), gate_w=o["gate_w"].cpu().numpy())


def _check(x, l, W, k, cfg, out_dtype):
    orc = Oracle()
    ref = orc.full(x, l, W, k)
    ref_out = orc.combine(ref["y"], ref["src_index"], ref["gate_w"], x.shape[0], k)
    g = _run(x, l, W, k, cfg)
    gu.assert_routing_exact(g, ref)
    gu.assert_y(g, ref, out_dtype)
    err = gu.rel_inf(g["out"], ref_out)
    assert err <= gu.Y_TOL[out_dtype], f"combine rel-inf {err:.3e}"
    return g


@pytest.mark.parametrize("mode", [mk.MK_MODE_FUSED, mk.MK_MODE_UNFUSED], ids=["fused", "unfused"])
@pytest.mark.parametrize("out_dtype", [mk.MK_OUT_BF16, mk.MK_OUT_F32], ids=["bf16", "f32"])
def test_combine_tiny(mode, out_dtype):
    w = synth.WORKLOADS[1]
    x, l, W = synth.make_inputs(w)
    _check(x, l, W, w.k, mk.make_config(mode=mode, out_dtype=out_dtype), out_dtype)
    assert mk.mk_last_launch_info()["launches"] == (1 if mode == mk.MK_MODE_FUSED else 5)


@pytest.mark.parametrize("shape", [
    (1, 64, 64, 1, 1),
    (7, 128, 192, 3, 2),
    (129, 256, 320, 5, 3),
    (1000, 512, 256, 64, 8),
    (300, 192, 128, 256, 8),
], ids=lambda s: "x".join(map(str, s)))
def test_combine_ragged_shapes(shape):
    T, H, F, E, k = shape
    x, l, W = _inputs(T, H, F, E, k, seed=T + E + 1)
    _check(x, l, W, k, mk.make_config(out_dtype=mk.MK_OUT_F32), mk.MK_OUT_F32)


def test_combine_fused_equals_unfused_and_leaves_y_unchanged():
    T, H, F, E, k = 1500, 256, 512, 16, 4
    x, l, W = _inputs(T, H, F, E, k, seed=41)
    a = _run(x, l, W, k, mk.make_config())
    b = _run(x, l, W, k, mk.make_config(mode=mk.MK_MODE_UNFUSED))
    plain = gu.run_gpu(*gu.to_device(x, l, W), k)
    for key in ("out", "y", "src_index", "gate_w", "expert_offsets"):
        np.testing.assert_array_equal(a[key], b[key])
    np.testing.assert_array_equal(a["y"], plain["y"])


def test_combine_rejected_in_dispatch_only_mode():
    T, H, F, E, k = 64, 64, 64, 4, 2
    x, l, W = gu.to_device(*_inputs(T, H, F, E, k))
    o = mk.alloc_outputs(T, F, E, k)
    out = torch.empty((T, F), dtype=torch.bfloat16, device="cuda")
    st = mk.mk_moe_dispatch_gemm_combine(x, l, T, H, E, k, W, F, o["y_sorted"], o["src_index"], o["expert_offsets"],
                                         o["gate_w"], out, None, mk.make_config(mode=mk.MK_MODE_DISPATCH_ONLY))
    assert st == mk.MK_ERR_INVALID_ARG


@pytest.mark.parametrize("wid", [2, 4, 5])
def test_combine_full_size_sampled_tokens(wid):
    w = synth.WORKLOADS[wid]
    x, l, W = synth.make_inputs(w)
    orc = Oracle()
    idx, gate = orc.route(l, w.k)
    offsets, src, gw = orc.dispatch(idx, gate, w.E)
    xd, ld, Wd = gu.to_device(x, l, W)
    del W
    o = mk.moe_layer(xd, ld, Wd, w.k)
    out = o["out"].float().cpu().numpy()
    row_of = np.empty(w.rows, dtype=np.int64)
    row_of[src] = np.arange(w.rows)
    tokens = np.random.default_rng(wid).choice(w.T, size=12, replace=False)
    ref = np.zeros((tokens.size, w.F))
    for i, t in enumerate(tokens):
        for j in range(w.k):
            r = int(row_of[t * w.k + j])
            e = int(np.searchsorted(offsets, r, side="right") - 1)
            off1 = np.array([0, offsets[e + 1] - offsets[e]], dtype=np.int32)
            yr = orc.expert_rows(x, synth.make_w_expert(w, e)[None], w.k, off1, src[offsets[e]:offsets[e + 1]],
                                 np.array([r - offsets[e]]))
            ref[i] += float(gw[r]) * yr[0]
    err = gu.rel_inf(out[tokens], ref)
    assert err <= gu.Y_TOL[mk.MK_OUT_BF16], f"{w.name}: combine rel-inf {err:.3e}"
