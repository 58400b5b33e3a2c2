"""Parity of the gated expert FFN (SwiGLU in the GEMM epilogue) with the CPU
oracle: h_sorted[r] = silu(x[t] . W1[e]) * (x[t] . W3[e]).  Routing and
offsets bit-exact; h within the product tolerances (1e-2 bf16, 1e-4 f32)."""
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
    W1 = synth.f32_to_bf16_bits(rng.standard_normal((E, H, F), dtype=np.float32) / np.float32(np.sqrt(H)))
    W3 = synth.f32_to_bf16_bits(rng.standard_normal((E, H, F), dtype=np.float32) / np.float32(np.sqrt(H)))
    return x, rng.standard_normal((T, E), dtype=np.float32), W1, W3


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


def _run(x, l, W1, W3, k, cfg):
    o = mk.moe_gated(_dev(x), torch.from_numpy(l).cuda(), _dev(W1), _dev(W3), k, cfg=cfg)
    torch.cuda.synchronize()
    y = o["y_sorted"]
    y = y.float().cpu().numpy() if y.dtype == torch.bfloat16 else y.cpu().numpy()
    return dict(y=y, src_index=o["src_index"].cpu().numpy(), expert_offsets=o["expert_offsets"].cpu().numpy(),
                gate_w=o["gate_w"].cpu().numpy())


def _check(x, l, W1, W3, k, cfg, out_dtype):
    ref = Oracle().gated_full(x, l, W1, W3, k)
    g = _run(x, l, W1, W3, k, cfg)
    gu.assert_routing_exact(g, ref)
    gu.assert_gates(g, ref)
    gu.assert_y(g, ref, out_dtype)
    return g


@pytest.mark.parametrize("mode", [mk.MK_MODE_FUSED, mk.MK_MODE_UNFUSED], ids=["fused", "unfused"])
@pytest.mark.parametrize("out_dtype", [mk.MK_OUT_BF16, mk.MK_OUT_F32], ids=["bf16", "f32"])
def test_gated_tiny(mode, out_dtype):
    _check(*_inputs(256, 512, 1024, 8, 2, seed=1), 2, mk.make_config(mode=mode, out_dtype=out_dtype), out_dtype)


@pytest.mark.parametrize("shape", [
    (1, 64, 64, 1, 1),
    (7, 128, 192, 3, 2),      # F = 192: last 128-column block half full
    (129, 256, 320, 5, 3),
    (1000, 512, 256, 64, 8),
    (300, 192, 128, 256, 8),
], ids=lambda s: "x".join(map(str, s)))
def test_gated_ragged_shapes(shape):
    T, H, F, E, k = shape
    _check(*_inputs(T, H, F, E, k, seed=T + 2), k, mk.make_config(out_dtype=mk.MK_OUT_F32), mk.MK_OUT_F32)


def test_gated_fused_equals_unfused():
    x, l, W1, W3 = _inputs(1500, 256, 512, 16, 4, seed=43)
    a = _run(x, l, W1, W3, 4, mk.make_config())
    b = _run(x, l, W1, W3, 4, mk.make_config(mode=mk.MK_MODE_UNFUSED))
    for key in a:
        np.testing.assert_array_equal(a[key], b[key])


def test_gated_refuses_sm_pairs():
    T, H, F, E, k = 64, 64, 64, 4, 2
    x, l, W1, W3 = _inputs(T, H, F, E, k)
    o = mk.alloc_outputs(T, F, E, k)
    st = mk.mk_moe_dispatch_gated(_dev(x), torch.from_numpy(l).cuda(), T, H, E, k, _dev(W1), _dev(W3), F,
                                  o["y_sorted"], o["src_index"], o["expert_offsets"], o["gate_w"], None,
                                  mk.make_config(mma_pair=mk.MK_MMA_PAIR))
    assert st == mk.MK_ERR_UNSUPPORTED


def test_gated_mixtral_like_sampled_rows():
    """The Mixtral-like layer with a second, independently drawn projection."""
    w = synth.WORKLOADS[2]
    x, l, W1 = synth.make_inputs(w)
    w3 = synth.Workload(w.name, w.T, w.H, w.F, w.E, w.k, w.seed + 7)
    W3 = synth.make_w(w3)
    orc = Oracle()
    idx, gate = orc.route(l, w.k)
    offsets, src, _ = orc.dispatch(idx, gate, w.E)
    g = _run(x, l, W1, W3, w.k, None)
    np.testing.assert_array_equal(g["expert_offsets"], offsets)
    np.testing.assert_array_equal(g["src_index"], src)
    rows = gu.sample_rows(offsets, 24, np.random.default_rng(2), w.rows)
    ref = orc.gated_rows(x, W1, W3, w.k, offsets, src, rows)
    err = gu.rel_inf(g["y"][rows], ref)
    assert err <= gu.Y_TOL[mk.MK_OUT_BF16], f"gated rel-inf {err:.3e}"
