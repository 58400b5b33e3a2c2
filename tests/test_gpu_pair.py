"""Parity of the SM-pair GEMM (cluster of two CTAs, cta_group::2, 256-row
tiles) with the CPU oracle, at the same bars as the single-SM path, and bit
for bit against it (same rows, same weights, same accumulation order)."""
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


def _inputs(T, H, F, E, k, seed=0):
    rng = np.random.default_rng(seed)
    x = synth.f32_to_bf16_bits(rng.standard_normal((T, H), dtype=np.float32))
    W = synth.f32_to_bf16_bits(rng.standard_normal((E, H, F), dtype=np.float32) / np.float32(np.sqrt(H)))
    return x, rng.standard_normal((T, E), dtype=np.float32), W


def _check(x, l, W, k, cfg, out_dtype):
    ref = gu.oracle_reference(x, l, W, k)
    g = gu.run_gpu(*gu.to_device(x, l, W), k, cfg=cfg)
    assert mk.mk_last_launch_info()["mma_pair"] == mk.MK_MMA_PAIR
    gu.assert_routing_exact(g, ref)
    gu.assert_gates(g, ref)
    gu.assert_y(g, ref, out_dtype)
    return g


MODES = [mk.MK_MODE_FUSED, mk.MK_MODE_UNFUSED]


@pytest.mark.parametrize("mode", MODES, ids=["fused", "unfused"])
@pytest.mark.parametrize("out_dtype", [mk.MK_OUT_BF16, mk.MK_OUT_F32], ids=["bf16", "f32"])
def test_pair_tiny_workload(mode, out_dtype):
    w = synth.WORKLOADS[1]
    x, l, W = synth.make_inputs(w)
    _check(x, l, W, w.k, mk.make_config(mode=mode, out_dtype=out_dtype, mma_pair=mk.MK_MMA_PAIR), out_dtype)


@pytest.mark.parametrize("shape", [
    (1, 64, 64, 1, 1),
    (7, 128, 192, 3, 2),
    (129, 256, 320, 5, 3),
    (1000, 512, 256, 64, 8),
    (300, 192, 128, 256, 8),
    (2000, 128, 512, 2, 1),
], ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("mode", MODES, ids=["fused", "unfused"])
def test_pair_ragged_shapes(shape, mode):
    T, H, F, E, k = shape
    x, l, W = _inputs(T, H, F, E, k, seed=T + E)
    _check(x, l, W, k, mk.make_config(mode=mode, out_dtype=mk.MK_OUT_F32, mma_pair=mk.MK_MMA_PAIR), mk.MK_OUT_F32)


@pytest.mark.parametrize("counts", [(256, 256), (255, 257), (128, 129), (511, 1), (513, 300)], ids=str)
def test_pair_tile_boundaries(counts):
    """Expert row counts on, below and above 256-row pair tiles (and the
    128-row half each CTA holds)."""
    T = sum(counts)
    E, k, H, F = len(counts), 1, 128, 256
    owner = np.repeat(np.arange(E), counts)
    np.random.default_rng(5).shuffle(owner)
    l = np.zeros((T, E), np.float32)
    l[np.arange(T), owner] = 3.0
    x, _, W = _inputs(T, H, F, E, k, seed=9)
    g = _check(x, l, W, k, mk.make_config(out_dtype=mk.MK_OUT_F32, mma_pair=mk.MK_MMA_PAIR), mk.MK_OUT_F32)
    assert list(np.diff(g["expert_offsets"])) == list(counts)


@pytest.mark.parametrize("dispatch_ctas,grid", [(2, 0), (5, 0), (0, 8), (6, 8), (60, 0)])
def test_pair_role_splits(dispatch_ctas, grid):
    T, H, F, E, k = 1500, 256, 512, 16, 4
    x, l, W = _inputs(T, H, F, E, k, seed=8)
    base = gu.run_gpu(*gu.to_device(x, l, W), k, cfg=mk.make_config(mode=mk.MK_MODE_UNFUSED,
                                                                     mma_pair=mk.MK_MMA_PAIR))
    g = gu.run_gpu(*gu.to_device(x, l, W), k, cfg=mk.make_config(dispatch_ctas=dispatch_ctas, grid_ctas=grid,
                                                                  mma_pair=mk.MK_MMA_PAIR))
    for key in ("expert_offsets", "src_index", "gate_w", "y"):
        np.testing.assert_array_equal(g[key], base[key])


def test_pair_repeated_calls_identical():
    T, H, F, E, k = 700, 256, 256, 8, 2
    x, l, W = gu.to_device(*_inputs(T, H, F, E, k, seed=12))
    cfg = mk.make_config(mma_pair=mk.MK_MMA_PAIR)
    first = gu.run_gpu(x, l, W, k, cfg=cfg)
    for _ in range(3):
        again = gu.run_gpu(x, l, W, k, cfg=cfg)
        for key in first:
            np.testing.assert_array_equal(again[key], first[key])


def test_pair_equals_single_bitwise():
    x, l, W = gu.to_device(*_inputs(1500, 256, 512, 16, 4, seed=14))
    a = gu.run_gpu(x, l, W, 4, cfg=mk.make_config(mma_pair=mk.MK_MMA_SINGLE))
    b = gu.run_gpu(x, l, W, 4, cfg=mk.make_config(mma_pair=mk.MK_MMA_PAIR))
    assert mk.mk_last_launch_info()["mma_pair"] == mk.MK_MMA_PAIR
    for key in a:
        np.testing.assert_array_equal(a[key], b[key])


def test_pair_combine_bitwise():
    x, l, W = gu.to_device(*_inputs(900, 256, 512, 8, 2, seed=15))
    a = mk.moe_layer(x, l, W, 2, cfg=mk.make_config(mma_pair=mk.MK_MMA_SINGLE))
    b = mk.moe_layer(x, l, W, 2, cfg=mk.make_config(mma_pair=mk.MK_MMA_PAIR))
    assert torch.equal(a["out"], b["out"]) and torch.equal(a["y_sorted"], b["y_sorted"])
