"""Parity of the wide GEMM tiles (one SM, 256-row tiles, two 128-row
accumulators sharing each staged block of the weights) with the CPU oracle,
at the same bars as the 128-row tiles, and bit for bit against them: every
output row meets the same weights in the same MMA order, only the tile that
carries it differs."""
import numpy as np
import pytest

import moe_token_dispatch_persistent_gb300 as mk
from moe_token_dispatch_persistent_gb300 import synth
from oracle.oracle import Oracle

import gpu_util as gu

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

WIDE = mk.MK_MMA_WIDE


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
    assert mk.mk_last_launch_info()["mma_pair"] == WIDE
    gu.assert_routing_exact(g, ref)
    gu.assert_gates(g, ref)
    gu.assert_y(g, ref, out_dtype)
    return g


MODES = [mk.MK_MODE_FUSED, mk.MK_MODE_UNFUSED]


@pytest.mark.parametrize("mode", MODES, ids=["fused", "unfused"])
@pytest.mark.parametrize("out_dtype", [mk.MK_OUT_BF16, mk.MK_OUT_F32], ids=["bf16", "f32"])
def test_wide_tiny_workload(mode, out_dtype):
    w = synth.WORKLOADS[1]
    x, l, W = synth.make_inputs(w)
    _check(x, l, W, w.k, mk.make_config(mode=mode, out_dtype=out_dtype, mma_pair=WIDE), out_dtype)


@pytest.mark.parametrize("shape", [
    (1, 64, 64, 1, 1),
    (7, 128, 192, 3, 2),
    (129, 256, 320, 5, 3),
    (1000, 512, 256, 64, 8),
    (300, 192, 128, 256, 8),
    (2000, 128, 512, 2, 1),
], ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("mode", MODES, ids=["fused", "unfused"])
def test_wide_ragged_shapes(shape, mode):
    T, H, F, E, k = shape
    x, l, W = _inputs(T, H, F, E, k, seed=T + E)
    _check(x, l, W, k, mk.make_config(mode=mode, out_dtype=mk.MK_OUT_F32, mma_pair=WIDE), mk.MK_OUT_F32)


@pytest.mark.parametrize("counts", [(256, 256), (255, 257), (128, 129), (511, 1), (513, 300), (127, 384)],
                         ids=str)
def test_wide_tile_boundaries(counts):
    """Expert row counts on, below and above 256-row tiles and the 128-row
    split between the two accumulators (a tile of at most 128 rows uses one)."""
    T = sum(counts)
    E, k, H, F = len(counts), 1, 128, 256
    owner = np.repeat(np.arange(E), counts)
    np.random.default_rng(5).shuffle(owner)
    l = np.zeros((T, E), np.float32)
    l[np.arange(T), owner] = 3.0
    x, _, W = _inputs(T, H, F, E, k, seed=9)
    g = _check(x, l, W, k, mk.make_config(out_dtype=mk.MK_OUT_F32, mma_pair=WIDE), mk.MK_OUT_F32)
    assert list(np.diff(g["expert_offsets"])) == list(counts)


@pytest.mark.parametrize("dispatch_ctas,grid", [(2, 0), (5, 0), (0, 8), (6, 8), (60, 0), (1, 3)])
def test_wide_role_splits(dispatch_ctas, grid):
    T, H, F, E, k = 1500, 256, 512, 16, 4
    x, l, W = _inputs(T, H, F, E, k, seed=8)
    base = gu.run_gpu(*gu.to_device(x, l, W), k, cfg=mk.make_config(mode=mk.MK_MODE_UNFUSED, mma_pair=WIDE))
    g = gu.run_gpu(*gu.to_device(x, l, W), k, cfg=mk.make_config(dispatch_ctas=dispatch_ctas, grid_ctas=grid,
                                                                  mma_pair=WIDE))
    for key in ("expert_offsets", "src_index", "gate_w", "y"):
        np.testing.assert_array_equal(g[key], base[key])


def test_wide_repeated_calls_identical():
    x, l, W = gu.to_device(*_inputs(700, 256, 256, 8, 2, seed=12))
    cfg = mk.make_config(mma_pair=WIDE)
    first = gu.run_gpu(x, l, W, 2, cfg=cfg)
    for _ in range(3):
        again = gu.run_gpu(x, l, W, 2, cfg=cfg)
        for key in first:
            np.testing.assert_array_equal(again[key], first[key])


@pytest.mark.parametrize("out_dtype", [mk.MK_OUT_BF16, mk.MK_OUT_F32], ids=["bf16", "f32"])
def test_wide_equals_single_bitwise(out_dtype):
    x, l, W = gu.to_device(*_inputs(1500, 256, 512, 16, 4, seed=14))
    a = gu.run_gpu(x, l, W, 4, cfg=mk.make_config(mma_pair=mk.MK_MMA_SINGLE, out_dtype=out_dtype))
    b = gu.run_gpu(x, l, W, 4, cfg=mk.make_config(mma_pair=WIDE, out_dtype=out_dtype))
    assert mk.mk_last_launch_info()["mma_pair"] == WIDE
    for key in a:
        np.testing.assert_array_equal(a[key], b[key])


def test_wide_combine_and_gated_bitwise():
    x, l, W1 = gu.to_device(*_inputs(900, 256, 384, 8, 2, seed=15))
    W3 = gu.to_device(*_inputs(900, 256, 384, 8, 2, seed=16))[2]
    a = mk.moe_layer(x, l, W1, 2, cfg=mk.make_config(mma_pair=mk.MK_MMA_SINGLE))
    b = mk.moe_layer(x, l, W1, 2, cfg=mk.make_config(mma_pair=WIDE))
    assert torch.equal(a["out"], b["out"]) and torch.equal(a["y_sorted"], b["y_sorted"])
    ga = mk.moe_gated(x, l, W1, W3, 2, cfg=mk.make_config(mma_pair=mk.MK_MMA_SINGLE))
    gb = mk.moe_gated(x, l, W1, W3, 2, cfg=mk.make_config(mma_pair=WIDE))
    torch.cuda.synchronize()
    assert mk.mk_last_launch_info()["mma_pair"] == WIDE
    assert torch.equal(ga["y_sorted"], gb["y_sorted"])


def test_wide_gated_against_oracle():
    T, H, F, E, k = 600, 256, 256, 4, 2
    x, l, W1 = _inputs(T, H, F, E, k, seed=17)
    _, _, W3 = _inputs(T, H, F, E, k, seed=18)
    xd, ld, W1d = gu.to_device(x, l, W1)
    W3d = gu.to_device(x, l, W3)[2]
    g = mk.moe_gated(xd, ld, W1d, W3d, k, cfg=mk.make_config(mma_pair=WIDE, out_dtype=mk.MK_OUT_F32))
    ref = Oracle().gated_full(x, l, W1, W3, k)
    err = gu.rel_inf(g["y_sorted"].cpu().numpy(), ref["y"])
    assert err <= gu.Y_TOL[mk.MK_OUT_F32], f"gated rel-inf {err:.3e}"


def test_wide_host_buffers_streamed():
    """The end-to-end entry point with host buffers and streamed result
    chunks, on wide tiles: the same bits as the device call."""
    T, H, F, E, k = 2000, 256, 512, 8, 2
    x, l, W = _inputs(T, H, F, E, k, seed=19)
    dev = gu.run_gpu(*gu.to_device(x, l, W), k, cfg=mk.make_config(mma_pair=WIDE))
    Wd = gu.to_device(x, l, W)[2]
    xh = torch.from_numpy(x.view(np.int16)).pin_memory()
    lh = torch.from_numpy(l).pin_memory()
    y = torch.empty((T * k, F), dtype=torch.int16).pin_memory()
    src = torch.empty(T * k, dtype=torch.int32).pin_memory()
    off = torch.empty(E + 1, dtype=torch.int32).pin_memory()
    gate = torch.empty(T * k, dtype=torch.float32).pin_memory()
    st = mk.mk_moe_dispatch_gemm_host(xh, lh, T, H, E, k, Wd, F, y, src, off, gate, None,
                                      mk.make_config(mma_pair=WIDE))
    assert st == mk.MK_OK and mk.mk_get_status() == mk.MK_OK
    np.testing.assert_array_equal(off.numpy(), dev["expert_offsets"])
    np.testing.assert_array_equal(src.numpy(), dev["src_index"])
    # the device result was read back as float32 from bf16: its top 16 bits are the bf16 bits
    np.testing.assert_array_equal(y.numpy().view(np.uint16), (dev["y"].view(np.uint32) >> 16).astype(np.uint16))


@pytest.mark.parametrize("wid", [2, 3, 5], ids=["mixtral_like", "skewed", "imbalanced"])
def test_wide_full_size_equals_single(wid):
    """Full-size workloads: bit-identical to 128-row tiles, and sampled rows
    against the oracle."""
    w = synth.WORKLOADS[wid]
    x, l, W = synth.make_inputs(w)
    xd, ld, Wd = gu.to_device(x, l, W)
    a = gu.run_gpu(xd, ld, Wd, w.k, cfg=mk.make_config(mma_pair=mk.MK_MMA_SINGLE))
    b = gu.run_gpu(xd, ld, Wd, w.k, cfg=mk.make_config(mma_pair=WIDE))
    for key in a:
        np.testing.assert_array_equal(a[key], b[key])
    orc = Oracle()
    idx, gate = orc.route(l, w.k)
    offsets, src, _ = orc.dispatch(idx, gate, w.E)
    rows = gu.sample_rows(offsets, 16, np.random.default_rng(wid), w.rows)
    ref = orc.expert_rows(x, W, w.k, offsets, src, rows)
    err = gu.rel_inf(b["y"][rows], ref)
    assert err <= gu.Y_TOL[mk.MK_OUT_BF16], f"rel-inf {err:.3e}"


@pytest.mark.parametrize("shape", [(700, 256, 256, 8, 2), (300, 192, 128, 4, 3), (1, 64, 64, 1, 1)],
                         ids=lambda s: "x".join(map(str, s)))
def test_wide_direct_rows_bitwise(shape):
    """Rows straight from x into wide tiles (each copy warp fills one 128-row
    block): the same bits as staged 128-row tiles."""
    T, H, F, E, k = shape
    x, l, W = gu.to_device(*_inputs(T, H, F, E, k, seed=23 + T))
    a = gu.run_gpu(x, l, W, k, cfg=mk.make_config(mma_pair=mk.MK_MMA_SINGLE))
    b = gu.run_gpu(x, l, W, k, cfg=mk.make_config(mma_pair=WIDE, gather=mk.MK_GATHER_DIRECT))
    info = mk.mk_last_launch_info()
    assert info["mma_pair"] == WIDE and info["gather"] == mk.MK_GATHER_DIRECT
    for key in a:
        np.testing.assert_array_equal(a[key], b[key])


def test_wide_direct_rows_full_size():
    w = synth.WORKLOADS[2]
    x, l, W = synth.make_inputs(w)
    xd, ld, Wd = gu.to_device(x, l, W)
    a = gu.run_gpu(xd, ld, Wd, w.k, cfg=mk.make_config(mma_pair=mk.MK_MMA_SINGLE))
    b = gu.run_gpu(xd, ld, Wd, w.k, cfg=mk.make_config(mma_pair=WIDE, gather=mk.MK_GATHER_DIRECT))
    for key in a:
        np.testing.assert_array_equal(a[key], b[key])


@pytest.mark.parametrize("R", [1, 2, 4, 8])
def test_wide_expert_parallel_bitwise(R):
    """The expert-parallel simulation on wide tiles: the same bits as the
    single-device path on 128-row tiles, tokens returned to their ranks."""
    x, l, W = gu.to_device(*_inputs(1500, 256, 512, 16, 4, seed=21))
    single = mk.moe_layer(x, l, W, 4, cfg=mk.make_config(mma_pair=mk.MK_MMA_SINGLE))
    g = mk.moe_ep_sim(x, l, W, 4, R, cfg=mk.make_config(mma_pair=WIDE))
    torch.cuda.synchronize()
    assert mk.mk_last_launch_info()["mma_pair"] == WIDE
    order = single["src_index"].long()
    assert torch.equal(g["src_index"], single["src_index"])
    assert torch.equal(g["y_tok"][order], single["y_sorted"])
    assert torch.equal(g["out"], single["out"])


@pytest.mark.parametrize("T,E,k,H,tiles,gather", [
    (4096, 8, 2, 64, WIDE, mk.MK_GATHER_STAGED),              # Mixtral-like shape: wide, staged (1 MiB of rows)
    (2048, 64, 8, 64, WIDE, mk.MK_GATHER_DIRECT),              # fine-grained routing: wide, rows straight from x
    (128, 256, 8, 64, mk.MK_MMA_SINGLE, mk.MK_GATHER_DIRECT),  # decode-shaped, under 1 MiB of rows
    (1000, 64, 8, 64, mk.MK_MMA_SINGLE, mk.MK_GATHER_DIRECT),  # 125 rows per expert, under 1 MiB of rows
    (2000, 64, 8, 64, mk.MK_MMA_SINGLE, mk.MK_GATHER_STAGED),  # 2 MiB of rows, not wide: staged
    (128, 256, 8, 7168, mk.MK_MMA_SINGLE, mk.MK_GATHER_STAGED),  # decode layer: 15 MB of rows, staged
    (256, 8, 2, 512, mk.MK_MMA_SINGLE, mk.MK_GATHER_DIRECT),   # the tiny layer: 0.5 MiB of rows
])
def test_auto_resolution(T, E, k, H, tiles, gather):
    """What AUTO picks, per shape (the reported launch facts)."""
    F = 64
    xd, ld, Wd = gu.to_device(*_inputs(T, H, F, E, k, seed=31))
    mk.moe_dispatch_gemm(xd, ld, Wd, k)
    torch.cuda.synchronize()
    info = mk.mk_last_launch_info()
    assert info["mma_pair"] == tiles and info["gather"] == gather
