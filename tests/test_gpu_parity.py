"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Routing, offsets and src_index must match bit for bit; gates within 2e-6
(fp32 expf vs fp64); y_sorted within ||Y - Yref||_inf / ||Yref||_inf of 1e-2
(bf16 output) or 1e-4 (fp32 output)."""
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


def _inputs(T, H, F, E, k, seed=0, logits=None):
    rng = np.random.default_rng(seed)
    x = synth.f32_to_bf16_bits(rng.standard_normal((T, H), dtype=np.float32))
    W = synth.f32_to_bf16_bits(rng.standard_normal((E, H, F), dtype=np.float32) / np.float32(np.sqrt(H)))
    if logits is None:
        logits = rng.standard_normal((T, E), dtype=np.float32)
    return x, np.ascontiguousarray(logits, dtype=np.float32), W


def _check_all(x, l, W, k, cfg=None, out_dtype=mk.MK_OUT_BF16, check_y=True):
    ref = gu.oracle_reference(x, l, W, k)
    g = gu.run_gpu(*gu.to_device(x, l, W), k, cfg=cfg)
    gu.assert_routing_exact(g, ref)
    gu.assert_gates(g, ref)
    if check_y:
        gu.assert_y(g, ref, out_dtype)
    return g, ref


MODES = [mk.MK_MODE_FUSED, mk.MK_MODE_UNFUSED]


@pytest.mark.parametrize("mode", MODES, ids=["fused", "unfused"])
@pytest.mark.parametrize("out_dtype", [mk.MK_OUT_BF16, mk.MK_OUT_F32], ids=["bf16", "f32"])
def test_tiny_workload(mode, out_dtype):
    w = synth.WORKLOADS[1]
    x, l, W = synth.make_inputs(w)
    _check_all(x, l, W, w.k, mk.make_config(mode=mode, out_dtype=out_dtype), out_dtype)


@pytest.mark.parametrize("shape", [
    (1, 64, 64, 1, 1),        # one token, one expert
    (7, 128, 192, 3, 2),      # ragged everything; F = 192 -> partial N-block
    (129, 256, 320, 5, 3),    # one past a tile; F = 320 -> last N-block 64 wide
    (1000, 512, 256, 64, 8),  # many experts, k = 8
    (300, 192, 128, 256, 8),  # E = 256, most experts small
    (2000, 128, 512, 2, 1),   # ~1000 rows per expert: several full tiles + tail
], ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("mode", MODES, ids=["fused", "unfused"])
def test_ragged_shapes(shape, mode):
    T, H, F, E, k = shape
    x, l, W = _inputs(T, H, F, E, k, seed=T + E)
    _check_all(x, l, W, k, mk.make_config(mode=mode, out_dtype=mk.MK_OUT_F32), mk.MK_OUT_F32)


@pytest.mark.parametrize("counts", [(128, 128), (127, 129), (256, 1), (129, 383)], ids=str)
def test_tile_boundaries(counts):
    """Experts whose row counts sit on, just below and just above 128-row tiles."""
    T = sum(counts)
    E, k, H, F = len(counts), 1, 128, 256
    owner = np.repeat(np.arange(E), counts)
    np.random.default_rng(5).shuffle(owner)
    l = np.zeros((T, E), np.float32)
    l[np.arange(T), owner] = 3.0
    x, _, W = _inputs(T, H, F, E, k, seed=9)
    g, ref = _check_all(x, l, W, k, mk.make_config(out_dtype=mk.MK_OUT_F32), mk.MK_OUT_F32)
    assert list(np.diff(g["expert_offsets"])) == list(counts)


def test_all_logits_equal():
    T, H, F, E, k = 300, 128, 128, 8, 4
    x, _, W = _inputs(T, H, F, E, k)
    l = np.zeros((T, E), np.float32)
    g, ref = _check_all(x, l, W, k)
    assert list(np.diff(g["expert_offsets"])) == [T] * 4 + [0] * 4
    assert np.all(g["gate_w"] == np.float32(0.25))


def test_one_expert_active_and_neg_inf():
    T, H, F, E, k = 500, 256, 256, 16, 2
    x, l, W = _inputs(T, H, F, E, k, seed=3)
    l[:, 5] += 50.0           # expert 5 first for everyone
    l[:, [1, 2, 9]] = -np.inf  # never chosen
    g, ref = _check_all(x, l, W, k)
    cnt = np.diff(g["expert_offsets"])
    assert cnt[5] == T and cnt[1] == cnt[2] == cnt[9] == 0


def test_rows_with_few_finite_logits():
    T, H, F, E, k = 64, 64, 64, 6, 3
    x, l, W = _inputs(T, H, F, E, k, seed=4)
    l[::2, :] = -np.inf
    l[::2, 4] = 1.0           # one finite logit: gates (1, 0, 0)
    l[1::4, :] = -np.inf      # nothing finite: gates all 0, experts 0..k-1
    _check_all(x, l, W, k)


def test_e_equals_k():
    T, H, F, E, k = 100, 64, 128, 4, 4
    x, l, W = _inputs(T, H, F, E, k, seed=6)
    g, _ = _check_all(x, l, W, k)
    assert list(np.diff(g["expert_offsets"])) == [T] * 4


def test_zero_tokens():
    E = 8
    out = mk.alloc_outputs(0, 128, E, 2)
    out["expert_offsets"].fill_(-1)
    x = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    l = torch.empty((0, E), dtype=torch.float32, device="cuda")
    W = torch.zeros((E, 64, 128), dtype=torch.bfloat16, device="cuda")
    mk.moe_dispatch_gemm(x, l, W, 2, out=out)
    assert out["expert_offsets"].cpu().tolist() == [0] * (E + 1)


def test_dispatch_only_matches_routing():
    w = synth.WORKLOADS[1]
    x, l, W = synth.make_inputs(w)
    ref = gu.oracle_reference(x, l, W, w.k)
    g = gu.run_gpu(*gu.to_device(x, l, W), w.k, cfg=mk.make_config(mode=mk.MK_MODE_DISPATCH_ONLY))
    gu.assert_routing_exact(g, ref)
    gu.assert_gates(g, ref)


@pytest.mark.parametrize("dispatch_ctas,grid", [(1, 0), (3, 0), (0, 8), (7, 8), (60, 0)])
def test_role_splits(dispatch_ctas, grid):
    """Any split of the grid between the roles gives the same bits."""
    T, H, F, E, k = 1500, 256, 512, 16, 4
    x, l, W = _inputs(T, H, F, E, k, seed=8)
    base = gu.run_gpu(*gu.to_device(x, l, W), k, cfg=mk.make_config(mode=mk.MK_MODE_UNFUSED))
    g = gu.run_gpu(*gu.to_device(x, l, W), k, cfg=mk.make_config(dispatch_ctas=dispatch_ctas, grid_ctas=grid))
    for key in ("expert_offsets", "src_index", "gate_w", "y"):
        np.testing.assert_array_equal(g[key], base[key])


def test_n_group_orders_agree():
    T, H, F, E, k = 1200, 128, 1024, 4, 2
    x, l, W = _inputs(T, H, F, E, k, seed=10)
    outs = [gu.run_gpu(*gu.to_device(x, l, W), k, cfg=mk.make_config(n_group=g)) for g in (1, 2, 3, 4)]
    for o in outs[1:]:
        np.testing.assert_array_equal(o["y"], outs[0]["y"])


def test_caller_workspace_reused_across_shapes():
    shapes = [(400, 128, 256, 8, 2), (90, 256, 128, 3, 3), (400, 128, 256, 8, 2)]
    big = max(mk.mk_workspace_size(T, H, F, E, k) for T, H, F, E, k in shapes)
    ws = torch.zeros(big, dtype=torch.uint8, device="cuda")
    for i, (T, H, F, E, k) in enumerate(shapes):
        x, l, W = _inputs(T, H, F, E, k, seed=20 + i)
        ref = gu.oracle_reference(x, l, W, k)
        xd, ld, Wd = gu.to_device(x, l, W)
        o = mk.moe_dispatch_gemm(xd, ld, Wd, k, workspace=ws, ws_bytes=big)
        g = dict(y=o["y_sorted"].float().cpu().numpy(), src_index=o["src_index"].cpu().numpy(),
                 expert_offsets=o["expert_offsets"].cpu().numpy(), gate_w=o["gate_w"].cpu().numpy())
        gu.assert_routing_exact(g, ref)
        gu.assert_y(g, ref, mk.MK_OUT_BF16)


def test_workspace_too_small_is_rejected():
    T, H, F, E, k = 64, 64, 64, 2, 1
    x, l, W = gu.to_device(*_inputs(T, H, F, E, k))
    need = mk.mk_workspace_size(T, H, F, E, k)
    ws = torch.zeros(need - 256, dtype=torch.uint8, device="cuda")
    out = mk.alloc_outputs(T, F, E, k)
    st = mk.mk_moe_dispatch_gemm_ex(x, l, T, H, E, k, W, F, out["y_sorted"], out["src_index"], out["expert_offsets"],
                                    out["gate_w"], None, None, ws, need - 256)
    assert st == mk.MK_ERR_WORKSPACE


def test_repeated_calls_are_identical():
    T, H, F, E, k = 700, 256, 256, 8, 2
    x, l, W = gu.to_device(*_inputs(T, H, F, E, k, seed=12))
    first = gu.run_gpu(x, l, W, k)
    for _ in range(5):
        again = gu.run_gpu(x, l, W, k)
        for key in first:
            np.testing.assert_array_equal(again[key], first[key])


def test_host_buffer_entry_point():
    T, H, F, E, k = 333, 128, 256, 8, 2
    x, l, W = _inputs(T, H, F, E, k, seed=13)
    ref = gu.oracle_reference(x, l, W, k)
    Wd = gu.to_device(x, l, W)[2]
    xh = torch.from_numpy(x.view(np.int16)).pin_memory()
    lh = torch.from_numpy(l).pin_memory()
    yh = torch.empty((T * k, F), dtype=torch.int16).pin_memory()
    sh = torch.empty(T * k, dtype=torch.int32).pin_memory()
    oh = torch.empty(E + 1, dtype=torch.int32).pin_memory()
    gh = torch.empty(T * k, dtype=torch.float32).pin_memory()
    st = mk.mk_moe_dispatch_gemm_host(xh, lh, T, H, E, k, Wd, F, yh, sh, oh, gh)
    assert st == mk.MK_OK
    g = dict(y=synth.bf16_bits_to_f32(yh.numpy().view(np.uint16)), src_index=sh.numpy(), expert_offsets=oh.numpy(),
             gate_w=gh.numpy())
    gu.assert_routing_exact(g, ref)
    gu.assert_gates(g, ref)
    gu.assert_y(g, ref, mk.MK_OUT_BF16)


def test_trace_records_phases():
    T, H, F, E, k = 2000, 256, 512, 8, 2
    x, l, W = gu.to_device(*_inputs(T, H, F, E, k))
    mk.moe_dispatch_gemm(x, l, W, k, cfg=mk.make_config(trace=1))
    info = mk.mk_last_launch_info()
    tr = mk.mk_read_trace(T, H, E, k, info["grid_ctas"])
    assert (tr[:, 0] > 0).all() and (tr[:, 15] >= tr[:, 0]).all()
    assert (tr[: info["dispatch_ctas"], 5] > 0).all()  # every dispatch CTA finished its gather


@pytest.mark.parametrize("gather", [mk.MK_GATHER_STAGED, mk.MK_GATHER_DIRECT], ids=["staged", "direct"])
@pytest.mark.parametrize("tiles", [mk.MK_MMA_SINGLE, mk.MK_MMA_WIDE], ids=["single", "wide"])
def test_trace_phase_order(gather, tiles):
    """Every CTA's stamps come in phase order: routing, its barrier, scan and
    scatter, the GEMM role, its first full stage at the tensor core, its
    last MMA, the exit.  (The role's end is stamped by the producer warp,
    which may finish before the MMA warp's last MMAs complete.)"""
    T, H, F, E, k = 3000, 512, 768, 16, 4
    x, l, W = gu.to_device(*_inputs(T, H, F, E, k, seed=61))
    mk.moe_dispatch_gemm(x, l, W, k, cfg=mk.make_config(trace=1, gather=gather, mma_pair=tiles))
    info = mk.mk_last_launch_info()
    tr = mk.mk_read_trace(T, H, E, k, info["grid_ctas"]).astype(np.int64)
    for slot in (0, 1, 2, 3, 15):
        assert (tr[:, slot] > 0).all(), slot
    assert (tr[:, 1] >= tr[:, 0]).all() and (tr[:, 2] >= tr[:, 1]).all() and (tr[:, 3] >= tr[:, 2]).all()
    gemm = tr[:, 10] > 0  # CTAs whose GEMM role issued at least one MMA
    assert gemm.sum() > 0
    assert (tr[gemm, 10] >= tr[gemm, 6]).all() and (tr[gemm, 11] >= tr[gemm, 10]).all()
    assert (tr[gemm, 15] >= tr[gemm, 11]).all() and (tr[gemm, 7] >= tr[gemm, 6]).all()


def test_two_streams_at_once():
    """Calls on two streams, enqueued back to back without synchronising:
    each stream has its own cached workspace and both results are right."""
    a_in = gu.to_device(*_inputs(1200, 256, 512, 8, 2, seed=51))
    b_in = gu.to_device(*_inputs(700, 256, 384, 16, 4, seed=52))
    ref_a = gu.run_gpu(*a_in, 2)
    ref_b = gu.run_gpu(*b_in, 4)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    outs = []
    for _ in range(3):
        with torch.cuda.stream(s1):
            oa = mk.moe_dispatch_gemm(*a_in, 2, stream=s1, check=False)
        with torch.cuda.stream(s2):
            ob = mk.moe_dispatch_gemm(*b_in, 4, stream=s2, check=False)
        outs.append((oa, ob))
    assert mk.mk_get_status(s1) == mk.MK_OK and mk.mk_get_status(s2) == mk.MK_OK
    for oa, ob in outs:
        assert np.array_equal(oa["y_sorted"].float().cpu().numpy(), ref_a["y"])
        assert np.array_equal(ob["y_sorted"].float().cpu().numpy(), ref_b["y"])
        assert np.array_equal(oa["src_index"].cpu().numpy(), ref_a["src_index"])
        assert np.array_equal(ob["src_index"].cpu().numpy(), ref_b["src_index"])
