"""Routing with a token's experts split over 2, 4 or 8 lanes (E = 64, 128,
256) against the CPU oracle.

The split form reads each lane's share of a token's logits with 16-byte
loads, keeps that share's best k, and merges the lanes' lists with warp
shuffles.  The best k under the key (value desc, expert id asc) is unique, so
the expert lists, offsets and src_index must match the oracle bit for bit and
the gates within 2e-6, as for one lane per token.  Token counts straddle the
chunk sizes (224 / lanes tokens) and the rows of a warp (32 / lanes tokens);
logits cover ties, -inf and skew."""
import numpy as np
import pytest

import moe_token_dispatch_persistent_gb300 as mk
from moe_token_dispatch_persistent_gb300 import synth

import gpu_util as gu
from oracle.oracle import Oracle

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


@pytest.fixture(scope="module")
def orc():
    return Oracle()


def _logits(T, E, kind, seed):
    rng = np.random.default_rng(seed)
    l = rng.standard_normal((T, E), dtype=np.float32)
    if kind == "ties":
        l = np.round(l * 2.0).astype(np.float32)  # a handful of distinct values per row
    elif kind == "neg_inf":
        l[rng.random((T, E)) < 0.9] = -np.inf
        l[::7, :] = -np.inf  # rows with nothing finite
    elif kind == "skewed":
        l = (l.astype(np.float64) + synth.zipf_bias(E)[None, :]).astype(np.float32)
    elif kind == "equal":
        l[:] = 0.5
    return np.ascontiguousarray(l)


def _route_gpu(l_dev, T, E, k, cfg):
    H, F = 64, 64
    x = torch.zeros((T, H), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((E, H, F), dtype=torch.bfloat16, device="cuda")
    o = mk.alloc_outputs(T, F, E, k)
    st = mk.mk_moe_dispatch_gemm_ex(x, l_dev, T, H, E, k, W, F, o["y_sorted"], o["src_index"],
                                    o["expert_offsets"], o["gate_w"], None, cfg)
    assert st == mk.MK_OK, mk.status_name(st)
    assert mk.mk_get_status() == mk.MK_OK
    info = mk.mk_last_launch_info()
    return ({key: o[key].cpu().numpy() for key in ("src_index", "expert_offsets", "gate_w")}, info)


def _check(orc, l, k, g):
    idx, gate = orc.route(l, k)
    offsets, src, gw = orc.dispatch(idx, gate, l.shape[1])
    np.testing.assert_array_equal(g["expert_offsets"], offsets)
    np.testing.assert_array_equal(g["src_index"], src)
    assert np.abs(g["gate_w"].astype(np.float64) - gw).max(initial=0.0) <= gu.GATE_TOL


DISPATCH = mk.MK_MODE_DISPATCH_ONLY


@pytest.mark.parametrize("E", [64, 128, 256])
@pytest.mark.parametrize("T", [1, 5, 27, 29, 57, 111, 113, 225, 1000, 4099])
@pytest.mark.parametrize("k", [1, 2, 8])
def test_split_routing_matches_oracle(orc, E, T, k):
    l = _logits(T, E, "normal", seed=T * 7 + E + k)
    g, info = _route_gpu(torch.from_numpy(l).cuda(), T, E, k, mk.make_config(mode=DISPATCH))
    assert info["route_lanes"] > 1
    _check(orc, l, k, g)


@pytest.mark.parametrize("kind", ["ties", "neg_inf", "skewed", "equal"])
@pytest.mark.parametrize("E,T", [(64, 300), (128, 333), (256, 130), (256, 1500)])
def test_split_routing_special_logits(orc, kind, E, T):
    k = 8 if kind != "equal" else 4
    l = _logits(T, E, kind, seed=E + T)
    g, info = _route_gpu(torch.from_numpy(l).cuda(), T, E, k, mk.make_config(mode=DISPATCH))
    assert info["route_lanes"] > 1
    _check(orc, l, k, g)
    if kind == "equal":  # ties go to the lowest expert ids
        assert list(np.diff(g["expert_offsets"])[:5]) == [T] * 4 + [0]


@pytest.mark.parametrize("E,T,grid,lanes", [
    (256, 128, 0, 8),      # decode-sized: 5 chunks of 28 tokens
    (256, 8192, 0, 4),     # 8 lanes: 293 chunks; 4 lanes: 147 chunks of 56 (37632 counts, scanned by columns)
    (256, 2048, 0, 8),     # 74 chunks of 28 tokens (18944 counts, scanned by columns)
    (256, 4099, 0, 8),     # 147 chunks of 28 tokens
    (128, 16384, 0, 2),    # 147 chunks of 112 tokens
    (64, 4096, 0, 2),
    (8, 4096, 0, 1),       # other expert counts keep a lane per token
    (8, 120000, 0, 1),     # 536 chunks, 3 or 4 per CTA: 4288 counts, scanned by columns
    (96, 500, 0, 1),
    (256, 1000, 8, 1),     # 8 CTAs: even two lanes give more chunks than CTAs
    (256, 1000, 10, 1),    # two lanes would fit 10 CTAs, but a lane scans at most 64 experts
    (256, 1000, 20, 4),    # 18 chunks of 56 tokens
    (128, 1000, 10, 2),    # 9 chunks of 112 tokens
])
def test_lanes_follow_the_shape(orc, E, T, grid, lanes):
    k = min(8, E)
    l = _logits(T, E, "normal", seed=T + E + grid)
    g, info = _route_gpu(torch.from_numpy(l).cuda(), T, E, k, mk.make_config(mode=DISPATCH, grid_ctas=grid))
    assert info["route_lanes"] == lanes
    assert info["route_chunks"] == -(-T // (224 // lanes))
    _check(orc, l, k, g)


def test_unaligned_logits_keep_a_lane_per_token(orc):
    T, E, k = 500, 256, 8
    l = _logits(T, E, "normal", seed=11)
    buf = torch.empty(T * E + 1, dtype=torch.float32, device="cuda")
    buf[1:].copy_(torch.from_numpy(l.reshape(-1)).cuda())
    l_dev = buf[1:].view(T, E)  # 4-byte aligned, not 16
    g, info = _route_gpu(l_dev, T, E, k, mk.make_config(mode=DISPATCH))
    assert info["route_lanes"] == 1
    _check(orc, l, k, g)


@pytest.mark.parametrize("mode", [mk.MK_MODE_FUSED, mk.MK_MODE_UNFUSED], ids=["fused", "unfused"])
def test_split_routing_full_path(mode):
    """The whole path with split routing: routing exact, y within tolerance."""
    T, H, F, E, k = 700, 256, 512, 128, 8
    rng = np.random.default_rng(5)
    x = synth.f32_to_bf16_bits(rng.standard_normal((T, H), dtype=np.float32))
    W = synth.f32_to_bf16_bits(rng.standard_normal((E, H, F), dtype=np.float32) / np.float32(np.sqrt(H)))
    l = _logits(T, E, "skewed", seed=6)
    ref = gu.oracle_reference(x, l, W, k)
    g = gu.run_gpu(*gu.to_device(x, l, W), k, cfg=mk.make_config(mode=mode))
    assert mk.mk_last_launch_info()["route_lanes"] == 4
    gu.assert_routing_exact(g, ref)
    gu.assert_gates(g, ref)
    gu.assert_y(g, ref, mk.MK_OUT_BF16)
