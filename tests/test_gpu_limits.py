"""The largest supported row widths (H = 32768: 64 KiB token rows, three
bulk-copy slots per dispatch CTA; F = 32768: 128 N-blocks per tile) in every
mode, against the oracle on sampled rows and bit for bit across modes; and
zero tokens through every entry point."""
import numpy as np
import pytest

import moe_token_dispatch_persistent_gb300 as mk
from moe_token_dispatch_persistent_gb300 import synth
from oracle.oracle import Oracle

import gpu_util as gu

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

H_MAX = F_MAX = 32768


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


MODES = {
    "staged": dict(),
    "direct": dict(gather=mk.MK_GATHER_DIRECT),
    "pair": dict(mma_pair=mk.MK_MMA_PAIR),
    "unfused": dict(mode=mk.MK_MODE_UNFUSED),
}


@pytest.mark.parametrize("shape", [(300, H_MAX, 256, 4, 2), (300, 128, F_MAX, 4, 2)], ids=["H_max", "F_max"])
def test_widest_rows_every_mode(shape):
    T, H, F, E, k = shape
    x, l, W = _inputs(T, H, F, E, k, seed=H + F)
    xd, ld, Wd = gu.to_device(x, l, W)
    orc = Oracle()
    idx, gate = orc.route(l, k)
    offsets, src, _ = orc.dispatch(idx, gate, E)
    rows = gu.sample_rows(offsets, 12, np.random.default_rng(3), T * k)
    ref = orc.expert_rows(x, W, k, offsets, src, rows)
    first = None
    for name, kw in MODES.items():
        g = gu.run_gpu(xd, ld, Wd, k, cfg=mk.make_config(**kw))
        np.testing.assert_array_equal(g["src_index"], src, err_msg=name)
        np.testing.assert_array_equal(g["expert_offsets"], offsets, err_msg=name)
        err = gu.rel_inf(g["y"][rows], ref)
        assert err <= gu.Y_TOL[mk.MK_OUT_BF16], f"{name}: rel-inf {err:.3e}"
        if first is None:
            first = g
        else:
            np.testing.assert_array_equal(g["y"], first["y"], err_msg=name)


@pytest.mark.parametrize("shape", [(300, H_MAX, 256, 4, 2), (300, 128, F_MAX, 4, 2)], ids=["H_max", "F_max"])
def test_widest_rows_combine_gated_ep(shape):
    T, H, F, E, k = shape
    x, l, W = _inputs(T, H, F, E, k, seed=H + F + 1)
    _, _, W3 = _inputs(T, H, F, E, k, seed=H + F + 2)
    xd, ld, Wd = gu.to_device(x, l, W)
    W3d = gu.to_device(x, l, W3)[2]
    layer = mk.moe_layer(xd, ld, Wd, k)
    ep = mk.moe_ep_sim(xd, ld, Wd, k, 2)
    torch.cuda.synchronize()
    src = layer["src_index"].cpu().numpy()
    assert torch.equal(ep["out"], layer["out"])
    assert torch.equal(ep["y_tok"][torch.from_numpy(src).long().cuda()], layer["y_sorted"])
    gated = mk.moe_gated(xd, ld, Wd, W3d, k)
    torch.cuda.synchronize()
    orc = Oracle()
    offsets = layer["expert_offsets"].cpu().numpy()
    rows = gu.sample_rows(offsets, 8, np.random.default_rng(4), T * k)
    ref = orc.gated_rows(x, W, W3, k, offsets, src, rows)
    err = gu.rel_inf(gated["y_sorted"].float().cpu().numpy()[rows], ref)
    assert err <= gu.Y_TOL[mk.MK_OUT_BF16], f"gated rel-inf {err:.3e}"


def test_zero_tokens_every_entry_point():
    E, H, F, k = 8, 64, 128, 2
    x = torch.empty((0, H), dtype=torch.bfloat16, device="cuda")
    l = torch.empty((0, E), dtype=torch.float32, device="cuda")
    W = torch.zeros((E, H, F), dtype=torch.bfloat16, device="cuda")
    for fn in (lambda: mk.moe_layer(x, l, W, k),
               lambda: mk.moe_gated(x, l, W, W, k),
               lambda: mk.moe_ep_sim(x, l, W, k, 4),
               lambda: mk.moe_dispatch_gemm(x, l, W, k, cfg=mk.make_config(gather=mk.MK_GATHER_DIRECT))):
        o = fn()
        assert o["expert_offsets"].cpu().tolist() == [0] * (E + 1)
    oh = torch.full((E + 1,), -1, dtype=torch.int32).pin_memory()
    st = mk.mk_moe_dispatch_gemm_host(torch.empty(0, dtype=torch.int16).pin_memory(),
                                      torch.empty(0, dtype=torch.float32).pin_memory(), 0, H, E, k, W, F,
                                      None, None, oh, None)
    assert st == mk.MK_OK and oh.tolist() == [0] * (E + 1)
