"""The host-buffer entry point with streamed results: the kernel raises a
flag per chunk of finished rows and a second stream copies each chunk to the
host while the GEMM goes on.  Its outputs must equal the device path's bit
for bit, whatever the chunking, and a call that gives up must still return
(the last CTA out releases every chunk)."""
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


def _host_call(x, l, Wd, k, cfg=None):
    T, H = x.shape
    E, _, F = Wd.shape
    f32 = cfg is not None and cfg.out_dtype == mk.MK_OUT_F32
    xh = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).pin_memory()
    lh = torch.from_numpy(l).pin_memory()
    yh = torch.empty((T * k, F), dtype=torch.float32 if f32 else torch.int16).pin_memory()
    yh.fill_(-1)
    sh = torch.empty(T * k, dtype=torch.int32).pin_memory()
    oh = torch.empty(E + 1, dtype=torch.int32).pin_memory()
    gh = torch.empty(T * k, dtype=torch.float32).pin_memory()
    st = mk.mk_moe_dispatch_gemm_host(xh, lh, T, H, E, k, Wd, F, yh, sh, oh, gh, None, cfg)
    return st, dict(y=yh.numpy().copy(), src_index=sh.numpy().copy(), expert_offsets=oh.numpy().copy(),
                    gate_w=gh.numpy().copy())


def _device_call(x, l, Wd, k, cfg=None):
    xd, ld, _ = gu.to_device(x, l, np.zeros((1, 1, 1), np.uint16))
    o = mk.moe_dispatch_gemm(xd, ld, Wd, k, cfg=cfg)
    torch.cuda.synchronize()
    y = o["y_sorted"]
    y = y.view(torch.int16).cpu().numpy() if y.dtype == torch.bfloat16 else y.cpu().numpy()
    return dict(y=y, src_index=o["src_index"].cpu().numpy(), expert_offsets=o["expert_offsets"].cpu().numpy(),
                gate_w=o["gate_w"].cpu().numpy())


@pytest.mark.parametrize("shape", [
    (333, 128, 256, 8, 2),      # 666 rows: three chunks of 256, the last ragged; copies of 1, 1, 1
    (100, 128, 192, 4, 2),      # one chunk, partial N-block
    (20000, 128, 128, 16, 2),   # 40000 rows: 53 chunks of 768; copies of 1, 1, 2, 4, 8, 16, 21
    (5000, 256, 512, 64, 8),
], ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("out_dtype", [mk.MK_OUT_BF16, mk.MK_OUT_F32], ids=["bf16", "f32"])
def test_streamed_host_results_equal_device(shape, out_dtype):
    T, H, F, E, k = shape
    x, l, W = _inputs(T, H, F, E, k, seed=T + k)
    Wd = gu.to_device(x, l, W)[2]
    cfg = mk.make_config(out_dtype=out_dtype)
    st, h = _host_call(x, l, Wd, k, cfg)
    assert st == mk.MK_OK
    d = _device_call(x, l, Wd, k, cfg)
    for key in d:
        np.testing.assert_array_equal(h[key], d[key])


def test_repeated_and_non_streamed_calls():
    """Sequence numbers advance call after call; the SM-pair configuration
    (no chunk flags) copies after the kernel, same bytes."""
    T, H, F, E, k = 3000, 128, 256, 8, 2
    x, l, W = _inputs(T, H, F, E, k, seed=21)
    Wd = gu.to_device(x, l, W)[2]
    d = _device_call(x, l, Wd, k)
    for _ in range(4):
        st, h = _host_call(x, l, Wd, k)
        assert st == mk.MK_OK
        np.testing.assert_array_equal(h["y"], d["y"])
    st, h = _host_call(x, l, Wd, k, mk.make_config(mma_pair=mk.MK_MMA_PAIR))
    assert st == mk.MK_OK and mk.mk_last_launch_info()["mma_pair"] == mk.MK_MMA_PAIR
    np.testing.assert_array_equal(h["y"], d["y"])
    st, h = _host_call(x, l, Wd, k)
    assert st == mk.MK_OK
    np.testing.assert_array_equal(h["y"], d["y"])


def test_call_that_gives_up_still_returns():
    w = synth.WORKLOADS[1]
    x, l, W = synth.make_inputs(w)
    Wd = gu.to_device(x, l, W)[2]
    cfg = mk.make_config(debug_fault=mk.MK_FAULT_DROP_TILE_FLAG, spin_limit_ns=50_000_000)
    st, _ = _host_call(x, l, Wd, w.k, cfg)
    assert st == mk.MK_ERR_TIMEOUT
    st, h = _host_call(x, l, Wd, w.k)
    assert st == mk.MK_OK
    ref = gu.oracle_reference(x, l, W, w.k)
    g = dict(h, y=synth.bf16_bits_to_f32(h["y"].view(np.uint16)))
    gu.assert_routing_exact(g, ref)
    gu.assert_y(g, ref, mk.MK_OUT_BF16)


def test_streamed_host_full_size_mixtral_like():
    w = synth.WORKLOADS[2]
    x, l, W = synth.make_inputs(w)
    Wd = gu.to_device(x, l, W)[2]
    del W
    st, h = _host_call(x, l, Wd, w.k)
    assert st == mk.MK_OK
    d = _device_call(x, l, Wd, w.k)
    for key in d:
        np.testing.assert_array_equal(h[key], d[key])


def test_host_entry_orders_work_tile_by_tile():
    """With the work order left to the library, the host entry takes all
    N-blocks of a tile together (groups as wide as the N-blocks), so its
    streamed rows complete in order; a caller's group width is kept.  The
    bytes equal the device path's, whose order groups N-blocks."""
    T, H, F, E, k = 256, 4096, 8192, 2, 1  # 64 MiB of weights per expert: the device path groups 4 of 32 N-blocks
    x, l, W = _inputs(T, H, F, E, k, seed=5)
    Wd = gu.to_device(x, l, W)[2]
    d = _device_call(x, l, Wd, k)
    assert mk.mk_last_launch_info()["n_group"] == 4
    st, h = _host_call(x, l, Wd, k)
    assert st == mk.MK_OK and mk.mk_last_launch_info()["n_group"] == F // 256
    for key in d:
        np.testing.assert_array_equal(h[key], d[key])
    st, h = _host_call(x, l, Wd, k, mk.make_config(n_group=8))
    assert st == mk.MK_OK and mk.mk_last_launch_info()["n_group"] == 8
    np.testing.assert_array_equal(h["y"], d["y"])
