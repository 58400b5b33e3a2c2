"""The random-shape sweep: T in {1, 7, 127, 129, 1000} x E in {1, 2, 3, 64, 256}
x every k <= min(8, E), small H and F (multiples of 64), seeded normal logits.
Every case runs the fused path with the default configuration and the f32
output, and is compared with the oracle: routing, offsets and src_index bit
for bit, gates within 2e-6, y_sorted within 1e-4 (rel-inf) on every row."""
import numpy as np
import pytest

import moe_token_dispatch_persistent_gb300 as mk
from moe_token_dispatch_persistent_gb300 import synth
from oracle.oracle import Oracle

import gpu_util as gu

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

TS = (1, 7, 127, 129, 1000)
ES = (1, 2, 3, 64, 256)
CASES = [(T, E, k) for T in TS for E in ES for k in range(1, min(8, E) + 1)]


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


def test_sweep_size():
    assert len(CASES) == 5 * (1 + 2 + 3 + 8 + 8)


@pytest.mark.parametrize("T,E,k", CASES, ids=[f"T{T}-E{E}-k{k}" for T, E, k in CASES])
def test_shape_sweep_against_oracle(orc, T, E, k):
    H, F = (128, 192) if E <= 64 else (64, 128)
    rng = np.random.default_rng(1000 * T + 10 * E + k)
    x = synth.f32_to_bf16_bits(rng.standard_normal((T, H), dtype=np.float32))
    W = synth.f32_to_bf16_bits(rng.standard_normal((E, H, F), dtype=np.float32) / np.float32(np.sqrt(H)))
    l = rng.standard_normal((T, E), dtype=np.float32)
    ref = orc.full(x, l, W, k)
    g = gu.run_gpu(*gu.to_device(x, l, W), k, cfg=mk.make_config(out_dtype=mk.MK_OUT_F32))
    gu.assert_routing_exact(g, ref)
    gu.assert_gates(g, ref)
    gu.assert_y(g, ref, mk.MK_OUT_F32)
