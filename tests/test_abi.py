"""The C-ABI library loads, exports every symbol include/mk.h declares, and
rejects bad arguments synchronously (no GPU needed: validation precedes any
CUDA call)."""
import ctypes
import os
import re

import pytest

import moe_token_dispatch_persistent_gb300 as mk
from moe_token_dispatch_persistent_gb300 import build as mkbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    mkbuild.build()
    return mk.lib()


def _declared():
    names = set()
    for h in os.listdir(os.path.join(ROOT, "include")):
        if not h.endswith(".h"):
            continue
        src = open(os.path.join(ROOT, "include", h)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names |= set(re.findall(r"\b(mk_[a-z0-9_]+)\s*\(", src))
    return names


def test_header_and_binding_agree():
    assert _declared() == set(mk.ABI_FUNCTIONS)


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings(lib):
    for s, name in [(0, "MK_OK"), (1, "MK_ERR_INVALID_ARG"), (4, "MK_ERR_TIMEOUT"), (7, "MK_ERR_WORKSPACE")]:
        assert mk.mk_status_string(s) == name
    assert mk.mk_version() >= 100


def test_config_defaults(lib):
    c = mk.mk_config_default()
    assert c.mode == mk.MK_MODE_FUSED and c.out_dtype == mk.MK_OUT_BF16
    assert c.dispatch_ctas == 0 and c.spin_limit_ns == 0 and list(c.reserved) == [0] * 4 and c.l2_prefetch == 0
    assert c.mma_pair == mk.MK_MMA_AUTO and c.gather == mk.MK_GATHER_AUTO


def test_struct_layouts_match_header(lib):
    assert ctypes.sizeof(mk.mk_config_t) == 64
    assert ctypes.sizeof(mk.mk_launch_info_t) == 40


@pytest.mark.parametrize("T,H,E,k,F,want", [
    (-1, 512, 8, 2, 1024, mk.MK_ERR_INVALID_ARG),   # negative T
    (16, 512, 8, 0, 1024, mk.MK_ERR_INVALID_ARG),   # k = 0
    (16, 512, 4, 5, 1024, mk.MK_ERR_INVALID_ARG),   # k > E
    (16, 512, 16, 9, 1024, mk.MK_ERR_INVALID_ARG),  # k > 8
    (16, 500, 8, 2, 1024, mk.MK_ERR_INVALID_ARG),   # H not a multiple of 64
    (16, 512, 8, 2, 1000, mk.MK_ERR_INVALID_ARG),   # F not a multiple of 64
    (16, 512, 300, 2, 1024, mk.MK_ERR_UNSUPPORTED),  # E > 256
    (16, 65536, 8, 2, 1024, mk.MK_ERR_UNSUPPORTED),  # H too large
    (2 ** 29, 512, 8, 8, 1024, mk.MK_ERR_UNSUPPORTED),  # T*k >= 2^31
])
def test_size_validation_is_synchronous(lib, T, H, E, k, F, want):
    st = mk.mk_moe_dispatch_gemm_ex(16, 16, T, H, E, k, 16, F, 16, 16, 16, 16, 1)
    assert st == want


def test_workspace_size(lib):
    assert mk.mk_workspace_size(4096, 4096, 14336, 8, 2) >= 4096 * 2 * 4096 * 2
    assert mk.mk_workspace_size(4096, 4000, 14336, 8, 2) == 0
    # grows with T*k*H (staging rows)
    a = mk.mk_workspace_size(1000, 512, 1024, 8, 2)
    b = mk.mk_workspace_size(2000, 512, 1024, 8, 2)
    assert b - a >= 1000 * 2 * 512 * 2


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(mk.MkLibraryMissing):
        mk.lib(str(tmp_path / "nope.so"))


def test_ep_workspace_size(lib):
    T, H, F, E, k = 4096, 4096, 14336, 8, 2
    for R in (1, 2, 4, 8):
        n = mk.mk_ep_workspace_size(T, H, F, E, k, R)
        # each rank can receive T * min(k, E/R) rows of H bf16 values
        assert n >= R * T * min(k, E // R) * H * 2
    assert mk.mk_ep_workspace_size(T, H, F, E, k, 3) == 0   # E not divisible by the ranks
    assert mk.mk_ep_workspace_size(T, H, F, E, k, 0) == 0
    assert mk.mk_ep_workspace_size(T, H, F, 16, k, 16) == 0  # more than 8 ranks
    assert mk.mk_ep_workspace_size(T, 4000, F, E, k, 2) == 0


def test_ep_argument_validation_is_synchronous(lib):
    # ranks must divide E and lie in 1..8; checked before any device work
    for R in (0, 3, 9):
        assert mk.mk_moe_ep_sim(16, 16, 64, 512, 8, 2, 16, 1024, R, 16, 16, 16, 16, 16, 1) == mk.MK_ERR_INVALID_ARG
