"""ctypes front end of the C oracle (TEST INFRASTRUCTURE ONLY).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg use this module.  It never imports the CUDA library or its binding; its
inputs come from the seeded generator in ``synth.py``.

The oracle computes top-k MoE routing, dispatch and the per-expert product
as written out in ``mk_oracle.h`` (the pages name "MoE Dispatch+GEMM" and
dynamic token routing to experts but print no steps).
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_LIBS: dict[str, ctypes.CDLL] = {}

_i64 = ctypes.c_int64
_int = ctypes.c_int
_p = ctypes.c_void_p


class OracleError(RuntimeError):
    pass


def load(path: str | None = None) -> ctypes.CDLL:
    """Load (building if needed) the oracle library; ``path`` selects a variant build."""
    path = path or _build.build()
    lib = _LIBS.get(path)
    if lib is None:
        lib = ctypes.CDLL(path)
        lib.mko_route.argtypes = [_p, _i64, _int, _int, _p, _p]
        lib.mko_dispatch.argtypes = [_p, _p, _i64, _int, _int, _p, _p, _p]
        lib.mko_expert_rows.argtypes = [_p, _p, _i64, _int, _int, _int, _int, _p, _p, _p, _i64, _p]
        lib.mko_combine.argtypes = [_p, _p, _p, _i64, _int, _int, _p]
        lib.mko_gated_rows.argtypes = [_p, _p, _p, _i64, _int, _int, _int, _int, _p, _p, _p, _i64, _p]
        lib.mko_ep_layout.argtypes = [_p, _i64, _int, _int, _int, _p, _p, _p]
        for f in (lib.mko_route, lib.mko_dispatch, lib.mko_expert_rows, lib.mko_combine, lib.mko_gated_rows,
                  lib.mko_ep_layout):
            f.restype = _int
        lib.mko_num_threads.restype = _int
        _LIBS[path] = lib
    return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(_p)


def _check(rc: int, what: str):
    if rc != 0:
        raise OracleError(f"{what} returned {rc}")


class Oracle:
    """Thin object wrapper so a test can point at a variant build of the oracle."""

    def __init__(self, path: str | None = None):
        self.lib = load(path)

    def num_threads(self) -> int:
        return int(self.lib.mko_num_threads())

    def route(self, logits: np.ndarray, k: int):
        logits = np.ascontiguousarray(logits, dtype=np.float32)
        T, E = logits.shape
        idx = np.zeros((T, k), dtype=np.int32)
        gate = np.zeros((T, k), dtype=np.float32)
        _check(self.lib.mko_route(_ptr(logits), T, E, k, _ptr(idx), _ptr(gate)), "mko_route")
        return idx, gate

    def dispatch(self, idx: np.ndarray, gate: np.ndarray, E: int):
        idx = np.ascontiguousarray(idx, dtype=np.int32)
        gate = np.ascontiguousarray(gate, dtype=np.float32)
        T, k = idx.shape
        offsets = np.zeros(E + 1, dtype=np.int32)
        src = np.zeros(T * k, dtype=np.int32)
        gw = np.zeros(T * k, dtype=np.float32)
        _check(self.lib.mko_dispatch(_ptr(idx), _ptr(gate), T, E, k, _ptr(offsets), _ptr(src), _ptr(gw)),
               "mko_dispatch")
        return offsets, src, gw

    def expert_rows(self, x_bits, W_bits, k, offsets, src, rows):
        """fp64 y for the sorted rows ``rows``; x_bits[T,H], W_bits[E,H,F] uint16 bf16 bits."""
        x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
        W_bits = np.ascontiguousarray(W_bits, dtype=np.uint16)
        T, H = x_bits.shape
        E, H2, F = W_bits.shape
        assert H2 == H
        offsets = np.ascontiguousarray(offsets, dtype=np.int32)
        src = np.ascontiguousarray(src, dtype=np.int32)
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        y = np.zeros((rows.size, F), dtype=np.float64)
        _check(self.lib.mko_expert_rows(_ptr(x_bits), _ptr(W_bits), T, H, F, E, k, _ptr(offsets), _ptr(src),
                                        _ptr(rows), rows.size, _ptr(y)), "mko_expert_rows")
        return y

    def gated_rows(self, x_bits, W1_bits, W3_bits, k, offsets, src, rows):
        """fp64 silu(x.W1) * (x.W3) for the sorted rows ``rows``."""
        x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
        W1_bits = np.ascontiguousarray(W1_bits, dtype=np.uint16)
        W3_bits = np.ascontiguousarray(W3_bits, dtype=np.uint16)
        T, H = x_bits.shape
        E, H2, F = W1_bits.shape
        assert H2 == H and W3_bits.shape == W1_bits.shape
        offsets = np.ascontiguousarray(offsets, dtype=np.int32)
        src = np.ascontiguousarray(src, dtype=np.int32)
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        y = np.zeros((rows.size, F), dtype=np.float64)
        _check(self.lib.mko_gated_rows(_ptr(x_bits), _ptr(W1_bits), _ptr(W3_bits), T, H, F, E, k, _ptr(offsets),
                                       _ptr(src), _ptr(rows), rows.size, _ptr(y)), "mko_gated_rows")
        return y

    def gated_full(self, x_bits, logits, W1_bits, W3_bits, k):
        E = W1_bits.shape[0]
        idx, gate = self.route(logits, k)
        offsets, src, gw = self.dispatch(idx, gate, E)
        y = self.gated_rows(x_bits, W1_bits, W3_bits, k, offsets, src, np.arange(src.size))
        return dict(topk_idx=idx, topk_gate=gate, expert_offsets=offsets, src_index=src, gate_w=gw, y=y)

    def combine(self, y, src, gate_w, T, k):
        """fp64 out[T,F] from the products y[T*k,F] of every sorted row."""
        y = np.ascontiguousarray(y, dtype=np.float64)
        src = np.ascontiguousarray(src, dtype=np.int32)
        gate_w = np.ascontiguousarray(gate_w, dtype=np.float32)
        F = y.shape[1]
        out = np.zeros((T, F), dtype=np.float64)
        _check(self.lib.mko_combine(_ptr(y), _ptr(src), _ptr(gate_w), T, k, F, _ptr(out)), "mko_combine")
        return out

    def ep_layout(self, idx: np.ndarray, E: int, R: int):
        """Expert-parallel exchange over R ranks: (cnt[R,E], recv_offsets[R+1], recv_src[T*k])."""
        idx = np.ascontiguousarray(idx, dtype=np.int32)
        T, k = idx.shape
        cnt = np.zeros((R, E), dtype=np.int32)
        roff = np.zeros(R + 1, dtype=np.int32)
        rsrc = np.zeros(T * k, dtype=np.int32)
        _check(self.lib.mko_ep_layout(_ptr(idx), T, E, k, R, _ptr(cnt), _ptr(roff), _ptr(rsrc)), "mko_ep_layout")
        return cnt, roff, rsrc

    def full(self, x_bits, logits, W_bits, k, rows=None):
        """Every output of the path; ``rows`` limits the fp64 product to a sample."""
        E = W_bits.shape[0]
        idx, gate = self.route(logits, k)
        offsets, src, gw = self.dispatch(idx, gate, E)
        if rows is None:
            rows = np.arange(src.size, dtype=np.int64)
        y = self.expert_rows(x_bits, W_bits, k, offsets, src, rows)
        return dict(topk_idx=idx, topk_gate=gate, expert_offsets=offsets, src_index=src, gate_w=gw,
                    rows=np.asarray(rows, dtype=np.int64), y=y)


_default: Oracle | None = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle()
    return _default


def oracle_threads() -> int:
    return default().num_threads()


def lib_path() -> str:
    return os.path.abspath(_build.build())
