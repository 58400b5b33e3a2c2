"""Seeded synthetic inputs for the MoE dispatch + expert-GEMM path.

This module is the only code shared by the CUDA path's tests/bench and the
CPU oracle.  It holds no routing, scan, gather or GEMM arithmetic: it only
draws the inputs (router logits, token activations, expert weights) with the
shapes and value distributions of the five workloads, and rounds float32
draws to bf16 bit patterns.

Recipe (per workload, all draws from ``numpy.random.default_rng``):

* ``SeedSequence(seed).spawn(2 + E)`` gives independent streams:
  child 0 -> logits (and the workload's logit modifications),
  child 1 -> x, child 2+e -> W[e].  Per-expert streams let any expert's
  weights be regenerated alone (sampled checks) and in parallel.
* logits: ``standard_normal((T, E), float32)``; then
    - "skewed": add ``b_e = 2*ln(w_{e+1})`` with Zipf(s=1.2) rank weights
      ``w_r = r**-1.2 / sum_j j**-1.2`` (in float64, rounded to float32);
      expert 0 is the hottest;
    - "imbalanced": a Bernoulli(0.1) token mask (``random(T) < 0.1``) gets
      +6 on expert 0 (float32), then 16 experts drawn without replacement
      from 1..E-1 are set to -inf for every token.
* x: ``standard_normal((T, H), float32)`` rounded to bf16 (nearest-even).
* W[e]: ``standard_normal((H, F), float32) / float32(sqrt(H))`` rounded to
  bf16 (nearest-even).

bf16 values travel as ``uint16`` bit patterns (numpy has no bf16 dtype).
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    F: int
    E: int
    k: int
    seed: int
    kind: str = "normal"  # "normal" | "skewed" | "imbalanced"

    @property
    def rows(self) -> int:
        return self.T * self.k

    @property
    def flop(self) -> int:
        return 2 * self.T * self.k * self.H * self.F

    def describe(self) -> str:
        return f"{self.name}(T={self.T},H={self.H},F={self.F},E={self.E},k={self.k},seed={self.seed})"


# The five workloads the path is measured and checked on.
WORKLOADS = {
    1: Workload("tiny", 256, 512, 1024, 8, 2, 0),
    2: Workload("mixtral_like", 4096, 4096, 14336, 8, 2, 1),
    3: Workload("fine_grained_skewed", 8192, 7168, 2048, 256, 8, 2, "skewed"),
    4: Workload("decode", 128, 7168, 2048, 256, 8, 3),
    5: Workload("imbalanced_large_batch", 16384, 4096, 1536, 128, 8, 4, "imbalanced"),
}


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); return uint16 bits."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32)
    return ((u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _streams(w: Workload):
    return np.random.SeedSequence(w.seed).spawn(2 + w.E)


def zipf_bias(E: int, s: float = 1.2) -> np.ndarray:
    """Per-expert logit bias 2*ln(w_r), r = e+1, Zipf(s) rank weights (float64)."""
    r = np.arange(1, E + 1, dtype=np.float64)
    w = r ** (-s)
    w /= w.sum()
    return 2.0 * np.log(w)


def make_logits(w: Workload, streams=None) -> np.ndarray:
    ch = streams if streams is not None else _streams(w)
    rng = np.random.default_rng(ch[0])
    logits = rng.standard_normal((w.T, w.E), dtype=np.float32)
    if w.kind == "skewed":
        logits = (logits.astype(np.float64) + zipf_bias(w.E)[None, :]).astype(np.float32)
    elif w.kind == "imbalanced":
        hot = rng.random(w.T) < 0.1
        logits[hot, 0] += np.float32(6.0)
        dead = rng.choice(np.arange(1, w.E), size=min(16, w.E - 1), replace=False)
        logits[:, dead] = -np.inf
    return np.ascontiguousarray(logits)


def make_x(w: Workload, streams=None) -> np.ndarray:
    ch = streams if streams is not None else _streams(w)
    rng = np.random.default_rng(ch[1])
    return f32_to_bf16_bits(rng.standard_normal((w.T, w.H), dtype=np.float32))


def make_w_expert(w: Workload, e: int, streams=None) -> np.ndarray:
    """W[e] as uint16 bf16 bits, shape (H, F)."""
    ch = streams if streams is not None else _streams(w)
    rng = np.random.default_rng(ch[2 + e])
    a = rng.standard_normal((w.H, w.F), dtype=np.float32)
    a /= np.float32(math.sqrt(w.H))
    return f32_to_bf16_bits(a)


def make_w(w: Workload, out: np.ndarray | None = None, threads: int | None = None) -> np.ndarray:
    """All expert weights, shape (E, H, F) uint16 bf16 bits (threaded per expert)."""
    ch = _streams(w)
    if out is None:
        out = np.empty((w.E, w.H, w.F), dtype=np.uint16)
    n = threads or min(16, os.cpu_count() or 1)

    def one(e):
        out[e] = make_w_expert(w, e, ch)

    with ThreadPoolExecutor(n) as ex:
        list(ex.map(one, range(w.E)))
    return out


def make_inputs(w: Workload, with_w: bool = True):
    """(x_bits[T,H] u16, logits[T,E] f32, W_bits[E,H,F] u16 or None)."""
    ch = _streams(w)
    logits = make_logits(w, ch)
    x = make_x(w, ch)
    W = make_w(w) if with_w else None
    return x, logits, W


def small_workload(T, H, F, E, k, seed=0, kind="normal", name="custom") -> Workload:
    return Workload(name, T, H, F, E, k, seed, kind)
