"""Checks that pin the CPU oracle to facts outside itself.

Each ``check_*`` takes an ``Oracle`` (the committed build or a variant with a
planted mistake) and raises ``AssertionError`` when the oracle disagrees with
something fixed independently of its code:

* brute force over all k-subsets and their orderings (top-k, tie-break);
* closed forms of the gate (k = 1; the logistic form at k = 2; the
  reciprocal form 1 / sum_i exp(l_i - l_j) for any k) and its invariants;
* invariants that together determine the dispatch uniquely (histogram sums,
  monotone offsets, src_index a bijection, rows grouped by expert and
  ascending within each expert);
* the product against ``numpy.matmul`` in float64, a dense per-token loop
  under one-hot routing, and bit-exact identity weights;
* a hand-worked example (``golden/worked_example.json``).

The pages name the operation (MoE Dispatch+GEMM: tokens routed dynamically
to experts, then the dense expert product; zubnet.ai para. 2, lefilia.fr
para. 3) but print no values, so these are the pins there are.
"""
from __future__ import annotations

import itertools
import json
import math
import os

import numpy as np

from moe_token_dispatch_persistent_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---------------------------------------------------------------- top-k ----

def _beats(l, a, b):
    return l[a] > l[b] or (l[a] == l[b] and a < b)


def brute_topk(l, k):
    """The unique k-subset whose every member beats every non-member, in the
    unique order where each slot beats the next (enumeration, no sorting)."""
    E = len(l)
    winners = []
    for S in itertools.combinations(range(E), k):
        rest = [b for b in range(E) if b not in S]
        if all(_beats(l, a, b) for a in S for b in rest):
            winners.append(S)
    assert len(winners) == 1, winners
    orders = [p for p in itertools.permutations(winners[0])
              if all(_beats(l, p[i], p[i + 1]) for i in range(k - 1))]
    assert len(orders) == 1
    return list(orders[0])


def _tie_heavy_logits(rng, T, E, with_neg_inf=True):
    l = rng.integers(-2, 3, size=(T, E)).astype(np.float32)
    if with_neg_inf:
        l[rng.random((T, E)) < 0.2] = -np.inf
    l[0, :] = 1.0  # all equal
    if T > 1:
        l[1, :] = -np.inf  # nothing finite
    return l


def check_topk_bruteforce(o):
    rng = np.random.default_rng(11)
    for E in (1, 2, 3, 5, 6):
        for k in range(1, min(E, 4) + 1):
            l = _tie_heavy_logits(rng, 12, E)
            idx, _ = o.route(l, k)
            for t in range(l.shape[0]):
                assert list(idx[t]) == brute_topk(list(l[t]), k), (E, k, t, l[t], idx[t])
    # continuous logits: no ties
    l = rng.standard_normal((40, 7)).astype(np.float32)
    idx, _ = o.route(l, 3)
    for t in range(40):
        assert list(idx[t]) == brute_topk(list(l[t]), 3)


def check_topk_special_cases(o):
    # all logits equal: experts 0..k-1 in order
    idx, _ = o.route(np.zeros((3, 8), np.float32), 4)
    assert (idx == np.arange(4)[None, :]).all()
    # E == k: every expert, ordered by logit then id
    l = np.array([[0.5, 2.0, 2.0, -1.0]], np.float32)
    idx, _ = o.route(l, 4)
    assert list(idx[0]) == [1, 2, 0, 3]
    # a +6 boost makes expert 0 slot 0
    l = np.zeros((1, 16), np.float32)
    l[0, 0] = 6.0
    idx, _ = o.route(l, 2)
    assert list(idx[0]) == [0, 1]


# ---------------------------------------------------------------- gates ----

def check_gate_closed_forms(o):
    rng = np.random.default_rng(12)
    # k = 1: the gate is exactly 1
    l = rng.standard_normal((50, 9)).astype(np.float32)
    _, g = o.route(l, 1)
    assert (g == 1.0).all()
    # k = 2: logistic of the logit gap
    idx, g = o.route(l, 2)
    for t in range(50):
        d = float(l[t, idx[t, 1]]) - float(l[t, idx[t, 0]])
        g0 = 1.0 / (1.0 + math.exp(d))
        assert abs(g[t, 0] - g0) <= 1e-7 and abs(g[t, 1] - (1.0 - g0)) <= 1e-7, (g[t], g0)
    # any k: g_j = 1 / sum_i exp(l_i - l_j) (normalised at slot j, not slot 0)
    for k in (3, 5, 8):
        ll = (3.0 * rng.standard_normal((30, 11))).astype(np.float32)
        idx, g = o.route(ll, k)
        for t in range(30):
            ch = [float(ll[t, e]) for e in idx[t]]
            for j in range(k):
                ref = 1.0 / sum(math.exp(ci - ch[j]) for ci in ch)
                assert abs(g[t, j] - ref) <= 1e-7 * max(1.0, ref) + 1e-12, (k, t, j, g[t, j], ref)


def check_gate_invariants(o):
    rng = np.random.default_rng(13)
    l = (2.0 * rng.standard_normal((64, 16))).astype(np.float32)
    for k in (2, 4, 8):
        idx, g = o.route(l, k)
        assert np.allclose(g.sum(axis=1), 1.0, atol=1e-6)
        assert (np.diff(g, axis=1) <= 0).all()  # slot order is descending logit
        assert (g > 0).all()
    # shifting every logit by a power of two changes nothing (exact in f32 here)
    li = rng.integers(-8, 9, size=(20, 10)).astype(np.float32) / 4
    i1, g1 = o.route(li, 3)
    i2, g2 = o.route(li + np.float32(16.0), 3)
    assert (i1 == i2).all() and (g1 == g2).all()
    # -inf entries get gate 0; a row with nothing finite gets all zeros
    l = np.full((2, 6), -np.inf, np.float32)
    l[0, 4] = 0.25
    idx, g = o.route(l, 3)
    assert list(idx[0]) == [4, 0, 1] and list(g[0]) == [1.0, 0.0, 0.0]
    assert list(idx[1]) == [0, 1, 2] and (g[1] == 0).all()


# ------------------------------------------------------------- dispatch ----

def check_dispatch_invariants(o):
    rng = np.random.default_rng(14)
    for (T, E, k) in [(1, 1, 1), (7, 3, 2), (129, 5, 3), (300, 16, 4), (64, 8, 8), (0, 4, 2)]:
        l = rng.integers(-3, 4, size=(T, E)).astype(np.float32)
        if E > 2 and T > 0:
            l[:, E - 1] = -np.inf  # forced-empty expert (k < E)
        idx, g = o.route(l, k)
        off, src, gw = o.dispatch(idx, g, E)
        n = T * k
        cnt = np.bincount(idx.ravel(), minlength=E) if n else np.zeros(E, np.int64)
        assert off[0] == 0 and off[E] == n
        assert (np.diff(off) == cnt).all()
        assert sorted(src.tolist()) == list(range(n))  # bijection onto (t, j)
        for e in range(E):
            seg = src[off[e]:off[e + 1]]
            assert (np.diff(seg) > 0).all()  # ascending (token, slot)
            assert (idx.ravel()[seg] == e).all()  # every row belongs to e
            assert np.array_equal(gw[off[e]:off[e + 1]], g.ravel()[seg])
        if E > 2 and k < E and T > 0:
            assert off[E] - off[E - 1] == 0


# --------------------------------------------------------------- product ----

def _bf16(a):
    return synth.f32_to_bf16_bits(np.asarray(a, np.float32))


def check_gemm_vs_numpy(o):
    rng = np.random.default_rng(15)
    for (T, H, F, E, k) in [(5, 8, 6, 3, 2), (9, 16, 5, 4, 3), (4, 3, 7, 2, 1)]:
        x = _bf16(rng.standard_normal((T, H)))
        W = _bf16(rng.standard_normal((E, H, F)))
        l = rng.standard_normal((T, E)).astype(np.float32)
        out = o.full(x, l, W, k)
        xf = synth.bf16_bits_to_f32(x).astype(np.float64)
        Wf = synth.bf16_bits_to_f32(W).astype(np.float64)
        off, src = out["expert_offsets"], out["src_index"]
        for r in range(T * k):
            e = int(np.searchsorted(off, r, side="right") - 1)
            ref = np.matmul(xf[src[r] // k], Wf[e])
            assert np.allclose(out["y"][r], ref, rtol=1e-12, atol=1e-12), (T, H, F, r)


def check_gemm_one_hot_dense_loop(o):
    rng = np.random.default_rng(16)
    T, H, F, E = 6, 5, 4, 3
    x = _bf16(rng.standard_normal((T, H)))
    W = _bf16(rng.standard_normal((E, H, F)))
    owner = rng.integers(0, E, size=T)
    l = np.zeros((T, E), np.float32)
    l[np.arange(T), owner] = 10.0
    out = o.full(x, l, W, 1)
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    Wf = synth.bf16_bits_to_f32(W).astype(np.float64)
    dense = np.zeros((T, F))
    for t in range(T):
        for f in range(F):
            for h in range(H):
                dense[t, f] += xf[t, h] * Wf[owner[t], h, f]
    # one-hot, k=1: sorted row r holds token src[r]
    for r in range(T):
        assert np.array_equal(out["y"][r], dense[out["src_index"][r]])
    assert (out["topk_gate"] == 1.0).all()


def check_identity_weights(o):
    rng = np.random.default_rng(17)
    T, H, F, E, k = 11, 6, 9, 4, 2
    x = _bf16(rng.standard_normal((T, H)))
    Wf = np.zeros((E, H, F), np.float32)
    for e in range(E):
        Wf[e, :, :H] = np.eye(H)
    l = rng.standard_normal((T, E)).astype(np.float32)
    out = o.full(x, l, _bf16(Wf), k)
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    for r in range(T * k):
        assert np.array_equal(out["y"][r, :H], xf[out["src_index"][r] // k])
        assert (out["y"][r, H:] == 0).all()


def check_worked_example(o):
    with open(os.path.join(GOLDEN, "worked_example.json")) as f:
        g = json.load(f)
    l = np.array([[(-np.inf if v == "-inf" else v) for v in row] for row in g["logits"]], np.float32)
    x = _bf16(g["x"])
    W = _bf16(g["W"])
    out = o.full(x, l, W, g["k"])
    assert out["topk_idx"].tolist() == g["topk_idx"]
    assert out["topk_gate"].tolist() == g["topk_gate"]
    assert out["expert_offsets"].tolist() == g["expert_offsets"]
    assert out["src_index"].tolist() == g["src_index"]
    assert out["gate_w"].tolist() == g["gate_w"]
    assert out["y"].tolist() == g["y"]


def check_workload_invariants(o):
    """Statistics the five workloads' recipes fix, on a cheap sub-sample."""
    w5 = synth.WORKLOADS[5]
    l = synth.make_logits(w5)
    idx, g = o.route(l[:2048], w5.k)
    dead = np.where(np.isneginf(l).all(axis=0))[0]
    assert len(dead) == 16 and 0 not in dead
    assert not np.isin(idx, dead).any()  # 112 finite experts >= k
    off, _, _ = o.dispatch(idx, g, w5.E)
    assert (np.diff(off)[dead] == 0).all()
    # expert 0 is the busiest: boosted for ~10% of tokens
    assert np.argmax(np.diff(off)) == 0
    w3 = synth.WORKLOADS[3]
    idx3, _ = o.route(synth.make_logits(w3)[:1024], w3.k)
    assert (idx3 == 0).any(axis=1).mean() > 0.99  # Zipf: expert 0 picked by ~every token
    assert (idx3[:, 0] == 0).mean() > 0.5
    assert len(np.unique(idx3)) < 80


# --------------------------------------------------------------- combine ----

def _oracle_combine(o, x, l, W, k):
    out = o.full(x, l, W, k)
    T = x.shape[0]
    return out, o.combine(out["y"], out["src_index"], out["gate_w"], T, k)


def check_combine_k1_is_the_row(o):
    rng = np.random.default_rng(18)
    T, H, F, E = 9, 8, 6, 4
    x = _bf16(rng.standard_normal((T, H)))
    W = _bf16(rng.standard_normal((E, H, F)))
    out, comb = _oracle_combine(o, x, rng.standard_normal((T, E)).astype(np.float32), W, 1)
    for r, q in enumerate(out["src_index"]):
        assert np.array_equal(comb[q], out["y"][r])  # gate 1, one row per token


def check_combine_shared_weights_is_dense(o):
    """Every expert the same W0: the gates sum to 1, so out = x . W0."""
    rng = np.random.default_rng(19)
    T, H, F, E, k = 12, 10, 7, 5, 3
    x = _bf16(rng.standard_normal((T, H)))
    W0 = rng.standard_normal((H, F))
    W = _bf16(np.repeat(W0[None], E, axis=0))
    _, comb = _oracle_combine(o, x, rng.standard_normal((T, E)).astype(np.float32), W, k)
    ref = np.matmul(synth.bf16_bits_to_f32(x).astype(np.float64), synth.bf16_bits_to_f32(W[0]).astype(np.float64))
    assert np.allclose(comb, ref, rtol=1e-6, atol=1e-6)


def check_combine_scaled_identity_experts(o):
    """W[e] = c_e * I: out[t] = x[t] * sum_j gate[t,j] * c[idx[t,j]]."""
    rng = np.random.default_rng(20)
    T, H, E, k = 15, 6, 6, 3
    c = np.array([1.0, -2.0, 0.5, 4.0, -0.25, 3.0])
    W = _bf16(c[:, None, None] * np.eye(H)[None])
    x = _bf16(rng.standard_normal((T, H)))
    l = rng.standard_normal((T, E)).astype(np.float32)
    idx, gate = o.route(l, k)
    _, comb = _oracle_combine(o, x, l, W, k)
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    for t in range(T):
        s = sum(float(gate[t, j]) * c[idx[t, j]] for j in range(k))
        assert np.allclose(comb[t], xf[t] * s, rtol=1e-12, atol=1e-12), t


# ------------------------------------------------------------ gated FFN ----

def check_gated_vs_numpy(o):
    """silu(x.W1) * (x.W3) with numpy matmuls and silu(z) = z * (1 + tanh(z/2)) / 2."""
    rng = np.random.default_rng(21)
    for (T, H, F, E, k) in [(6, 8, 5, 3, 2), (10, 12, 9, 4, 3)]:
        x = _bf16(rng.standard_normal((T, H)))
        W1 = _bf16(2.0 * rng.standard_normal((E, H, F)))
        W3 = _bf16(rng.standard_normal((E, H, F)))
        l = rng.standard_normal((T, E)).astype(np.float32)
        out = o.gated_full(x, l, W1, W3, k)
        xf = synth.bf16_bits_to_f32(x).astype(np.float64)
        W1f = synth.bf16_bits_to_f32(W1).astype(np.float64)
        W3f = synth.bf16_bits_to_f32(W3).astype(np.float64)
        off, src = out["expert_offsets"], out["src_index"]
        for r in range(T * k):
            e = int(np.searchsorted(off, r, side="right") - 1)
            a = np.matmul(xf[src[r] // k], W1f[e])
            b = np.matmul(xf[src[r] // k], W3f[e])
            ref = a * (1.0 + np.tanh(a / 2.0)) / 2.0 * b
            assert np.allclose(out["y"][r], ref, rtol=1e-11, atol=1e-12), (T, r)


def check_gated_zero_gate_projection(o):
    rng = np.random.default_rng(22)
    T, H, F, E, k = 8, 6, 4, 3, 2
    x = _bf16(rng.standard_normal((T, H)))
    W1 = _bf16(np.zeros((E, H, F)))
    W3 = _bf16(rng.standard_normal((E, H, F)))
    out = o.gated_full(x, rng.standard_normal((T, E)).astype(np.float32), W1, W3, k)
    assert (out["y"] == 0).all()


def check_gated_odd_part(o):
    """One-hot routing to W1 = +I or -I with W3 = I: silu(z) - silu(-z) = z,
    so the two rows of a token differ by x**2."""
    rng = np.random.default_rng(23)
    T, H = 10, 6
    x = _bf16(rng.standard_normal((T, H)))
    eye = np.eye(H)
    W1 = _bf16(np.stack([eye, -eye]))
    W3 = _bf16(np.stack([eye, eye]))
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    hp = o.gated_full(x, np.tile(np.array([[5.0, 0.0]], np.float32), (T, 1)), W1, W3, 1)
    hm = o.gated_full(x, np.tile(np.array([[0.0, 5.0]], np.float32), (T, 1)), W1, W3, 1)
    # one expert per call: sorted rows are the tokens in order
    assert np.allclose(hp["y"] - hm["y"], xf * xf, rtol=1e-13, atol=1e-15)


# ------------------------------------------------------- expert parallel ----

def _ep_cases():
    rng = np.random.default_rng(23)
    for (T, E, k, R) in [(40, 8, 2, 2), (37, 8, 3, 4), (50, 16, 4, 8), (3, 8, 2, 8), (29, 12, 5, 3),
                         (64, 6, 6, 6), (17, 4, 1, 1)]:
        yield T, E, k, R, _tie_heavy_logits(rng, T, E, with_neg_inf=False)


def check_ep_layout_is_the_global_sort(o):
    """Experts and tokens owned in contiguous blocks: the ranks' receive
    buffers, one after another, are the single-device sorted order."""
    for T, E, k, R, l in _ep_cases():
        idx, gate = o.route(l, k)
        offsets, src, _ = o.dispatch(idx, gate, E)
        cnt, roff, rsrc = o.ep_layout(idx, E, R)
        assert np.array_equal(rsrc, src), (T, E, k, R)
        assert np.array_equal(roff, offsets[::E // R]), (T, E, k, R)


def check_ep_exchange_structure(o):
    """Counts by brute force per rank; every received row belongs to one of
    the destination's experts; inside an expert the sources come in rank
    order and each source's tokens lie in its own range, ascending."""
    for T, E, k, R, l in _ep_cases():
        idx, _ = o.route(l, k)
        cnt, roff, rsrc = o.ep_layout(idx, E, R)
        bounds = [T * r // R for r in range(R + 1)]
        owner = lambda t: max(r for r in range(R) if bounds[r] <= t)  # noqa: E731
        for r in range(R):
            for e in range(E):
                n = sum(1 for t in range(bounds[r], bounds[r + 1]) for j in range(k) if idx[t, j] == e)
                assert cnt[r, e] == n, (r, e)
        assert sorted(rsrc.tolist()) == list(range(T * k))
        epr = E // R
        for q in range(R):
            rows = rsrc[roff[q]:roff[q + 1]]
            es = [int(idx[v // k, v % k]) for v in rows]
            assert all(q * epr <= e < (q + 1) * epr for e in es), q
            assert es == sorted(es), q
            assert roff[q + 1] - roff[q] == cnt[:, q * epr:(q + 1) * epr].sum()
            for e in set(es):
                toks = [int(v) // k for v, ee in zip(rows, es) if ee == e]
                srcs = [owner(t) for t in toks]
                assert srcs == sorted(srcs), (q, e)
                assert toks == sorted(toks), (q, e)


ALL_CHECKS = [
    check_topk_bruteforce,
    check_topk_special_cases,
    check_gate_closed_forms,
    check_gate_invariants,
    check_dispatch_invariants,
    check_gemm_vs_numpy,
    check_gemm_one_hot_dense_loop,
    check_identity_weights,
    check_worked_example,
    check_combine_k1_is_the_row,
    check_combine_shared_weights_is_dense,
    check_combine_scaled_identity_experts,
    check_gated_vs_numpy,
    check_gated_zero_gate_projection,
    check_gated_odd_part,
    check_ep_layout_is_the_global_sort,
    check_ep_exchange_structure,
]
