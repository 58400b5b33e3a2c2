"""Plant plausible mistakes in a copy of the oracle and check the pins catch each.

Every mutation is a one-spot edit of ``oracle/mk_oracle.c`` (a flipped
tie-break, a dropped or sign-flipped gate term, an inclusive scan, a swapped
sort key, a transposed weight, a wrong token index ...).  Each mutant is
compiled on the CPU into a temporary library and run through the same checks
as the real oracle; at least one check must fail, otherwise the pins would not
notice that mistake.
"""
import os

import pytest

import pins
from oracle import build as obuild
from oracle.oracle import Oracle

SRC = os.path.join(os.path.dirname(obuild.__file__), "mk_oracle.c")

MUTANTS = {
    "tie_break_higher_id": ("if (l[a] == l[b] && a < b) return 1;", "if (l[a] == l[b] && a > b) return 1;"),
    "ties_by_ge": ("if (l[a] > l[b]) return 1;", "if (l[a] >= l[b]) return 1;"),
    "ascending_logit": ("if (l[a] > l[b]) return 1;", "if (l[a] < l[b]) return 1;"),
    "gate_sum_drops_slot0": ("for (int j = 0; j < k; ++j) s += exp(", "for (int j = 1; j < k; ++j) s += exp("),
    "gate_sign_flip": ("(float)(exp((double)l[topk_idx[t * k + j]] - l0) / s)",
                       "(float)(exp(l0 - (double)l[topk_idx[t * k + j]]) / s)"),
    "gate_no_normalise": ("(float)(exp((double)l[topk_idx[t * k + j]] - l0) / s)",
                          "(float)(exp((double)l[topk_idx[t * k + j]] - l0))"),
    "inclusive_scan": ("        expert_offsets[e] = (int32_t)run;\n        run += count[e];",
                       "        run += count[e];\n        expert_offsets[e] = (int32_t)run;"),
    "order_e_j_t": ("        for (int64_t t = 0; t < T; ++t)\n            for (int j = 0; j < k; ++j)\n                if (topk_idx",
                    "        for (int j = 0; j < k; ++j)\n            for (int64_t t = 0; t < T; ++t)\n                if (topk_idx"),
    "src_index_slot_major": ("src_index[r] = (int32_t)(t * k + j);", "src_index[r] = (int32_t)(j * T + t);"),
    "gate_w_token_order": ("gate_w[r] = topk_gate[t * k + j];", "gate_w[r] = topk_gate[r];"),
    "transposed_w": ("yr[f] += xv * bf16_to_double(wrow[f]);", "yr[f] += xv * bf16_to_double(We[(int64_t)f * H + h]);"),
    "wrong_token": ("const int64_t t = src_index[r] / k;\n        const uint16_t* xt = x + t * (int64_t)H;\n        const uint16_t* We",
                    "const int64_t t = r / k;\n        const uint16_t* xt = x + t * (int64_t)H;\n        const uint16_t* We"),
    "dropped_first_h": ("for (int h = 0; h < H; ++h) {\n            const double xv = bf16_to_double(xt[h]);\n            const uint16_t* wrow",
                        "for (int h = 1; h < H; ++h) {\n            const double xv = bf16_to_double(xt[h]);\n            const uint16_t* wrow"),
    "wrong_expert_weights": ("const uint16_t* We = W + (int64_t)e * H * F;", "const uint16_t* We = W;"),
    "bf16_decode_shift": ("uint32_t u = (uint32_t)b << 16;", "uint32_t u = (uint32_t)b << 15;"),
    "combine_wrong_token": ("const int64_t t = src_index[r] / k;\n        const double g", "const int64_t t = src_index[r] % k;\n        const double g"),
    "combine_ignores_gate": ("const double g = (double)gate_w[r];", "const double g = 1.0;"),
    "combine_overwrites": ("out[t * F + f] += g * y[r * F + f];", "out[t * F + f] = g * y[r * F + f];"),
    "gated_exp_sign": ("yr[f] = a[f] / (1.0 + exp(-a[f])) * b[f];", "yr[f] = a[f] / (1.0 + exp(a[f])) * b[f];"),
    "gated_swapped_projections": ("yr[f] = a[f] / (1.0 + exp(-a[f])) * b[f];", "yr[f] = b[f] / (1.0 + exp(-b[f])) * a[f];"),
    "gated_no_up_projection": ("yr[f] = a[f] / (1.0 + exp(-a[f])) * b[f];", "yr[f] = a[f] / (1.0 + exp(-a[f]));"),
    "gated_w3_is_w1": ("const uint16_t* W3e = W3 + (int64_t)e * H * F;", "const uint16_t* W3e = W1 + (int64_t)e * H * F;"),
    "combine_uniform_gate": ("const double g = (double)gate_w[r];", "const double g = 1.0 / k;"),
    "ep_sources_reversed": ("block[(int64_t)r * E + e] = run;", "block[(int64_t)(R - 1 - r) * E + e] = run;"),
    "ep_rank_major_blocks": ("for (int e = q * epr; e < (q + 1) * epr; ++e)\n            for (int r = 0; r < R; ++r) {",
                             "for (int r = 0; r < R; ++r)\n            for (int e = q * epr; e < (q + 1) * epr; ++e) {"),
    "ep_strided_experts": ("for (int e = q * epr; e < (q + 1) * epr; ++e)", "for (int e = q; e < E; e += R)"),
    "ep_token_split_ceil": ("static int64_t ep_token0(int64_t T, int R, int r) { return (T * (int64_t)r) / R; }",
                            "static int64_t ep_token0(int64_t T, int R, int r) { return (T * (int64_t)r + R - 1) / R; }"),
    "ep_counts_double": ("cnt[(int64_t)r * E + topk_idx[t * k + j]] += 1;", "cnt[(int64_t)r * E + topk_idx[t * k + j]] += 1 + (j > 0);"),
}


def _fails_some_check(o):
    failures = []
    for check in pins.ALL_CHECKS:
        try:
            check(o)
        except Exception as exc:  # an assertion, or a crash-free error return
            failures.append(f"{check.__name__}: {type(exc).__name__}")
    return failures


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    with open(SRC) as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mutated = tmp_path / "mk_oracle.c"
    mutated.write_text(src.replace(old, new))
    (tmp_path / "mk_oracle.h").write_text(open(os.path.join(os.path.dirname(SRC), "mk_oracle.h")).read())
    so = obuild.build(str(mutated), str(tmp_path / "libmutant.so"), force=True)
    failures = _fails_some_check(Oracle(so))
    assert failures, f"no pin caught mutant {name}"
