"""Plant plausible mistakes in a private copy of the oracle and check that the
pins catch each one.  Everything here runs on the CPU; the real oracle is
never modified.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "moe_oracle.c")

MUTATIONS = {
    # ties go to the higher expert index
    "tie_rule": ("if (best < 0 || L[e] > L[best]) best = e;",
                 "if (best < 0 || L[e] >= L[best]) best = e;"),
    # destination order by slot before token
    "perm_order": ("for (int t = 0; t < T; ++t)\n            for (int j = 0; j < k; ++j)\n                if (topk_idx",
                   "for (int j = 0; j < k; ++j)\n            for (int t = 0; t < T; ++t)\n                if (topk_idx"),
    # softmax denominator drops one term
    "softmax_sum": ("\n        for (int e = 0; e < E; ++e) s += exp((double)L[e] - m);",
                    "\n        for (int e = 1; e < E; ++e) s += exp((double)L[e] - m);"),
    # the same slip in the gates of given picks
    "gates_softmax_sum": ("\n            for (int e = 0; e < E; ++e) s += exp((double)L[e] - m);",
                          "\n            for (int e = 1; e < E; ++e) s += exp((double)L[e] - m);"),
    # transposed weight operand
    "gemm_transpose": ("const uint16_t* wrow = We + (size_t)i * N;\n                for (int n = 0; n < N; ++n) acc[n] += a * bf16_to_double(wrow[n]);",
                       "for (int n = 0; n < N; ++n) acc[n] += a * bf16_to_double(We[((size_t)n * d + i) % ((size_t)d * N)]);"),
    # gather by slot index instead of token index
    "gather_index": ("int t = perm[row] / k;", "int t = perm[row] % T;"),
    # combine weights indexed by token instead of slot
    "combine_weight": ("acc += w[s] * Y[(size_t)dest[s] * N + n];", "acc += w[t] * Y[(size_t)dest[s] * N + n];"),
    # renormalised gates: denominator drops the first pick
    "renorm_sum": ("for (int j = 0; j < k; ++j) s += exp((double)L[sel[j]] - M);",
                   "for (int j = 1; j < k; ++j) s += exp((double)L[sel[j]] - M);"),
    # renormalised gates: numerator taken from the wrong slot
    "renorm_slot": ("topk_w[(size_t)t * k + j] = exp((double)L[sel[j]] - M) / s;",
                    "topk_w[(size_t)t * k + j] = exp((double)L[sel[k - 1 - j]] - M) / s;"),
    # selection bias subtracted instead of added
    "bias_sign": ("volatile float sum = logits[(size_t)t * E + e] + bias[e];",
                  "volatile float sum = logits[(size_t)t * E + e] - bias[e];"),
    # logistic with the wrong sign
    "sigmoid_sign": ("w[j] = 1.0 / (1.0 + exp(-(double)L[sel[j]]));",
                     "w[j] = 1.0 / (1.0 + exp((double)L[sel[j]]));"),
    # ties between equal keys go to the higher index
    "bias_tie": ("if (best < 0 || key[e] > key[best]) best = e;",
                 "if (best < 0 || key[e] >= key[best]) best = e;"),
    # gated activation applied to the up half instead of the gate half
    "swiglu_swap": ("H[(size_t)i * F + f] = g / (1.0 + exp(-g)) * u;",
                    "H[(size_t)i * F + f] = u / (1.0 + exp(-u)) * g;"),
    # bf16 rounding: ties away from zero instead of to even
    "round_tie": ("if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;",
                  "if (frac >= 0.5) r += 1.0;"),
    # histogram off by one in the prefix sum
    "prefix": ("offsets[e + 1] = offsets[e] + counts[e];", "offsets[e + 1] = offsets[e] + counts[e] + (e == 0);"),
}


def _build_mutant(tmp_path, name):
    before, after = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(before) == 1, name
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(before, after))
    so = tmp_path / f"{name}.so"
    subprocess.check_call(["gcc", "-O1", "-ffp-contract=off", "-fPIC", "-shared", "-o", str(so), str(path), "-lm"])
    return so


def _swap_lib(oracle_mod, so):
    import oracle.oracle as o
    o._load()
    saved = o._lib
    o._lib = None
    real = o._LIB_PATH
    o._LIB_PATH = str(so)
    build = o.build_oracle
    o.build_oracle = lambda force=False: str(so)
    try:
        o._load()
    finally:
        o._LIB_PATH = real
        o.build_oracle = build
    return saved


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_mutation(tmp_path, oracle_mod, name):
    import oracle.oracle as o
    import tests.test_oracle_pins as pins
    so = _build_mutant(tmp_path, name)
    saved = _swap_lib(oracle_mod, so)
    try:
        checks = [
            lambda: pins.test_handworked_example(o),
            *[(lambda s=s: pins.test_topk_matches_full_sort(o, s)) for s in range(6)],
            lambda: pins.test_topk_special_cases(o),
            lambda: pins.test_gate_weight_two_experts_is_logistic(o),
            lambda: pins.test_renorm_gates_closed_forms(o),
            lambda: pins.test_renorm_gates_ignore_unchosen_logits(o),
            lambda: pins.test_biased_selection_brute_force(o),
            lambda: pins.test_biased_selection_forces_the_biased_experts(o),
            lambda: pins.test_gates_at_closed_forms(o),
            lambda: pins.test_swiglu_closed_forms(o),
            lambda: pins.test_round_bf16_ties_and_library(o),
            *[(lambda s=s: pins.test_histogram_and_permutation_brute_force(o, s)) for s in range(4)],
            lambda: pins.test_gather_is_fancy_index(o),
            lambda: pins.test_gemm_single_expert_is_plain_matmul(o),
            lambda: pins.test_gemm_uses_each_rows_own_expert(o),
            lambda: pins.test_combine_single_slot_unit_gate_undoes_the_permutation(o),
            lambda: pins.test_combine_matches_fancy_index_sum(o),
            lambda: pins.test_combine_k_equals_e_with_constant_expert_outputs(o),
        ]
        caught = 0
        for c in checks:
            try:
                c()
            except (AssertionError, ValueError):
                caught += 1
        assert caught > 0, f"mutation {name} passed every pin"
    finally:
        o._lib = saved
