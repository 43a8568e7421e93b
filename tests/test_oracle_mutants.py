"""The pins must catch plausible mistakes in the oracle.

Each case plants one mistake (a dropped term, a wrong sign, a wrong index, a
transposed operand, a swapped operand) into a temporary copy of the oracle
source, builds it on the CPU and requires at least one pin of
test_oracle_pins.py to fail against it. The committed oracle is untouched.
"""
import os

import pytest

import oracle
import test_oracle_pins as pins

MUTANTS = {
    "sa_uses_b": ("acc += S[i * N + j] * a[j];", "acc += S[i * N + j] * b[j];"),
    "update_drops_sa_b": (
        "S[i * N + j] = S[i * N + j] * w[j] + v[i] * k[j] + sa[i] * b[j];",
        "S[i * N + j] = S[i * N + j] * w[j] + v[i] * k[j];"),
    "update_transposes_vk": (
        "S[i * N + j] = S[i * N + j] * w[j] + v[i] * k[j] + sa[i] * b[j];",
        "S[i * N + j] = S[i * N + j] * w[j] + v[j] * k[i] + sa[i] * b[j];"),
    "update_decay_row_index": (
        "S[i * N + j] = S[i * N + j] * w[j] + v[i] * k[j] + sa[i] * b[j];",
        "S[i * N + j] = S[i * N + j] * w[i] + v[i] * k[j] + sa[i] * b[j];"),
    "readout_transposed": ("acc += S[i * N + j] * r[j];", "acc += S[j * N + i] * r[j];"),
    "forward_ignores_s_init": (
        "if (s_init) std::memcpy(S.data(), s_init + hd * NN, NN * sizeof(F));", ""),
    "dr_uses_prev_state": ("acc += St[i * N + j] * dy[i];", "acc += Sp[i * N + j] * dy[i];"),
    "dy_r_transposed": ("G[i * N + j] += dy[i] * r[j];", "G[i * N + j] += dy[j] * r[i];"),
    "dk_uses_k": ("ak += G[i * N + j] * v[i];", "ak += G[i * N + j] * k[i];"),
    "db_wrong_index": ("ab += G[i * N + j] * sa[i];", "ab += G[i * N + j] * sa[j];"),
    "dw_uses_next_state": ("aw += G[i * N + j] * Sp[i * N + j];", "aw += G[i * N + j] * St[i * N + j];"),
    "dv_uses_v": ("av += G[i * N + j] * k[j];", "av += G[i * N + j] * v[j];"),
    "dsa_uses_a": ("as += G[i * N + j] * b[j];", "as += G[i * N + j] * a[j];"),
    "da_uses_next_state": ("acc += dsa[i] * Sp[i * N + j];", "acc += dsa[i] * St[i * N + j];"),
    "carry_drops_decay": (
        "G[i * N + j] = G[i * N + j] * w[j] + dsa[i] * a[j];",
        "G[i * N + j] = G[i * N + j] + dsa[i] * a[j];"),
    "carry_sign": (
        "G[i * N + j] = G[i * N + j] * w[j] + dsa[i] * a[j];",
        "G[i * N + j] = G[i * N + j] * w[j] - dsa[i] * a[j];"),
    "carry_uses_b": (
        "G[i * N + j] = G[i * N + j] * w[j] + dsa[i] * a[j];",
        "G[i * N + j] = G[i * N + j] * w[j] + dsa[i] * b[j];"),
    "dS_init_not_written": (
        "if (dS_init) std::memcpy(dS_init, G.data(), NN * sizeof(F));",
        "if (dS_init) std::memset(dS_init, 0, NN * sizeof(F));"),
    "dS_final_ignored": ("if (dS_final) std::memcpy(G.data(), dS_final, NN * sizeof(F));", ""),
    "dS_final_transposed": (
        "if (dS_final) std::memcpy(G.data(), dS_final, NN * sizeof(F));",
        "if (dS_final) for (int i = 0; i < N; ++i) for (int j = 0; j < N; ++j) G[i * N + j] = dS_final[j * N + i];"),
}

# Cheapest first; the run stops at the first pin that fails.
PIN_TESTS = [
    pins.test_memoryless_closed_form,
    pins.test_pure_accumulation_closed_form,
    pins.test_unrolled_product_brute_force,
    pins.test_homogeneity_identities,
    pins.test_finite_differences_every_coordinate,
    pins.test_structure_causality_linearity_zero_b,
    pins.test_row_permutation_equivariance,
    pins.test_finite_differences_sampled_tiny_workload,
    pins.test_final_state_gradient_euler_identity,
    pins.test_final_state_gradient_finite_differences,
    pins.test_exact_rational_forward_and_gradients,
]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path, gen_mod):
    old, new = MUTANTS[name]
    src = open(oracle._SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    path = tmp_path / "mutant.cpp"
    path.write_text(src.replace(old, new))
    mutant = oracle.Oracle(oracle.compile_library(str(path), str(tmp_path / "libmutant.so")))
    caught = []
    for pin in PIN_TESTS:
        try:
            pin(mutant, gen_mod)
        except AssertionError:
            caught.append(pin.__name__)
            break
    assert caught, f"no pin catches mutant {name}"
