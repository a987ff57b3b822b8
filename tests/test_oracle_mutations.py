"""The pins catch plausible mistakes in the oracle.

Each case compiles a copy of the oracle's C source with one planted mistake
(a flipped sign, a dropped term, a transposed operand, a wrong index, a wrong
head mapping, a skipped emission) into a temporary directory, swaps it in
for the real library, and checks that at least one pin of
test_oracle_pins.py fails on it.  The committed oracle is never modified.
"""
import ctypes
import os
import subprocess

import pytest

import oracle
from oracle import build as obuild
from tests import test_oracle_pins as pins

MUTATIONS = {
    "sign_of_erase_term": ("*sij = alpha * *sij - b * kt[i] * ka[j]", "*sij = alpha * *sij + b * kt[i] * ka[j]"),
    "decay_dropped_in_erase": ("ka[j] += kt[i] * (alpha * s[(size_t)i * d_v + j]);", "ka[j] += kt[i] * s[(size_t)i * d_v + j];"),
    "state_transposed_in_erase": ("ka[j] += kt[i] * (alpha * s[(size_t)i * d_v + j]);", "ka[j] += kt[i] * (alpha * s[(size_t)j * d_v + i]);"),
    "key_used_as_query": ("ot[j] += s[(size_t)i * d_v + j] * qt[i];", "ot[j] += s[(size_t)i * d_v + j] * kt[i];"),
    "value_term_dropped": (" + b * kt[i] * vt[j];", ";"),
    "gva_mapping_modulo": ("const int kh = head / (h_v / h_k);", "const int kh = head % h_k;"),
    "first_emission_skipped": ("(t + 1) % emit_every == 0", "(t + 1) % emit_every == 0 && t + 1 > emit_every"),
    "decay_dropped_on_state": ("*sij = alpha * *sij", "*sij = *sij"),
}

PIN_FUNCS = [
    pins.test_worked_example_by_hand,
    lambda: pins.test_exact_rational_bruteforce(0),
    pins.test_beta_zero_is_pure_decay,
    pins.test_delta_rule_overwrites_along_unit_key,
    pins.test_orthonormal_keys_store_and_retrieve,
    pins.test_update_is_a_gradient_step_on_the_regression_loss,
    pins.test_beta_two_is_a_householder_reflection,
    pins.test_scalar_case_is_a_first_order_linear_filter,
    pins.test_gva_equals_repeated_key_heads,
    pins.test_emitted_states_equal_truncated_runs,
    lambda: pins.test_chunked_form_matches_token_oracle(16),
]


def _build_mutant(tmp_path, name, old, new):
    src = open(obuild.SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    lib = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                    "-o", str(lib), str(path), "-lm"], check=True)
    return str(lib)


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_a_pin_fails_on_planted_mistake(tmp_path, name, monkeypatch):
    old, new = MUTATIONS[name]
    path = _build_mutant(tmp_path, name, old, new)
    real = oracle.load()
    mutant = ctypes.CDLL(path)
    mutant.gdn_oracle_chains.restype = real.gdn_oracle_chains.restype
    mutant.gdn_oracle_chains.argtypes = real.gdn_oracle_chains.argtypes
    monkeypatch.setattr(oracle, "_lib", mutant)
    failed = []
    for f in PIN_FUNCS:
        try:
            f()
        except AssertionError:
            failed.append(getattr(f, "__name__", "lambda"))
    assert failed, f"no pin caught mutation {name}"


def test_real_oracle_passes_every_pin():
    for f in PIN_FUNCS:
        f()
