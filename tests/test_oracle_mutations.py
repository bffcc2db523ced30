"""The pins of tests/test_oracle_pins.py must catch plausible mistakes in the
oracle.  Each case plants one mistake in a copy of oracle/gdn_oracle.c
(on the CPU), builds it with gcc, routes the oracle through it, and checks
that at least one pin fails."""
import os
import subprocess
import tempfile

import pytest

import oracle
import test_oracle_pins as pins

# (name, original text, planted text); each original occurs exactly once.
MUTATIONS = [
    ("delta rule: correction sign", "decay * (s - beta * p[i] * k[j])", "decay * (s + beta * p[i] * k[j])"),
    ("delta rule: decay on the correction dropped", "decay * (s - beta * p[i] * k[j])", "decay * s - beta * p[i] * k[j]"),
    ("delta rule: write term without beta", "+ beta * v[i] * k[j];", "+ v[i] * k[j];"),
    ("delta rule: output from the old state", "for (int j = 0; j < dk; ++j) acc += S[(size_t)i * dk + j] * q[j];",
     "for (int j = 0; j < dk; ++j) acc += S[(size_t)i * dk + j] * k[j] * 0.0 + S[(size_t)i * dk + j] * q[j] * decay;"),
    ("gates: softplus dropped", "softplus(a_in + dt_bias)", "(a_in + dt_bias)"),
    ("gates: exp(A_log) dropped", "double g = -exp(A_log) * softplus", "double g = -(A_log) * softplus"),
    ("gates: sigmoid sign", "*beta = sigmoid(b_in);", "*beta = sigmoid(-b_in);"),
    ("norm: q scale not applied", "oracle_l2norm(dk, q, d->eps_l2, d->q_scale);", "oracle_l2norm(dk, q, d->eps_l2, 1.0);"),
    ("norm: epsilon dropped", "double inv = 1.0 / sqrt(ss + eps);", "double inv = 1.0 / sqrt(ss);"),
    ("rmsnorm: sum instead of mean", "sqrt(ss / dv + eps)", "sqrt(ss + eps)"),
    ("silu: sigmoid only", "static double silu(double x) { return x * sigmoid(x); }",
     "static double silu(double x) { return sigmoid(x); }"),
    ("conv: taps reversed", "bf16_value(conv_w[(size_t)c * 4 + j])", "bf16_value(conv_w[(size_t)c * 4 + 3 - j])"),
    ("conv: tail read newest-last", "int tail_next = 2;", "int tail_next = 0;"),
    ("heads: key head h % Hk", "const int kh = h / G;", "const int kh = h % Hk;"),
    ("record: tail shifted by one", "memcpy(rec_tail + ((size_t)t * 3 + m) * CH, hist[m + 1], sizeof(uint16_t) * CH);",
     "memcpy(rec_tail + ((size_t)t * 3 + m) * CH, hist[m], sizeof(uint16_t) * CH);"),
    ("tree: parents ignored", "if (node >= 0) node = parent ? parent[node] : node - 1;", "if (node >= 0) node = node - 1;"),
    ("rmsnorm: z read at the key head", "zz[i] = bf16_value(z[((size_t)t * Hv + h) * dv + i]);",
     "zz[i] = bf16_value(z[((size_t)t * Hv + kh) * dv + i]);"),
    ("rmsnorm: w_norm reversed", "wn[i] = bf16_value(norm_w[i]);", "wn[i] = bf16_value(norm_w[dv - 1 - i]);"),
    ("chunked: Gamma exponent sign", "double m = bc[t] * exp(Gc[t] - Gc[s]) * A[t * C + s];",
     "double m = bc[t] * exp(Gc[s] - Gc[t]) * A[t * C + s];"),
    ("chunked: state term of U dropped", "U[(size_t)t * dv + i] -= acc;", "U[(size_t)t * dv + i] -= 0.0 * acc;"),
    ("chunked: diagonal of P dropped", "for (int s = 0; s <= t; ++s) {", "for (int s = 0; s < t; ++s) {"),
]

PINS = [
    pins.test_delta_rule_hand_worked_golden,
    lambda: pins.test_delta_rule_brute_force_matrices(3, 5),
    pins.test_delta_rule_single_rank1_closed_form,
    pins.test_delta_rule_write_invariant,
    pins.test_delta_rule_identity_case,
    pins.test_gates_hand_worked_golden,
    pins.test_gates_against_library_routines,
    pins.test_l2norm_unit_length_and_direction,
    pins.test_gated_rmsnorm_special_cases,
    pins.test_conv_current_tap_reduces_to_silu_and_library_norm,
    lambda: pins.test_conv_past_taps_follow_the_tail(0),
    lambda: pins.test_conv_past_taps_follow_the_tail(2),
    pins.test_grouped_head_mapping,
    pins.test_layer_output_is_gated_rmsnorm_of_its_own_head,
    pins.test_layer_recurrence_matches_explicit_matrix_chain,
    pins.test_tree_node_equals_chain_along_its_path,
    lambda: pins.test_chunked_form_equals_sequential_recurrence(37, 4),
    lambda: pins.test_chunked_form_equals_sequential_recurrence(130, 64),
]


def _build_mutant(original: str, planted: str, workdir: str) -> str:
    with open(oracle.source_path()) as f:
        src = f.read()
    assert src.count(original) == 1, f"mutation anchor not unique: {original!r}"
    path_c = os.path.join(workdir, "mutant.c")
    path_so = os.path.join(workdir, "libmutant.so")
    with open(path_c, "w") as f:
        f.write(src.replace(original, planted))
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", path_so, path_c, "-lm"])
    return path_so


@pytest.mark.parametrize("name,original,planted", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_mistake(name, original, planted):
    with tempfile.TemporaryDirectory() as d:
        lib = _build_mutant(original, planted, d)
        failed = []
        with oracle.using_library(lib):
            for pin in PINS:
                try:
                    pin()
                except (AssertionError, ValueError):
                    failed.append(getattr(pin, "__name__", "pin"))
        assert failed, f"no pin caught the planted mistake: {name}"


def test_unmutated_oracle_passes_every_pin():
    for pin in PINS:
        pin()
