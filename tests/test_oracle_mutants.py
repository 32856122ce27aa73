"""Mutation check of the oracle's pins.

Each case plants one plausible mistake in a private copy of the oracle source (a dropped
term, a wrong sign, index or operand order), builds it on the CPU and checks that at least
one pin of ``test_oracle_pins`` fails against it.  The product code is never touched.
"""
import os
import tempfile

import pytest

import oracle
import test_oracle_pins as pins

MUTANTS = {
    "delta drops the decay": (
        "p[cc] = b * (vt[cc] - alpha * p[cc]);", "p[cc] = b * (vt[cc] - p[cc]);"),
    "decay applied after the write": (
        "hrow[cc] = alpha * hrow[cc] + ki * p[cc];", "hrow[cc] = alpha * (hrow[cc] + ki * p[cc]);"),
    "tiled GQA order in the token form": (
        "const int kh = j / (hv / hk);\n    const int c0", "const int kh = j % hk;\n    const int c0"),
    "exclusive cumulative decay": (
        "acc += gc[t];\n        G[t] = acc;", "G[t] = acc;\n        acc += gc[t];"),
    "A keeps the diagonal": (
        "for (int j = 0; j < t; ++j) {\n            double dot",
        "for (int j = 0; j <= t; ++j) {\n            double dot"),
    "forward substitution sign": (
        "Tm[(size_t)t * L + c] -= a * Tm", "Tm[(size_t)t * L + c] += a * Tm"),
    "w without exp(G)": ("bc[j] * exp(G[j]) * kc", "bc[j] * kc"),
    "k_tilde decay inverted": ("exp(GL - G[j]) * kc", "exp(G[j] - GL) * kc"),
    "attn_i strictly lower": ("if (j <= t) {", "if (j < t) {"),
    "transposed k_tilde^T w": (
        "s->kt[(size_t)t * K + a] * s->w[(size_t)t * K + b]",
        "s->kt[(size_t)t * K + b] * s->w[(size_t)t * K + a]"),
    "M composition drops gamma": (
        "M[(size_t)a * K + b] = s.gamma * M[(size_t)a * K + b] - x;",
        "M[(size_t)a * K + b] = M[(size_t)a * K + b] - x;"),
    "scan drops U": ("double x = Ur[(size_t)a * V + c];", "double x = 0.0;"),
    "uneven split puts the extra chunks last": (
        "*c0 = r * base + (r < extra ? r : extra);\n    *c1 = *c0 + base + (r < extra ? 1 : 0);",
        "*c0 = r * base + (r > P - 1 - extra ? r - (P - extra) : 0);\n"
        "    *c1 = *c0 + base + (r >= P - extra ? 1 : 0);"),
}


def _run_all_pins():
    """Returns the names of the pins that fail."""
    failed = []
    cases = [
        ("exact", pins.test_exact_rational_brute_force, ()),
        ("hand", pins.test_hand_worked_2x2, ()),
        ("gqa", pins.test_gqa_grouped_order, ()),
        ("beta0", pins.test_beta_zero_is_pure_decay, ()),
        ("ortho", pins.test_orthonormal_keys_is_decayed_linear_attention, ()),
        ("overwrite", pins.test_overwrite_with_repeated_orthonormal_keys, ()),
        ("padding", pins.test_padding_is_a_no_op, ()),
        ("segments", pins.test_segment_count_invariance_and_empty_segments, ()),
        ("factors", pins.test_chunk_factors_against_linear_solve, ()),
        ("lowrank", pins.test_low_rank_summary_equals_dense_transition, ()),
        ("scan", pins.test_scan_is_exclusive_and_ordered, ()),
        ("stages", pins.test_prepare_and_emit_stages_compose, ()),
        ("brute", pins.test_forms_match_dense_brute_force, (1, [13, 27], 8)),
    ]
    for name, fn, args in cases:
        try:
            fn(*args)
        except (AssertionError, ValueError, FloatingPointError):
            failed.append(name)
    return failed


def test_unmutated_oracle_passes_every_pin():
    assert _run_all_pins() == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    before, after = MUTANTS[name]
    src = open(oracle._SRC).read()
    assert src.count(before) >= 1, f"mutation site for '{name}' not found"
    mutated = src.replace(before, after, 1)
    path = tmp_path / "mutant.c"
    path.write_text(mutated)
    lib = oracle.build(force=True, src=str(path), out=str(tmp_path / "libmutant.so"))
    with oracle.use_library(lib):
        failed = _run_all_pins()
    assert failed, f"no pin catches the mutant '{name}'"
