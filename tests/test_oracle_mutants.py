"""Planted mistakes: each mutant is a copy of the oracle's C source with one plausible
error (a dropped head, a wrong sign, a reversed tiebreak, an off-by-one window, a
transposed index, ...), compiled on the CPU. The pins in test_oracle_pins.py must
reject every one of them; a mutant that passes all pins would mean the pins do not
cover that part of the oracle.
"""
import os
import tempfile

import pytest

from oracle import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "kpool_oracle.c")

MUTANTS = {
    "drop_last_head": ("for (int h = 0; h < heads; ++h)", "for (int h = 0; h < heads - 1; ++h)"),
    "scale_outside_relu": ("double v = (double)scale * dot;\n    if (v < 0.0) v = 0.0;",
                           "double v = dot;\n    if (v < 0.0) v = 0.0;\n    v *= (double)scale;"),
    "relu_flipped": ("if (v < 0.0) v = 0.0;", "if (v > 0.0) v = 0.0;"),
    "weight_of_head0": ("s += (double)w_row[h] * v;", "s += (double)w_row[0] * v;"),
    "q_transposed": ("(int64_t)h * head_dim + c", "(int64_t)c * heads + h"),
    "tiebreak_larger_index": ("if (x->pool < y->pool) return -1;\n  if (x->pool > y->pool) return 1;",
                              "if (x->pool > y->pool) return -1;\n  if (x->pool < y->pool) return 1;"),
    "ascending_scores": ("if (x->score > y->score) return -1;\n  if (x->score < y->score) return 1;",
                         "if (x->score < y->score) return -1;\n  if (x->score > y->score) return 1;"),
    "eligible_one_short": ("const int64_t eligible = (t + 1) / kpool;", "const int64_t eligible = t / kpool;"),
    "eligible_own_incomplete_pool": ("const int64_t eligible = (t + 1) / kpool;",
                                     "const int64_t eligible = (t + kpool) / kpool;"),
    "tail_off_by_one": ("const int64_t tail_len = (t + 1) % kpool;", "const int64_t tail_len = t % kpool;"),
    "global_row_index": ("const int64_t t = row - start;", "const int64_t t = row;"),
    "pool_offset_dropped": ("kp + (size_t)(pool_off[b] + p) * (size_t)head_dim",
                            "kp + (size_t)(p) * (size_t)head_dim"),
    "expand_without_stride": ("(int32_t)((int64_t)ids[j] * kpool + r)", "(int32_t)((int64_t)ids[j] + r)"),
    "sum_not_mean": ("float mean = sum / (float)kpool;", "float mean = sum;"),
    "bf16_truncate": ("if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;", ""),
    "bf16_ties_away": ("(lower == 0x8000u && (upper & 1u))", "(lower == 0x8000u)"),
    "pool_reads_wrong_key": ("(start + p * kpool + j) * head_dim + c", "(start + p * kpool) * head_dim + c"),
    "gated_unnormalised": ("exp((double)gate[(t0 + j) * head_dim + c] - m) / den;",
                           "exp((double)gate[(t0 + j) * head_dim + c] - m);"),
    "gated_ape_per_channel_only": ("(double)ape[(int64_t)j * head_dim + c]", "(double)ape[c]"),
    "gated_ape_dropped": (" + (double)ape[(int64_t)j * head_dim + c])", ")"),
    "gated_gate_of_first_token": ("double wj = exp((double)gate[(t0 + j) * head_dim + c] - m) / den;",
                                  "double wj = exp((double)gate[t0 * head_dim + c] - m) / den;"),
    "budget_one_short": ("const int64_t kept = eligible < budget ? eligible : budget;",
                         "const int64_t kept = eligible < budget ? eligible : budget - 1;"),
}

PIN_CALLS = [
    lambda lib: pins.test_golden_tie_straddles_cutoff("f32", lib=lib),
    lambda lib: pins.test_golden_tie_straddles_cutoff("bf16", lib=lib),
    lambda lib: pins.test_golden_signs_and_scale(lib=lib),
    lambda lib: pins.test_golden_varlen_tail_kpool3(lib=lib),
    lambda lib: pins.test_golden_per_token_kpool1(lib=lib),
    lambda lib: pins.test_golden_bf16_pool_rounding(lib=lib),
    lambda lib: pins.test_brute_force_tiny(lib=lib),
    lambda lib: pins.test_h1_unit_weight_reduces_to_relu_qk(lib=lib),
    lambda lib: pins.test_kpool1_is_per_token_indexer(lib=lib),
    lambda lib: pins.test_pool_mean_closed_form_on_integers(3, lib=lib),
    lambda lib: pins.test_invariants_ragged_packed(31, lib=lib),
    lambda lib: pins.test_short_rows_and_empty_sequences(lib=lib),
    lambda lib: pins.test_packed_equals_alone(lib=lib),
    lambda lib: pins.test_gated_pool_hand_example("f32", lib=lib),
    lambda lib: pins.test_gated_pool_hand_example("bf16", lib=lib),
    lambda lib: pins.test_gated_pool_zero_gate_zero_ape_is_the_mean("bf16", lib=lib),
    lambda lib: pins.test_gated_pool_one_hot_gate_picks_a_position(lib=lib),
]


@pytest.fixture(scope="module")
def workdir():
    with tempfile.TemporaryDirectory(prefix="kpool_mutants_") as d:
        yield d


def test_unmutated_oracle_passes_every_pin(workdir):
    lib = oracle.open_library(oracle.compile_source(SRC, os.path.join(workdir, "orig.so")))
    for call in PIN_CALLS:
        call(lib)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(name, workdir):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique in the oracle source"
    path = os.path.join(workdir, f"{name}.c")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    lib = oracle.open_library(oracle.compile_source(path, os.path.join(workdir, f"{name}.so")))
    caught = []
    for i, call in enumerate(PIN_CALLS):
        try:
            call(lib)
        except (AssertionError, ValueError):
            caught.append(i)
            break
    assert caught, f"no pin rejects the planted mistake {name!r}"
