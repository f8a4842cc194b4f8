"""The oracle pins must catch plausible mistakes.

Each case copies the oracle source, plants one mistake (a dropped term, a
wrong sign, index or anchor, a transposed layout), compiles the copy on the
CPU and checks that the pins of test_oracle_pins reject it.
"""

import os
import subprocess
import tempfile

import numpy as np
import pytest

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTANTS = {
    "ds_without_rowsum_term": ("pij * (z * dP - Di)", "pij * (z * dP)"),
    "dk_without_scale": ("dkj[d] += p->scale * dS * qi[d]", "dkj[d] += dS * qi[d]"),
    "dv_without_dropout": ("*pz_out = pij * z;", "*pz_out = pij;"),
    "causal_top_left_anchor": ("case 3: return j <= i + (skv - sq);", "case 3: return j <= i;"),
    "bit_index_row_major_heads": ("int64_t index = base + (h * sq + i) * skv + j;",
                                  "int64_t index = base + (i * p->Nq + h) * skv + j;"),
    "sink_missing_from_sum": ("if (p->sink) l += exp(p->sink[h] - m);", ""),
    "dsink_wrong_sign": ("dsink[h] -= exp(p->sink[h] - smax[r])", "dsink[h] += exp(p->sink[h] - smax[r])"),
    "gqa_interleaved_heads": ("const int64_t G = p->Nq / p->Nkv, g = h / G, D = p->D;",
                              "const int64_t G = p->Nq / p->Nkv, g = h % p->Nkv, D = p->D;"),
    "band_exclusive_edge": ("(j - i >= -pre) && (j - i <= next)", "(j - i > -pre) && (j - i <= next)"),
    "atten_mask_transposed": ("p->atten_mask[i * p->mask_cols + j]", "p->atten_mask[j * p->mask_cols + i]"),
    "atten_mask_mode0_without_band": (
        "return !masked && (j - i >= -p->pre_tokens) && (j - i <= p->next_tokens);", "return !masked;"),
    "prefix_inclusive": ("j < p->prefix[b]", "j <= p->prefix[b]"),
    "prefix_top_left_anchor": ("case 6: return j <= i + (skv - sq)", "case 6: return j <= i"),
    "pse_rows_above_not_along_diagonal": ("        c = j - r;\n        r = 0;", "        r = 0;"),
    "pse_type_swapped": ("return p->pse_type == 1 ? p->scale * (qk + pse)", "return p->pse_type == 0 ? p->scale * (qk + pse)"),
    "generated_alibi_sign": ("return -slope * (p->pse_type == 2 ? dist : sqrt(dist));",
                             "return slope * (p->pse_type == 2 ? dist : sqrt(dist));"),
    "generated_alibi_without_sqrt": ("return -slope * (p->pse_type == 2 ? dist : sqrt(dist));",
                                     "return -slope * dist;"),
    "generated_pse_before_scale": ("return p->pse_type == 1 ? p->scale * (qk + pse)",
                                   "return p->pse_type != 0 ? p->scale * (qk + pse)"),
    "dp_drops_last_value_column": ("const double dP = dot(dy + r * Dv, vj, Dv);", "const double dP = dot(dy + r * Dv, vj, Dv - 1);"),
    "drow_drops_last_value_column": ("Drow[r] = dot(dy + r * Dv, out + r * Dv, Dv);", "Drow[r] = dot(dy + r * Dv, out + r * Dv, Dv - 1);"),
}


def _pin_suite(ora):
    """Run the pins that exercise every term; True if all pass."""
    try:
        for ci in range(len(pins.CASES)):
            pins.test_forward_and_grad_match_autograd(ora, ci)
        for mode, pre, nxt in [(3, pins.INF, pins.INF), (4, 3, 0), (4, 2, 3)]:
            for sq, skv in [(5, 9), (7, 7)]:
                pins.test_mask_predicate_matches_explicit_matrix(ora, mode, pre, nxt, sq, skv)
        pins.test_dropout_bit_layout_bruteforce(ora)
        pins.test_ds_row_sums(ora, True)
        pins.test_gqa_equals_repeated_mha(ora)
        for mode, pre, nxt in [(1, pins.INF, pins.INF), (0, 3, 1)]:
            pins.test_atten_mask_predicate_matches_explicit_matrix(ora, mode, pre, nxt, 5, 9)
        pins.test_prefix_predicate_matches_explicit_matrix(ora, 5, 9)
        for ci in range(len(pins.MASK_CASES)):
            pins.test_masked_forward_and_grad_match_autograd(ora, ci)
        for pse_type in (0, 1):
            pins.test_alibi_pse_matches_autograd_with_the_full_bias(ora, pse_type, [1300, 40])
            pins.test_random_pse_short_sequences_match_autograd(ora, pse_type)
        for ci in range(len(pins.DV_CASES)):
            pins.test_unequal_head_dims_match_autograd(ora, ci)
        pins.test_generated_alibi_causal_equals_a_column_bias_in_one_more_dim(ora)
        for pse_type in (2, 3):
            pins.test_generated_alibi_matches_autograd(ora, pse_type, True)
    except AssertionError:
        return False
    return True


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_planted_mistake(name):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) >= 1, name
    with tempfile.TemporaryDirectory() as tmp:
        src = os.path.join(tmp, "mutant.c")
        so = os.path.join(tmp, "libmutant.so")
        open(src, "w").write(text.replace(old, new))
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", src, "-o", so, "-lm"])
        oracle.build()
        prev = oracle.use_library(oracle.bind(so))
        try:
            assert not _pin_suite(oracle), f"pins accepted the planted mistake {name}"
        finally:
            oracle.use_library(prev)


def test_unmutated_source_passes_suite():
    oracle.build()
    oracle.use_library(None)
    assert _pin_suite(oracle)
