"""Plant plausible mistakes in the oracle (on the CPU) and check the pins catch each one.

Every mutant is a one-line edit of a copy of oracle/spec_oracle.c, compiled into
a temporary library and swapped in for the real one; at least one pin of
test_oracle_pins.py must then fail.
"""

from __future__ import annotations

import os
import tempfile

import pytest

import oracle
from oracle.build import build_oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "spec_oracle.c")

MUTANTS = [
    ("scale dropped", "s[j] = sc * dot;", "s[j] = dot;"),
    ("ancestors invisible", "visible[ncache_cand + p] = 1;", "(void)0;"),
    ("own draft key invisible", "visible[ncache_cand + i] = 1;", "(void)0;"),
    ("GQA head map", "int hk = h / G;", "int hk = h % Hkv;"),
    ("duplicate indices allowed", "t > ib[j - 1]", "t >= ib[j - 1]"),
    ("lse without the max", "double l = mx + log(sum);", "double l = log(sum);"),
    ("window one short", "for (int t = n - w0; t < n; ++t) chosen[t] = 1;",
     "for (int t = n - w0 + 1; t < n; ++t) chosen[t] = 1;"),
    ("ties to the higher index", "return a->index < b->index; /* equal",
     "return a->index > b->index; /* equal"),
    ("NaN ranks first", "if (an) return 0;\n    if (bn) return 1;", "if (an) return 1;\n    if (bn) return 0;"),
    ("full-context shortcut one early", "if (budget >= n) {", "if (budget >= n - 1) {"),
    ("draft K transposed", "krow = k_draft + (((int64_t)b * N + (j - ncache_cand)) * Hkv + hk) * d;",
     "krow = k_draft + (((int64_t)b * Hkv + hk) * N + (j - ncache_cand)) * d;"),
    ("Q transposed", "q + (((int64_t)b * N + i) * Hq + h) * d;", "q + (((int64_t)b * Hq + h) * N + i) * d;"),
    ("merge weight of part b", "double wa = exp(la - l), wb = exp(lb - l);",
     "double wa = exp(la - l), wb = exp(la - l);"),
    ("one extra draft-tier token", "int m = top_m;", "int m = top_m + 1;"),
    ("tier 1 ranks by the target score", "pool[t - rest_lo].score = ds[t];", "pool[t - rest_lo].score = ts[t];"),
    ("cache V read from K", "o[c] += p * cache_value(cl, v_cache, vs, coff[j], c);",
     "o[c] += p * cache_value(cl, k_cache, vs, coff[j], c);"),
    ("probability not normalised", "double p = exp(s[j] - l);", "double p = exp(s[j] - mx);"),
    ("sink one short", "for (int t = 0; t < s0; ++t) chosen[t] = 1;", "for (int t = 1; t < s0; ++t) chosen[t] = 1;"),
    ("paged: row inside the block", "(t % cl->block_size) * cl->st", "((t + 1) % cl->block_size) * cl->st"),
    ("paged: the next block's entry", "cl->table[b * cl->table_ld + t / cl->block_size]",
     "cl->table[b * cl->table_ld + t / cl->block_size + 1]"),
    ("paged: block stride for the head stride", "*off = blk * cl->sb + hk * cl->sh", "*off = blk * cl->sh + hk * cl->sh"),
    ("paged: an entry one past the pool accepted", "blk >= cl->num_blocks", "blk > cl->num_blocks"),
    ("fp8: subnormal exponent", "ldexp((double)m / 8.0, 1 - 7)", "ldexp((double)m / 8.0, 0 - 7)"),
    ("fp8: exponent bias", "ldexp(1.0 + (double)m / 8.0, e - 7)", "ldexp(1.0 + (double)m / 8.0, e - 8)"),
    ("fp8: sign dropped", "return sgn ? -v : v;", "return v;"),
    ("fp8: the V scale on K", "cache_value(cl, k_cache, ks, coff[j], c)", "cache_value(cl, k_cache, vs, coff[j], c)"),
    ("fp8: the next head's scale", "cl->k_scale + (int64_t)b * Hkv + hk", "cl->k_scale + (int64_t)b * Hkv + (hk + 1) % Hkv"),
]

PIN_CALLS = [
    lambda: pins.test_attention_matches_bruteforce(1),
    pins.test_attention_bruteforce_ragged_and_sparse,
    pins.test_closed_form_golden,
    lambda: pins.test_lse_merge_of_parts_equals_monolithic([0, 4, 11]),
    pins.test_oracle_lse_merge_function,
    lambda: pins.test_chain_equals_causal_attention(9),
    pins.test_budget_covering_context_equals_dense,
    pins.test_closed_forms,
    lambda: pins.test_needle(64),
    pins.test_bad_inputs_are_reported,
    pins.test_selection_golden,
    lambda: pins.test_selection_matches_bruteforce(0),
    pins.test_selection_all_equal_scores,
    lambda: pins.test_paged_equals_contiguous(4),
    lambda: pins.test_paged_bad_block_entry("pool_size"),
    pins.test_paged_entries_past_the_context_are_not_read,
    pins.test_e4m3_decoding_table,
    lambda: pins.test_fp8_equals_bf16_on_the_numbers_it_stands_for("dense"),
    pins.test_fp8_v_scale_scales_the_cache_output_only,
]


def _any_pin_fails() -> bool:
    for call in PIN_CALLS:
        try:
            call()
        except (AssertionError, ValueError):
            return True
    return False


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(name, old, new):
    with open(SRC) as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation site not unique or missing: {old!r}"
    with tempfile.TemporaryDirectory() as td:
        msrc = os.path.join(td, "mutant.c")
        with open(msrc, "w") as f:
            f.write(src.replace(old, new))
        lib = oracle.load_library(build_oracle(msrc, os.path.join(td, "libmutant.so")))
        oracle._load()
        prev = oracle.set_library(lib)
        try:
            caught = _any_pin_fails()
        finally:
            oracle.set_library(prev)
    assert caught, f"no pin caught the mutant: {name}"


def test_unmutated_oracle_passes_all_pins():
    assert not _any_pin_fails()
