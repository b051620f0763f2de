"""The oracle's pins must catch plausible slips: each mutant below is a copy of
the C oracle with one deliberate mistake, compiled on the CPU, and at least one
pin from test_oracle_pins.py has to fail against it."""
import os
import subprocess

import pytest

import oracle
from tests import test_oracle_pins as pins

MUTANTS = {
    "dropped_normalisation": ("for (int j = 0; j < cp; ++j) w[j] /= s;", ""),
    "exponent_sign": ("exp(L[j] - m)", "exp(m - L[j])"),
    "no_max_shift": ("exp(L[j] - m)", "exp(L[j]) * exp(-m)"),
    "base_swapped": ("lse_base_e ? 1.0 : log(2.0)", "lse_base_e ? log(2.0) : 1.0"),
    "merged_lse_drops_log": ("(m + log(s)) / to_e", "m / to_e"),
    "merged_lse_base_kept_e": ("(m + log(s)) / to_e", "(m + log(s))"),
    "routing_transposed": ("const int h = r * Hl + i;", "const int h = i * cp + r;"),
    "lse_stride_ignored": ("b * lse_row + (int64_t)h * lse_head", "b * H + h"),
    "zero_weight_still_read": ("if (w[j] == 0.0) continue;", ""),
    "empty_row_not_special": ("if (m == -INFINITY) {", "if (0) {"),
    "src_head_stride_ignored": ("(int64_t)h * src_head + d", "(int64_t)h * D + d"),
    "interleave_ignored": ("if ((t / interleave) % cp == j) return 1;", "if (t % cp == j) return 1;"),
    "seq_len_mask_ignored": ("if (seq_lens && !shard_owns_tokens", "if (0 && !shard_owns_tokens"),
    "seq_len_off_by_one": ("for (int64_t t = 0; t < len; ++t) {", "for (int64_t t = 0; t <= len; ++t) {"),
}

# pins that take only the oracle module (and, where parametrised, fixed args)
PIN_CALLS = [
    (pins.test_cp1_is_identity, dict(base_e=True)),
    (pins.test_cp1_is_identity, dict(base_e=False)),
    (pins.test_equal_lse_gives_exact_mean, dict(cp=4, base_e=True)),
    (pins.test_equal_lse_gives_exact_mean, dict(cp=4, base_e=False)),
    (pins.test_hand_worked_dyadic_case, dict(base_e=False)),
    (pins.test_hand_worked_dyadic_case, dict(base_e=True)),
    (pins.test_neg_inf_source_has_zero_weight_even_with_nan_payload, {}),
    (pins.test_row_with_every_source_empty, {}),
    (pins.test_base2_and_base_e_agree, {}),
    (pins.test_shift_invariance, dict(shift=1000.0)),
    (pins.test_nested_merges_are_associative, {}),
    (pins.test_one_hot_head_routing, {}),
    (pins.test_lse_strides_skip_padding, {}),
    (pins.test_padded_source_rows, {}),
    (pins.test_non_contiguous_head_storage, {}),
    (pins.test_merge_of_split_attention_is_full_attention, dict(split="halves", base_e=True)),
    (pins.test_seq_len_mask_gives_attention_over_the_row_context, dict(cp=4, interleave=4, lens=[3, 9, 17])),
    (pins.test_seq_len_mask_gives_attention_over_the_row_context, dict(cp=4, interleave=1, lens=[1, 2, 64])),
    (pins.test_zero_length_context_is_an_empty_row, {}),
]


class _MutantOracle:
    """Same Python surface as the oracle package, bound to a mutant library."""

    def __init__(self, lib):
        self._lib = lib

    def merge(self, *a, **k):
        saved = oracle._lib
        oracle._lib = self._lib
        try:
            return oracle.merge(*a, **k)
        finally:
            oracle._lib = saved

    def half_bits_to_double(self, *a):
        saved = oracle._lib
        oracle._lib = self._lib
        try:
            return oracle.half_bits_to_double(*a)
        finally:
            oracle._lib = saved


def _build_mutant(tmp_path, name, old, new):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "dcp_merge_oracle.c")).read()
    assert src.count(old) >= 1, f"mutant {name}: pattern not found"
    c = tmp_path / f"{name}.c"
    so = tmp_path / f"lib{name}.so"
    c.write_text(src.replace(old, new))
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-shared", "-fPIC", "-o", str(so), str(c), "-lm"],
                   check=True)
    return oracle.open_library(str(so))


def test_unmutated_oracle_passes_every_listed_pin(oracle_mod):
    for fn, kw in PIN_CALLS:
        fn(oracle_mod, **kw)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, oracle_mod, name):
    old, new = MUTANTS[name]
    mutant = _MutantOracle(_build_mutant(tmp_path, name, old, new))
    caught = []
    for fn, kw in PIN_CALLS:
        try:
            with __import__("warnings").catch_warnings():
                __import__("warnings").simplefilter("ignore")
                fn(mutant, **kw)
        except AssertionError:
            caught.append(fn.__name__)
    assert caught, f"no pin caught mutant {name}"
