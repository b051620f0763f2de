"""The attention oracle's pins must catch plausible slips too: each mutant is
a copy of oracle/attention.py with one deliberate mistake, loaded in place of
the real module, and at least one pin from test_oracle_pins.py has to fail
against it (an assertion, or an error such as a shape mismatch)."""
import os
import types

import pytest

import oracle.attention
from tests import test_oracle_pins as pins

MUTANTS = {
    "scale_dropped": ("s = scale * np.einsum", "s = np.einsum"),
    "keys_without_rope": ('np.einsum("rhd,td->rht", q, kv)', 'np.einsum("rhd,td->rht", q[..., :dv], kv[:, :dv])'),
    "max_not_added_back": ("lse = m[..., 0] + np.log(z)", "lse = np.log(z)"),
    "normalisation_dropped": ("p / z[..., None]", "p"),
    "base2_conversion_inverted": ("lse = lse / np.log(2.0)", "lse = lse * np.log(2.0)"),
    "natural_log_for_base2_skipped": ("if not base_e:", "if False:"),
    "values_include_rope": ("kv[:, :dv])", "kv[:, :dv] * 0 + kv[:, -dv:])"),
    "empty_set_lse_zero": ("np.full((R, H), -np.inf)", "np.zeros((R, H))"),
    "min_instead_of_max": ("m = s.max(axis=-1, keepdims=True)", "m = s.min(axis=-1, keepdims=True)"),
}

PIN_CALLS = [
    (pins.test_attention_over_one_token_is_that_value, {}),
    (pins.test_attention_with_zero_query_is_the_value_mean, {}),
    (pins.test_attention_two_tokens_closed_form, {}),
    (pins.test_attention_is_invariant_under_token_permutation, {}),
    (pins.test_attention_is_stable_for_widely_spread_scores, {}),
    (pins.test_merge_of_split_attention_is_full_attention, dict(split="halves", base_e=True)),
    (pins.test_merge_of_split_attention_is_full_attention, dict(split="halves", base_e=False)),
    (pins.test_empty_shard_in_split_attention, {}),
]


def _mutant_module(name, old, new):
    src = open(os.path.join(os.path.dirname(oracle.attention.__file__), "attention.py")).read()
    assert src.count(old) == 1, f"mutant {name}: pattern not found once"
    mod = types.ModuleType(f"attention_mutant_{name}")
    exec(compile(src.replace(old, new), f"<mutant {name}>", "exec"), mod.__dict__)
    return mod


def _run_pins(oracle_mod):
    failed = []
    for fn, kw in PIN_CALLS:
        args = (oracle_mod,) if "oracle_mod" in fn.__code__.co_varnames[:fn.__code__.co_argcount] else ()
        try:
            fn(*args, **kw)
        except (AssertionError, ValueError, IndexError, FloatingPointError):
            failed.append(fn.__name__)
    return failed


def test_unmutated_attention_oracle_passes_every_listed_pin(oracle_mod):
    assert _run_pins(oracle_mod) == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_attention_mutant_is_caught(oracle_mod, monkeypatch, name):
    mod = _mutant_module(name, *MUTANTS[name])
    monkeypatch.setattr(oracle.attention, "attention", mod.attention)
    monkeypatch.setattr(oracle.attention, "split_partials", mod.split_partials)
    with __import__("warnings").catch_warnings():
        __import__("warnings").simplefilter("ignore")
        caught = _run_pins(oracle_mod)
    assert caught, f"no pin caught mutant {name}"
