"""Planted mistakes in the oracle must each trip at least one pin (CPU).

Every mutant is a textual edit of ``oracle/gqa_oracle.c`` compiled into a
temporary library; the real oracle source is never modified.  All edits keep
memory accesses in bounds.
"""
import os

import pytest

import oracle
from tests import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "gqa_oracle.c")

MUTANTS = {
    "kv_head_modulo": ("h / group", "h % hkv"),
    "scale_one_over_d": ("1.0 / sqrt((double)d)", "1.0 / (double)d"),
    "no_scale": ("w[j] = dot * scale;", "w[j] = dot;"),
    "causal_excludes_self": ("causal ? i + 1 : S", "causal ? (i > 0 ? i : 1) : S"),
    "causal_sees_one_more": ("causal ? i + 1 : S", "causal ? (i + 2 < S ? i + 2 : S) : S"),
    "no_max_subtraction": ("w[j] = exp(w[j] - m);", "w[j] = exp(w[j]);"),
    "exp2_for_exp": ("w[j] = exp(w[j] - m);", "w[j] = exp2(w[j] - m);"),
    "unnormalised": ("w[j] /= l;", "w[j] /= 1.0;"),
    "dropped_last_feature": ("for (int c = 0; c < d; ++c)\n            dot +=",
                             "for (int c = 0; c < d - 1; ++c)\n            dot +="),
    "k_used_as_v": ("const uint16_t *vrow = v +", "const uint16_t *vrow = k +"),
    "sign_flip": ("dot += bf16_bits_to_double(qrow[c])", "dot -= bf16_bits_to_double(qrow[c])"),
    "q_row_zero": ("q + ((size_t)i * hq + h) * d", "q + ((size_t)0 * hq + h) * d"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert old in text, f"mutation site for {name} not found"
    src = tmp_path / "mutant.c"
    src.write_text(text.replace(old, new))
    lib = oracle.OracleLib(oracle.compile_source(str(src), str(tmp_path / "libmutant.so")))
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(lib)
        except (AssertionError, ValueError, FloatingPointError):
            caught.append(pin.__name__)
    assert caught, f"planted mistake {name} passed every pin"
