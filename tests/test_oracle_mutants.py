"""Planted mistakes in copies of the oracle must each fail at least one pin.

Each mutant is a textual edit of attn_oracle.c compiled into a temporary
library (CPU only); the real oracle source is never modified.
"""
from __future__ import annotations

import os

import pytest

import oracle
from tests import pins

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "attn_oracle.c")

# (name, original text, replacement) -- each a plausible slip in writing the definition.
MUTANTS = [
    ("dropped_scale", "s[j] = J->scale * acc;", "s[j] = acc;"),
    ("causal_direction", "int vis = (!J->causal || j <= i) && j < klen;",
     "int vis = (!J->causal || j >= i) && j < klen;"),
    ("key_len_off_by_one", "int vis = (!J->causal || j <= i) && j < klen;",
     "int vis = (!J->causal || j <= i) && j <= klen;"),
    ("exp_sign", "l += exp(s[j] - m);", "l += exp(m - s[j]);"),
    ("lse_log2", "*lse_out = m + log(l);", "*lse_out = m + log2(l);"),
    ("lse_drops_max", "*lse_out = m + log(l);", "*lse_out = log(l);"),
    ("k_for_v", "const uint16_t *vj = vp + j * d;", "const uint16_t *vj = kp + j * d;"),
    ("q_for_k", "const uint16_t *kj = kp + j * d;", "const uint16_t *kj = J->q + (bh * N + j) * d;"),
    ("no_normaliser", "double p = exp(s[j] - m) / l;", "double p = exp(s[j] - m);"),
    ("masked_lse_zero", "*lse_out = -INFINITY;", "*lse_out = 0.0;"),
    ("max_over_all_keys", "        if (!vis) continue;\n        if (!any || s[j] > m) m = s[j];",
     "        if (!any || s[j] > m) m = s[j];\n        if (!vis) continue;"),
    ("prob_matrix_unnormalised", "prow[j] = any ? prow[j] / l : 0.0;", "prow[j] = any ? prow[j] : 0.0;"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new):
    src = open(SRC).read()
    count = src.count(old)
    assert count >= 1, f"mutation anchor for {name} not found"
    mutated = src.replace(old, new)
    path = tmp_path / "mut.c"
    path.write_text(mutated)
    lib = oracle.compile_source(str(path), str(tmp_path / "libmut.so"))
    orc = oracle.Oracle(lib)
    caught = []
    for pin_name, pin in pins.ALL_PINS:
        try:
            pin(orc)
        except AssertionError:
            caught.append(pin_name)
    assert caught, f"mutant {name} passed every pin"


def test_unmutated_copy_passes_every_pin(tmp_path):
    lib = oracle.compile_source(SRC, str(tmp_path / "libcopy.so"))
    orc = oracle.Oracle(lib)
    for _, pin in pins.ALL_PINS:
        pin(orc)
