"""The backward oracle against its pins, and planted mistakes in copies of it
(CPU only; the real oracle source is never modified)."""
from __future__ import annotations

import os

import pytest

import oracle
from tests import pins_backward

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "attn_oracle.c")


@pytest.mark.parametrize("name,pin", pins_backward.ALL_PINS, ids=[p[0] for p in pins_backward.ALL_PINS])
def test_backward_oracle_pin(name, pin):
    pin(oracle)


# (name, original text, replacement): each a plausible slip in writing steps 1-5.
MUTANTS = [
    ("dropped_row_term", "const double ds = p[j] * (dp[j] - r);", "const double ds = p[j] * dp[j];"),
    ("dq_without_scale", "dqi[t] += J->scale * ds * bf16_bits_to_double(kj[t]);",
     "dqi[t] += ds * bf16_bits_to_double(kj[t]);"),
    ("dk_from_k", "dk_acc[j * d + t] += J->scale * ds * qrow[t];",
     "dk_acc[j * d + t] += J->scale * ds * bf16_bits_to_double(kj[t]);"),
    ("dv_from_ds", "dv_acc[j * d + t] += p[j] * grow[t];", "dv_acc[j * d + t] += ds * grow[t];"),
    ("dp_from_k", "acc += grow[t] * bf16_bits_to_double(vp[j * d + t]);",
     "acc += grow[t] * bf16_bits_to_double(kp[j * d + t]);"),
    ("row_term_unweighted", "for (int64_t j = 0; j < N; ++j) r += dp[j] * p[j];",
     "for (int64_t j = 0; j < N; ++j) r += dp[j];"),
    ("backward_p_unnormalised", "for (int64_t j = 0; j < N; ++j) p[j] /= l;", ""),
    ("dk_sign", "dk_acc[j * d + t] += J->scale * ds * qrow[t];", "dk_acc[j * d + t] -= J->scale * ds * qrow[t];"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_backward_mutant_is_caught(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    path = tmp_path / "mut.c"
    path.write_text(src.replace(old, new))
    orc = oracle.Oracle(oracle.compile_source(str(path), str(tmp_path / "libmut.so")))
    caught = []
    for pin_name, pin in pins_backward.ALL_PINS:
        try:
            pin(orc)
        except AssertionError:
            caught.append(pin_name)
    assert caught, f"mutant {name} passed every pin"
