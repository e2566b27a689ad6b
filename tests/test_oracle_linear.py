"""The causal linear attention oracle against its pins, and planted mistakes
in copies of it (CPU only; the real oracle source is never modified)."""
from __future__ import annotations

import os

import pytest

import oracle
from tests import pins_linear

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "attn_oracle.c")


@pytest.mark.parametrize("name,pin", pins_linear.ALL_PINS, ids=[p[0] for p in pins_linear.ALL_PINS])
def test_linear_oracle_pin(name, pin):
    pin(oracle)


# (name, original text, replacement): plausible slips in writing the method down.
MUTANTS = [
    ("elu_without_plus_one", "return x > 0.0 ? x + 1.0 : exp(x);", "return x > 0.0 ? x : exp(x) - 1.0;"),
    ("relu_feature_map", "return x > 0.0 ? x + 1.0 : exp(x);", "return x > 0.0 ? x : 0.0;"),
    ("mask_ignored", "kt[e] = i < kl ? phi_elu1((double)kh[i * E + e]) : 0.0;",
     "kt[e] = phi_elu1((double)kh[i * E + e]);"),
    ("no_normaliser", "for (int64_t m = 0; m < M; ++m) oh[i * M + m] /= den;", ""),
    ("eps_dropped", "double den = J->eps;", "double den = 0.0;"),
    ("state_after_read",  # row i reads the state before its own key and value are added (j < i)
     "            /* the state takes row i's key and value (a masked key adds nothing) */\n"
     "            for (int64_t e = 0; e < E; ++e) kt[e] = i < kl ? phi_elu1((double)kh[i * E + e]) : 0.0;\n"
     "            for (int64_t e = 0; e < E; ++e) {\n"
     "                s[e] += kt[e];\n"
     "                for (int64_t m = 0; m < M; ++m) S[e * M + m] += kt[e] * (double)vh[i * M + m];\n"
     "            }\n"
     "            /* row i's output from the state */\n"
     "            double den = J->eps;\n"
     "            for (int64_t m = 0; m < M; ++m) oh[i * M + m] = 0.0;\n"
     "            for (int64_t e = 0; e < E; ++e) {\n"
     "                const double qt = phi_elu1((double)qh[i * E + e]);\n"
     "                den += qt * s[e];\n"
     "                for (int64_t m = 0; m < M; ++m) oh[i * M + m] += qt * S[e * M + m];\n"
     "            }\n"
     "            for (int64_t m = 0; m < M; ++m) oh[i * M + m] /= den;\n",
     "            double den = J->eps;\n"
     "            for (int64_t m = 0; m < M; ++m) oh[i * M + m] = 0.0;\n"
     "            for (int64_t e = 0; e < E; ++e) {\n"
     "                const double qt = phi_elu1((double)qh[i * E + e]);\n"
     "                den += qt * s[e];\n"
     "                for (int64_t m = 0; m < M; ++m) oh[i * M + m] += qt * S[e * M + m];\n"
     "            }\n"
     "            for (int64_t m = 0; m < M; ++m) oh[i * M + m] /= den;\n"
     "            for (int64_t e = 0; e < E; ++e) kt[e] = i < kl ? phi_elu1((double)kh[i * E + e]) : 0.0;\n"
     "            for (int64_t e = 0; e < E; ++e) {\n"
     "                s[e] += kt[e];\n"
     "                for (int64_t m = 0; m < M; ++m) S[e * M + m] += kt[e] * (double)vh[i * M + m];\n"
     "            }\n"),
    ("query_unmapped", "const double qt = phi_elu1((double)qh[i * E + e]);", "const double qt = (double)qh[i * E + e];"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_linear_mutant_is_caught(tmp_path, name, old, new):
    with open(SRC) as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    path = tmp_path / "mut.c"
    path.write_text(src.replace(old, new))
    orc = oracle.Oracle(oracle.compile_source(str(path), str(tmp_path / "libmut.so")))
    caught = []
    for pin_name, pin in pins_linear.ALL_PINS:
        try:
            pin(orc)
        except AssertionError:
            caught.append(pin_name)
    assert caught, f"mutant {name} passed every pin"
