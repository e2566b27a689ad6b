"""The GPU comparison harness on the CPU: the exact result rounded to bf16
always passes, and an error past the bar always fails."""
from __future__ import annotations

import numpy as np
import pytest

from exact_softmax_attention_fattn_gb300.inputs import bf16_bits_to_f32, f32_to_bf16_bits
from tests.gpu_helpers import bf16_ulp, compare


def rounded(x):
    return bf16_bits_to_f32(f32_to_bf16_bits(x.astype(np.float32))).astype(np.float64)


def test_bf16_ulp_values():
    np.testing.assert_array_equal(bf16_ulp(np.array([1.0, 1.5, 2.0, 3.99, 4.0, -5.0, 0.25])),
                                  [2.0**-7, 2.0**-7, 2.0**-6, 2.0**-6, 2.0**-5, 2.0**-5, 2.0**-9])


def test_correctly_rounded_output_passes():
    rng = np.random.default_rng(0)
    o = rng.normal(size=(64, 128)) * 0.5
    o[0, :8] = [4.01, 4.49, -4.7, 5.9, 7.99, -7.5, 3.999, 6.2]
    lse = rng.normal(size=64)
    compare(rounded(o), lse.astype(np.float32).astype(np.float64), o, lse, log=False)


def test_error_past_bar_fails():
    o = np.full((4, 8), 1.0)
    bad = o.copy()
    bad[1, 3] += 0.011
    with pytest.raises(AssertionError):
        compare(bad, np.zeros(4), o, np.zeros(4), log=False)
    big = np.full((4, 8), 4.3)
    bad = big.copy()
    bad[0, 0] += 1e-2 + 2.0**-6 + 1e-4  # past 1e-2 + half an ulp (2^-5 in [4, 8))
    with pytest.raises(AssertionError):
        compare(bad, np.zeros(4), big, np.zeros(4), log=False)
    # a full ulp used to pass at |O| >= 4; it no longer does
    bad = big.copy()
    bad[2, 5] += 2.0**-5
    with pytest.raises(AssertionError):
        compare(bad, np.zeros(4), big, np.zeros(4), log=False)
    # below 4 the bar is the stated 1e-2, with no ulp allowance
    mid = np.full((4, 8), 3.9)
    bad = mid.copy()
    bad[3, 1] += 0.0101
    with pytest.raises(AssertionError):
        compare(bad, np.zeros(4), mid, np.zeros(4), log=False)


def test_wider_bar_is_counted():
    """Elements past 1e-2 (only allowed at |O| >= 4, within 1e-2 + half an
    ulp) are counted and reported in ulps."""
    big = np.full((2, 64), 4.3)
    got = big.copy()
    got[0, 0] += 0.02   # within 0.0256; the mean stays under 1e-3
    got[1, 3] -= 0.015
    st = compare(got, np.zeros(2), big, np.zeros(2), "wide", log=False)
    assert st.n_over_1e2 == 2
    assert abs(st.worst_over_ulps - 0.02 / 2.0**-5) < 1e-9
    st = compare(big, np.zeros(2), big, np.zeros(2), "exact", log=False)
    assert st.n_over_1e2 == 0 and st.worst_over_ulps == 0.0


def test_mean_and_lse_bars():
    o = np.zeros((100, 8))
    with pytest.raises(AssertionError):
        compare(o + 0.002, np.zeros(100), o, np.zeros(100), log=False)
    with pytest.raises(AssertionError):
        compare(o, np.full(100, 0.0011), o, np.zeros(100), log=False)


def test_masked_row_pattern_must_match():
    o = np.zeros((2, 8))
    with pytest.raises(AssertionError):
        compare(o, np.array([-np.inf, 0.0]), o, np.array([0.0, 0.0]), log=False)
    compare(o, np.array([-np.inf, 0.0]), o, np.array([-np.inf, 0.0]), log=False)
