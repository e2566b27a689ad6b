"""Pins for the fp64 CPU oracle (no GPU).

The oracle is the definition of the attention forward written out; these tests
tie it to things other than itself: closed forms, brute force on tiny inputs,
invariants the pages state (two-block online softmax equals one-shot softmax,
rows of P sum to one, P = exp(S - L)), special cases (N = 1, N = 2, Q = 0,
constant V, a fully masked row) and a library restatement (torch fp64
softmax).  test_oracle_mutants.py checks that planted mistakes fail them.
"""
from __future__ import annotations

import math

import numpy as np
import pytest

import oracle
from exact_softmax_attention_fattn_gb300.inputs import (
    WORKLOADS,
    Workload,
    f32_to_bf16_bits,
    make_inputs,
)
from tests import pins


def test_n1_closed_form():
    pins.pin_n1(oracle)


def test_n2_logistic():
    pins.pin_n2_logistic(oracle)


def test_causal_row0_is_v0():
    pins.pin_causal_row0(oracle)


@pytest.mark.parametrize("mode", ["causal", "keylen", "full", "causal_keylen"])
def test_q_zero_prefix_mean_and_log_count(mode):
    pins.pin_q_zero(oracle, mode)


def test_constant_v_returned():
    pins.pin_constant_v(oracle)


def test_linearity_in_v():
    pins.pin_linear_v(oracle)


def test_permutation_invariance():
    pins.pin_permutation(oracle)


def test_lse_bounds():
    pins.pin_lse_bounds(oracle)


def test_rows_sum_to_one_and_p_from_lse():
    pins.pin_probs(oracle)


@pytest.mark.parametrize("causal,use_kl", [(False, False), (True, False), (False, True), (True, True)])
def test_online_blocks_equal_one_shot(causal, use_kl):
    pins.pin_online_recurrence(oracle, causal, use_kl)


@pytest.mark.parametrize("causal,use_kl", [(False, False), (True, False), (False, True), (True, True)])
def test_torch_fp64_cross_check(causal, use_kl):
    pins.pin_torch(oracle, causal, use_kl)


def test_key_blocks_merge_to_the_whole():
    pins.pin_block_merge(oracle)


def test_brute_force_tiny():
    pins.pin_brute(oracle)


def test_fully_masked_rows():
    pins.pin_fully_masked(oracle)


def test_masked_keys_do_not_matter():
    pins.pin_masked_keys_irrelevant(oracle)


def test_key_len_clamped():
    w = Workload("t", 2, 1, 9, 4, False, 11)
    x = make_inputs(w)
    o1, l1 = oracle.forward(x.q, x.k, x.v, 0.5, False, key_len=np.array([99, -3], np.int32))
    o2, l2 = oracle.forward(x.q, x.k, x.v, 0.5, False, key_len=np.array([9, 0], np.int32))
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def test_rows_subset_matches_full():
    w = Workload("t", 2, 3, 37, 16, True, 5)
    x = make_inputs(w)
    o, lse = oracle.forward(x.q, x.k, x.v, w.softmax_scale, True)
    rows = np.array([0, 36, 37, 100, 2 * 3 * 37 - 1], dtype=np.int64)
    os_, ls_ = oracle.forward(x.q, x.k, x.v, w.softmax_scale, True, rows=rows)
    np.testing.assert_array_equal(os_, o.reshape(-1, 16)[rows])
    np.testing.assert_array_equal(ls_, lse.reshape(-1)[rows])


def test_threads_do_not_change_results():
    w = WORKLOADS["b1h1n128d64_causal"]
    x = make_inputs(w)
    a = oracle.forward(x.q, x.k, x.v, w.softmax_scale, True, threads=1)
    b = oracle.forward(x.q, x.k, x.v, w.softmax_scale, True, threads=7)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_bad_arguments_rejected():
    x = make_inputs(Workload("t", 1, 1, 4, 4, False, 0))
    with pytest.raises(RuntimeError):
        oracle.forward(x.q, x.k, x.v, 1.0, False, rows=np.array([4], np.int64))
    with pytest.raises(TypeError):
        oracle.forward(x.q.astype(np.int32), x.k, x.v, 1.0, False)


def test_bf16_rounding_is_nearest_even():
    # 1 + 2^-8 is halfway between two bf16 values: ties go to the even one (1.0);
    # 1 + 3*2^-8 ties up to 1 + 2^-6... (even mantissa), 1 + 2^-8 + 2^-20 rounds up.
    vals = np.array([1.0 + 2.0**-8, 1.0 + 3 * 2.0**-8, 1.0 + 2.0**-8 + 2.0**-20, -2.5], np.float32)
    bits = f32_to_bf16_bits(vals)
    assert bits.tolist() == [0x3F80, 0x3F82, 0x3F81, 0xC020]


def test_config_one_closed_form_checks():
    """Workload b1h1n128d64 (both masks) against the torch restatement."""
    for name in ("b1h1n128d64", "b1h1n128d64_causal"):
        w = WORKLOADS[name]
        x = make_inputs(w)
        o, lse = oracle.forward(x.q, x.k, x.v, w.softmax_scale, w.causal)
        from tests._ref_helpers import torch_reference

        ot, lt = torch_reference(x.q, x.k, x.v, w.softmax_scale, w.causal)
        np.testing.assert_allclose(o, ot, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse, lt, rtol=0, atol=1e-12)
        assert math.isclose(w.softmax_scale, 1 / 8)
