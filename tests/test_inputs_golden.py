"""The seeded generator and the stored golden values (no GPU)."""
from __future__ import annotations

import hashlib
import json
import os

import numpy as np
import pytest

import oracle
from exact_softmax_attention_fattn_gb300.inputs import (
    WORKLOADS,
    _GOLDEN,
    _mix64,
    bf16_bits_to_f32,
    causal_flops,
    make_inputs,
    normal,
)

GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_splitmix64_published_vector():
    # SplitMix64 with state 1234567: the first five outputs of the reference
    # generator (Steele, Lea, Flood 2014; the java.util.SplittableRandom mix).
    with np.errstate(over="ignore"):
        idx = np.arange(1, 6, dtype=np.uint64)
        got = _mix64(np.uint64(1234567) + idx * _GOLDEN)
    assert [int(x) for x in got] == [
        6457827717110365317, 3203168211198807973, 9817491932198370423,
        4593380528125082431, 16408922859458223821,
    ]


def test_normal_moments():
    z = normal(7, 1, 400_001, sigma=2.0).astype(np.float64)
    assert abs(z.mean()) < 0.02
    assert abs(z.std() - 2.0) < 0.02
    assert z.dtype == np.float64 and np.all(np.isfinite(z))


def test_chunking_does_not_change_draws():
    a = normal(3, 2, 1000)
    b = normal(3, 2, 1001)[:1000]
    np.testing.assert_array_equal(a, b)


def test_key_len_range_and_determinism():
    w = WORKLOADS["b8h16n2048d128_keylen"].replace(N=64, H=1, d=8, key_len_range=(32, 64))
    x1, x2 = make_inputs(w), make_inputs(w)
    assert x1.key_len.dtype == np.int32 and x1.key_len.shape == (8,)
    assert np.all((x1.key_len >= 32) & (x1.key_len <= 64))
    np.testing.assert_array_equal(x1.key_len, x2.key_len)
    np.testing.assert_array_equal(x1.q, x2.q)


def test_keylen_workload_draws():
    w = WORKLOADS["b8h16n2048d128_keylen"]
    kl = make_inputs(w.replace(H=1, N=2048, d=8)).key_len
    assert np.all((kl >= 1024) & (kl <= 2048))


def test_flop_counts():
    w = WORKLOADS["b2h16n4096d128_causal"]
    assert causal_flops(w) == pytest.approx(137.438953472e9)
    w5 = WORKLOADS["b8h16n2048d128_keylen"]
    kl = np.full(8, 1024, np.int32)
    assert causal_flops(w5, kl) == pytest.approx(4 * 16 * 2048 * 128 * 1024 * 8)


@pytest.mark.parametrize("name", ["b1h1n128d64", "b1h1n128d64_causal"])
def test_golden(name):
    with open(os.path.join(GOLDEN_DIR, f"{name}.json")) as f:
        g = json.load(f)
    w = WORKLOADS[name]
    x = make_inputs(w)
    assert hashlib.sha256(x.q.tobytes()).hexdigest() == g["sha256_q_bits"]
    assert hashlib.sha256(x.k.tobytes()).hexdigest() == g["sha256_k_bits"]
    assert hashlib.sha256(x.v.tobytes()).hexdigest() == g["sha256_v_bits"]
    o, lse = oracle.forward(x.q, x.k, x.v, g["scale"], g["causal"])
    exp_lse = np.array([float.fromhex(t) for t in g["lse"]])
    np.testing.assert_allclose(lse[0, 0], exp_lse, rtol=0, atol=1e-12)
    for r, row in zip(g["rows"], g["o_rows"]):
        np.testing.assert_allclose(o[0, 0, r], [float.fromhex(t) for t in row], rtol=0, atol=1e-12)
    # values are bf16-exact in fp32
    assert np.all(bf16_bits_to_f32(x.q).view(np.uint32) & 0xFFFF == 0)


def test_linear_workload_recipe():
    """The linear-attention workloads: fp32 N(0, 1) Q, K, V of the stated
    shapes from their own seeds, key lengths in range, deterministic, and the
    FLOP count the bench reports (the recurrence's 4 E M + 4 E per row)."""
    from exact_softmax_attention_fattn_gb300.inputs import LINEAR_WORKLOADS, linear_flops, make_linear_inputs

    w = LINEAR_WORKLOADS["lin_b2h16n4096e64"]
    assert (w.B, w.H, w.N, w.E, w.M, w.seed, w.key_len_range) == (2, 16, 4096, 64, 64, 8, None)
    assert linear_flops(w) == 2 * 16 * 4096 * (4 * 64 * 64 + 4 * 64) == 2181038080
    wk = LINEAR_WORKLOADS["lin_b8h8n2048e64_keylen"]
    assert (wk.B, wk.H, wk.N, wk.E, wk.M, wk.seed, wk.key_len_range) == (8, 8, 2048, 64, 64, 9, (1024, 2048))
    small = wk.__class__("t", 8, 2, 64, 8, 4, 9, key_len_range=(1024, 2048))
    x1, x2 = make_linear_inputs(small), make_linear_inputs(small)
    assert x1.q.dtype == np.float32 and x1.q.shape == (8, 2, 64, 8) and x1.v.shape == (8, 2, 64, 4)
    np.testing.assert_array_equal(x1.q, x2.q)
    np.testing.assert_array_equal(x1.v, x2.v)
    assert x1.key_len.dtype == np.int32 and np.all((x1.key_len >= 1024) & (x1.key_len <= 2048))
    np.testing.assert_array_equal(x1.key_len, x2.key_len)
    big = make_linear_inputs(w.__class__("m", 1, 1, 4096, 64, 64, 8))
    z = big.q.astype(np.float64)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1.0) < 0.01
    assert not np.array_equal(big.q, big.k)  # Q and K from separate streams
