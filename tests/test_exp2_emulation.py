"""The kernel's FMA-pipe 2^x (round-to-integer split, fitted cubic, exponent
add), replayed step by step in numpy float32 with the constants read from the
kernel source, against exp2 in float64 (no GPU)."""
from __future__ import annotations

import os
import re

import numpy as np

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "exact_softmax_attention_fattn_gb300", "csrc", "fattn_kernel.cuh")


def constants():
    text = open(SRC).read()
    get = lambda n: np.float32(float(re.search(rf"{n} = ([0-9.e+-]+)f;", text).group(1)))
    return [get(f"EXP2_C{i}") for i in range(4)], get("ROUND_MAGIC")


def emulate(x: np.ndarray) -> np.ndarray:
    (c0, c1, c2, c3), magic = constants()
    x = np.maximum(x.astype(np.float32), np.float32(-126.0))
    t = (x + magic).astype(np.float32)
    r = (t - magic).astype(np.float32)
    f = (x - r).astype(np.float32)
    q = ((c3 * f + c2) * f + c1).astype(np.float32) * f + c0
    q = q.astype(np.float32)
    bits = (q.view(np.int32).astype(np.int64) + (t.view(np.int32).astype(np.int64) << 23)) & 0xFFFFFFFF
    return bits.astype(np.uint32).view(np.float32)


def test_split_is_exact_round_to_nearest():
    _, magic = constants()
    x = np.linspace(-126, 16, 100001, dtype=np.float32)
    t = (x + magic).astype(np.float32)
    r = (t - magic).astype(np.float32)
    assert np.all(np.abs(x - r) <= 0.5)
    assert np.all(r == np.round(r))


def test_relative_error_over_the_used_range():
    x = np.concatenate([np.linspace(-126, 16, 400001), np.linspace(-1, 1, 100001)]).astype(np.float32)
    y = emulate(x).astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    normal = x > -125.5  # below this the result is denormal or flushed: checked separately
    rel = np.abs(y[normal] / ref[normal] - 1.0)
    assert rel.max() < 1.0e-4, rel.max()


def test_tiny_and_masked_inputs_give_zero_or_tiny_nonnegative():
    x = np.array([-np.inf, -1e30, -500.0, -127.0, -126.0], dtype=np.float32)
    y = emulate(x)
    assert np.all(y >= 0.0) and np.all(y < 2.0 ** -125) and np.all(np.isfinite(y))
