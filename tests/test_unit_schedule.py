"""The forward's unit schedule (fattn_unit_schedule, host only, no GPU): where
the library replaces the snake order, every round deals exactly the units
the snake deals in that round (so each round keeps the same K/V working
set), the first round is the snake's, and the largest CTA total is below
the snake's.  Unit costs are recomputed here from the causal mask: the key
tiles of 128 that the two query tiles of 128 rows of a unit visit, plus 2."""
from __future__ import annotations

import pytest

from exact_softmax_attention_fattn_gb300 import binding, build


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load_library()


def n_qblocks(N):
    return (N + 255) // 256


def unit_cost(u, BH, N):
    """Causal key tiles of the unit's two 128-row query tiles, plus 2."""
    units = BH * n_qblocks(N)
    if u >= units:
        return 0
    qb = n_qblocks(N) - 1 - u // BH
    cost = 2
    for t in range(2):
        row0 = (2 * qb + t) * 128
        if row0 < N:
            last_row = min(N, row0 + 128)  # rows row0 .. last_row-1 see keys < last_row
            cost += (last_row + 127) // 128
    return cost


def snake(r, c, G):
    return r * G + (G - 1 - c if r % 2 else c)


def totals(table, G, R, BH, N):
    return [sum(unit_cost(table[r * G + c], BH, N) for r in range(R)) for c in range(G)]


SHAPES = [(2, 16, 4096), (1, 40, 4096), (16, 16, 1024), (1, 32, 16384), (8, 16, 2048), (1, 16, 4096),
          (4, 8, 1024), (3, 5, 3000), (1, 1, 128)]


@pytest.mark.parametrize("B,H,N", SHAPES)
def test_schedule_is_a_per_round_permutation_that_lowers_the_maximum(lib, B, H, N):
    BH = B * H
    units = BH * n_qblocks(N)
    G = min(units, 152)
    R = -(-units // G)
    table = binding.unit_schedule(B, H, N, 152)
    snake_table = [snake(r, c, G) for r in range(R) for c in range(G)]
    snake_max = max(totals(snake_table, G, R, BH, N))
    if table is None:
        return  # the library keeps the snake for this shape
    assert len(table) == R * G
    for r in range(R):
        row = table[r * G:(r + 1) * G]
        assert sorted(row) == list(range(r * G, (r + 1) * G)), f"round {r} is not the snake's set of units"
    assert table[:G] == snake_table[:G], "the first round is dealt as the snake deals it"
    assert max(totals(table, G, R, BH, N)) < snake_max


def test_headline_shape_gets_a_table_within_one_step_of_the_mean(lib):
    """B2 H16 N4096: 512 units for 152 CTAs; the snake's largest total is 123
    tile steps against a mean of 117.9; the table brings it to 119."""
    B, H, N = 2, 16, 4096
    table = binding.unit_schedule(B, H, N, 152)
    assert table is not None
    G, R = 152, 4
    t = totals(table, G, R, B * H, N)
    snake_t = totals([snake(r, c, G) for r in range(R) for c in range(G)], G, R, B * H, N)
    assert max(snake_t) == 123 and sum(t) == sum(snake_t) == 17920
    assert max(t) <= 119


def test_single_round_and_bad_arguments_keep_the_snake(lib):
    assert binding.unit_schedule(4, 8, 1024, 152) is None  # 128 units, one round
    assert lib.fattn_unit_schedule(0, 1, 128, 152, None, 0) == 0
    assert lib.fattn_unit_schedule(1, 1, 128, 0, None, 0) == 0


def test_too_small_a_buffer_is_refused(lib):
    import ctypes

    n = lib.fattn_unit_schedule(2, 16, 4096, 152, None, 0)
    assert n == 4 * 152
    buf = (ctypes.c_int * 8)()
    assert lib.fattn_unit_schedule(2, 16, 4096, 152, buf, 8) == -1
    assert list(buf) == [0] * 8


def test_deterministic(lib):
    assert binding.unit_schedule(2, 16, 4096, 152) == binding.unit_schedule(2, 16, 4096, 152)
