"""The split-KV plan (fattn_splitkv_plan, host only, no GPU): a forced split
count is honoured up to one split per key tile; the automatic choice splits
only when the query blocks alone leave SMs idle, and does so on the
low-occupancy shapes."""
from __future__ import annotations

import pytest

from exact_softmax_attention_fattn_gb300 import binding, build


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load_library()


def n_tiles(N):
    return (N + 127) // 128


def units(B, H, N):
    return B * H * ((N + 255) // 256)


@pytest.mark.parametrize("N", [1, 127, 128, 129, 300, 1000, 1024, 4096, 16384])
@pytest.mark.parametrize("req", [1, 2, 3, 5, 8, 16, 1000])
def test_forced_split_count(lib, N, req):
    assert binding.splitkv_plan(2, 3, N, True, 152, req) == min(req, n_tiles(N))


def split_runs(n_blk, splits):
    """Split s of a block with n_blk key tiles takes [s*n_blk/splits, (s+1)*n_blk/splits)."""
    return [(s * n_blk // splits, (s + 1) * n_blk // splits) for s in range(splits)]


@pytest.mark.parametrize("n_blk", [1, 2, 7, 8, 64, 128])
@pytest.mark.parametrize("splits", [1, 2, 3, 5, 16])
def test_split_runs_partition_the_key_tiles(n_blk, splits):
    """The runs the kernel and the combine kernel both use: contiguous, in
    order, covering [0, n_blk) exactly, sizes differing by at most one."""
    runs = split_runs(n_blk, splits)
    assert runs[0][0] == 0 and runs[-1][1] == n_blk
    assert all(a[1] == b[0] for a, b in zip(runs, runs[1:]))
    sizes = [j1 - j0 for j0, j1 in runs]
    assert max(sizes) - min(sizes) <= 1 and min(sizes) >= 0


@pytest.mark.parametrize("B,H,N,causal", [
    (2, 16, 4096, True),     # 512 query blocks
    (1, 32, 16384, True),    # 2048
    (8, 16, 2048, False),    # 1024
    (1, 1, 128, False),      # one key tile: nothing to split
    (1, 1, 128, True),
])
def test_no_split_when_nothing_to_gain(lib, B, H, N, causal):
    assert binding.splitkv_plan(B, H, N, causal, 152, 0) == 1


@pytest.mark.parametrize("B,H,N,causal", [
    (1, 2, 16384, True),     # 128 query blocks, 2 to 128 key tiles each
    (1, 1, 8192, False),     # 32 query blocks, 64 key tiles each
    (1, 2, 4096, True),
])
def test_low_occupancy_shapes_split(lib, B, H, N, causal):
    assert units(B, H, N) < 152
    n = binding.splitkv_plan(B, H, N, causal, 152, 0)
    assert 2 <= n <= 16


def test_short_causal_shape_keeps_one_split(lib):
    """B4 H8 N1024 causal: 128 query blocks of at most 8 key tiles.  Splitting
    would give 256 or more units for 152 CTAs, so each CTA still walks as many
    key-tile steps and pays one more fixed per-unit cost; measured on a GB300
    (2 and 4 forced splits 103 and 82 TFLOP/s against 126 unsplit), and the
    plan agrees."""
    assert units(4, 8, 1024) < 152
    assert binding.splitkv_plan(4, 8, 1024, True, 152, 0) == 1


def test_more_sms_never_fewer_splits(lib):
    """32 query blocks of 64 key tiles: more SMs can only help by splitting more."""
    prev = 1
    for sms in (1, 2, 4, 8, 16, 32, 152):
        n = binding.splitkv_plan(1, 1, 256 * 32, False, sms, 0)
        assert n >= prev
        prev = n
    assert prev >= 4


def test_invalid_arguments(lib):
    assert binding.splitkv_plan(0, 1, 128, False, 152) == 0
    assert binding.splitkv_plan(1, 1, 0, False, 152) == 0
    assert binding.splitkv_plan(1, 1, 128, False, 0) == 0
    assert binding.splitkv_plan(1, 1, 128, False, 152, -1) == 0
