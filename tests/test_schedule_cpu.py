"""The main pass's work decomposition, checked on the host (no GPU).

dora_selftest_schedule plans a bf16 single-module norm exactly as
dora_factored_norm does and enumerates every piece of work the launched CTA
pairs would run, through the same functions the kernel uses: K segments
handed out in item order, static ranges (one contiguous run of
(pair tile, K tile) iterations per pair, issued from the last piece to the
first), or a piece table (one K range of one pair tile per pair, with fewer
pair tiles than pairs).  A sound plan covers every pair tile's K tiles once, in K order,
with pieces numbered 0 .. n - 1 and n at most the 16 partial planes of the
workspace; a mistake in that arithmetic would drop or double-count part of
a row's sums.  dora_selftest_grouped_schedule does the same for a grouped
launch: the module order, each module's K segments or whole-K items, and
the item -> module search the kernel runs."""
from __future__ import annotations

import random

import pytest

from dora_parameter_efficient_gb300 import api
from dora_parameter_efficient_gb300._lib import DoraError

GB300_PAIRS = 76


TABLE, RANGES, SEGMENTS = api.SCHEDULE_TABLE, api.SCHEDULE_RANGES, api.SCHEDULE_SEGMENTS
WHOLE = api.SCHEDULE_WHOLE_TABLE


@pytest.mark.parametrize("d_out,d_in,r,schedule", [
    (8192, 8192, 384, TABLE),     # fewer pair tiles (32) than pairs: one piece per pair
    (8100, 4104, 40, TABLE),
    (9000, 4104, 296, TABLE),
    (2048, 8192, 384, TABLE),
    (16384, 8192, 384, TABLE),
    (19500, 4104, 40, RANGES),    # 77 pair tiles: static ranges
    (19500, 4104, 296, RANGES),
    (20000, 4096, 384, RANGES),
    (28672, 8192, 384, WHOLE),    # 112 pair tiles: one whole tile per pair + pieces of 36
])
def test_known_shapes(d_out, d_in, r, schedule):
    got, most, defects = api.dora_selftest_schedule(d_out, d_in, r, GB300_PAIRS)
    assert defects == 0
    assert got == schedule
    assert 1 <= most <= 16


def test_piece_table_of_the_metric_workload():
    """8192 x 8192, r = 384 on 76 pairs: 32 pair tiles of 140 K tiles; the
    24 pairs behind the Gram kernel start about 26 K tiles late.  One piece
    per pair: 26 tiles in two early pieces of 70, 6 tiles in four late
    pieces of 35 (the longest piece 70, against 75 for K segments 7:4:2)."""
    got, most, defects = api.dora_selftest_schedule(8192, 8192, 384, GB300_PAIRS)
    assert (got, most, defects) == (TABLE, 4, 0)


def test_whole_tiles_of_the_moe_shaped_module():
    """28672 x 8192, r = 384 on 76 pairs: 112 pair tiles of 140 K tiles.
    Every pair runs one whole tile (76 tiles); the 36 left over are cut into
    at most one piece per pair by the piece table (early pieces for the
    first pairs, shorter late pieces for the pairs behind the Gram kernel),
    so no tile has more than two pieces."""
    got, most, defects = api.dora_selftest_schedule(28672, 8192, 384, GB300_PAIRS)
    assert (got, most, defects) == (WHOLE, 2, 0)
    # a few tiles left over would be cut into pieces shorter than the drain
    # they cost: static ranges there (79 pair tiles, 3 left over)
    got, _, defects = api.dora_selftest_schedule(20000, 8192, 384, GB300_PAIRS)
    assert (got, defects) == (RANGES, 0)


def test_seeded_sweep_of_shapes_and_grids():
    rng = random.Random(2026)
    seen = {TABLE: 0, RANGES: 0, SEGMENTS: 0, WHOLE: 0}
    for _ in range(4000):
        d_out = rng.choice([rng.randint(1, 300), rng.randint(1, 5000), rng.randint(1, 200000)])
        d_in = rng.choice([rng.randint(1, 64), rng.randint(1, 20000), rng.randint(1, 100000)])
        r = rng.choice([rng.randint(1, 16), rng.randint(1, 512)])
        pairs = rng.choice([1, 2, 3, 7, 16, 60, 74, GB300_PAIRS, 148, 1000])
        schedule, most, defects = api.dora_selftest_schedule(d_out, d_in, r, pairs)
        assert defects == 0, (d_out, d_in, r, pairs)
        assert 1 <= most <= 16, (d_out, d_in, r, pairs)
        seen[schedule] += 1
    assert min(seen.values()) > 100, seen      # every schedule exercised


@pytest.mark.parametrize("d_out", [1, 255, 256, 257, 76 * 256 - 1, 76 * 256, 76 * 256 + 1])
@pytest.mark.parametrize("d_in", [1, 64, 65, 8192])
def test_boundaries_of_tiles_and_of_the_range_rule(d_out, d_in):
    """Row counts around one tile and around as many pair tiles as pairs
    (where the plan switches to static ranges), K around one tile."""
    for r in (8, 128, 384, 512):
        schedule, most, defects = api.dora_selftest_schedule(d_out, d_in, r, GB300_PAIRS)
        assert defects == 0 and most <= 16
        if (d_out + 255) // 256 < GB300_PAIRS:
            assert schedule != RANGES


@pytest.mark.parametrize("args", [
    (0, 64, 8, 76), (64, 0, 8, 76), (64, 64, 0, 76), (64, 64, 513, 76), (64, 64, 8, 0),
    (1 << 31, 64, 8, 76),
])
def test_rejects_bad_arguments(args):
    with pytest.raises(DoraError):
        api.dora_selftest_schedule(*args)


# ------------------------------------------------------------------ grouped launches
def test_grouped_stack_of_the_7b_like_model():
    """196 modules of seven shapes: enough pair tiles for whole-K items."""
    from synthetic import configs
    cfg = configs.get(4)
    most, defects = api.dora_selftest_grouped_schedule(
        [(m.d_out, m.d_in) for m in cfg.modules], cfg.r, GB300_PAIRS)
    assert defects == 0
    assert most == 1


def test_grouped_few_modules_take_k_segments():
    most, defects = api.dora_selftest_grouped_schedule([(300, 256), (64, 512), (520, 136)], 24,
                                                       GB300_PAIRS)
    assert defects == 0
    assert most == 3


def test_grouped_seeded_sweep():
    rng = random.Random(77)
    for _ in range(400):
        n = rng.choice([1, 2, 3, 7, 50, 300])
        shapes = [(rng.choice([rng.randint(1, 600), rng.randint(1, 20000)]),
                   rng.choice([rng.randint(1, 200), rng.randint(1, 20000)])) for _ in range(n)]
        r = rng.choice([8, 64, 128, 384, 512, rng.randint(1, 512)])
        pairs = rng.choice([1, 16, GB300_PAIRS, 148])
        most, defects = api.dora_selftest_grouped_schedule(shapes, r, pairs)
        assert defects == 0, (n, r, pairs)
        assert 1 <= most <= 16


@pytest.mark.parametrize("shapes,r,pairs", [
    ([], 8, 76), ([(0, 64)], 8, 76), ([(64, 0)], 8, 76), ([(64, 64)], 0, 76),
    ([(64, 64)], 8, 0),
])
def test_grouped_rejects_bad_arguments(shapes, r, pairs):
    with pytest.raises(DoraError):
        api.dora_selftest_grouped_schedule(shapes, r, pairs)
