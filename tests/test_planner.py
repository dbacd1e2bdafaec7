"""The host planner on the CPU (mxa2a_plan_preview: no device): the split,
tail-split, CTA-pair, grid and raster-group choices for the benchmark
workloads on a GB300 (152 SMs, 76 CTA pairs resident at once), each expected
value worked out by hand from the rules the header states."""
import pytest

from all_mxfp8_block_gb300 import build, mxa2a

m = mxa2a

GB300 = dict(sm_count=152, max_pairs_fused=76, max_pairs_unfused=76)
KEYS = [m.MXA2A_INFO_CTA_PAIR, m.MXA2A_INFO_CTA_PAIR_UNFUSED, m.MXA2A_INFO_TAIL_SPLIT,
        m.MXA2A_INFO_TAIL_SPLIT_UNFUSED, m.MXA2A_INFO_ITEMS, m.MXA2A_INFO_GRID_FUSED, m.MXA2A_INFO_GRID_UNFUSED,
        m.MXA2A_INFO_SPLITS, m.MXA2A_INFO_SPLITS_UNFUSED, m.MXA2A_INFO_GROUP_FUSED, m.MXA2A_INFO_GROUP_UNFUSED,
        m.MXA2A_INFO_TILE_N_FUSED, m.MXA2A_INFO_STEPS, m.MXA2A_INFO_MTILES, m.MXA2A_INFO_NTILES]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    m.load()


def preview(shape, options=(), **dev):
    return m.plan_preview(*shape, keys=KEYS, options=options, **{**GB300, **dev})


R8_8192 = (8, 8192, 1024, 8192, 512, 4)


def test_8192_cube():
    """64 x 32 tiles.  Fused: the ring holds 4 x 512 rows = 16 m-tiles, 8 pair
    rows x 32 = 256 pair tiles >= 2 x 76: CTA pairs.  1024 pair tiles on 76
    pairs leave 1024 % 76 = 36 for the last round, 2 x 36 <= 76 and K = 8192:
    split in two, 1024 - 36 + 72 = 1060 items.  Raster group: half the ring,
    2 steps of 2 pair rows.  Unfused: single CTAs, 2048 % 152 = 72 split too;
    group 16 m rows."""
    v = preview(R8_8192)
    assert v[m.MXA2A_INFO_CTA_PAIR] == 1 and v[m.MXA2A_INFO_CTA_PAIR_UNFUSED] == 0
    assert v[m.MXA2A_INFO_TAIL_SPLIT] == 2 and v[m.MXA2A_INFO_TAIL_SPLIT_UNFUSED] == 2
    assert v[m.MXA2A_INFO_ITEMS] == 1060
    assert v[m.MXA2A_INFO_GRID_FUSED] == 152 and v[m.MXA2A_INFO_GRID_UNFUSED] == 152
    assert v[m.MXA2A_INFO_SPLITS] == 1 and v[m.MXA2A_INFO_SPLITS_UNFUSED] == 1
    assert v[m.MXA2A_INFO_GROUP_FUSED] == 4 and v[m.MXA2A_INFO_GROUP_UNFUSED] == 16
    assert (v[m.MXA2A_INFO_STEPS], v[m.MXA2A_INFO_MTILES], v[m.MXA2A_INFO_NTILES]) == (16, 64, 32)


def test_8192_cube_options():
    # whole tiles: 1024 pair items
    assert preview(R8_8192, [(m.MXA2A_OPT_TAIL_SPLIT, 0)])[m.MXA2A_INFO_ITEMS] == 1024
    # single CTAs: 2048 tiles, 72 left for the last round -> 2048 - 72 + 144
    v = preview(R8_8192, [(m.MXA2A_OPT_CTA_PAIR, 0)])
    assert v[m.MXA2A_INFO_CTA_PAIR] == 0 and v[m.MXA2A_INFO_ITEMS] == 2120
    assert v[m.MXA2A_INFO_GROUP_FUSED] == 8   # half the ring in m-tiles
    # pairs on both paths
    v = preview(R8_8192, [(m.MXA2A_OPT_CTA_PAIR, 1)])
    assert v[m.MXA2A_INFO_CTA_PAIR] == 1 and v[m.MXA2A_INFO_CTA_PAIR_UNFUSED] == 1
    # a 128-column tile keeps the automatic choice on single CTAs
    v = preview(R8_8192, [(m.MXA2A_OPT_TILE_N, 128)])
    assert v[m.MXA2A_INFO_CTA_PAIR] == 0 and v[m.MXA2A_INFO_TILE_N_FUSED] == 128


def test_window_limited_problems_stay_single():
    """4 x 2048 x 4096 x 4096: the ring holds 2 x 256 rows = 4 m-tiles, 2 pair
    rows x 16 = 32 pair tiles < 152: single CTAs; K = 4096 < 8192: no tail
    split; 256 tiles, group of one step's 2 m-tiles.  8 x 4096 x 2048, K 7168:
    16 m-tiles in the ring, 8 pair rows x 8 = 64 < 152."""
    v = preview((4, 2048, 1024, 4096, 256, 2))
    assert v[m.MXA2A_INFO_CTA_PAIR] == 0 and v[m.MXA2A_INFO_TAIL_SPLIT] == 1
    assert v[m.MXA2A_INFO_ITEMS] == 256 and v[m.MXA2A_INFO_GROUP_FUSED] == 2
    v = preview((8, 4096, 896, 2048, 512, 4))
    assert v[m.MXA2A_INFO_CTA_PAIR] == 0 and v[m.MXA2A_INFO_TAIL_SPLIT] == 1 and v[m.MXA2A_INFO_ITEMS] == 256


def test_small_m_split():
    """16 x 64 x 8192 x 7168: one m-tile, 28 n-tiles; 28 x 4 <= 152 so the K
    split is min(R = 16, 152 // 28 = 5) = 5 (K / 5 >= 512): 140 items on 140
    CTAs; no pairs (one m-tile)."""
    v = preview((16, 64, 512, 7168, 64, 2))
    assert v[m.MXA2A_INFO_SPLITS] == 5 and v[m.MXA2A_INFO_SPLITS_UNFUSED] == 5
    assert v[m.MXA2A_INFO_ITEMS] == 140 and v[m.MXA2A_INFO_GRID_FUSED] == 140
    assert v[m.MXA2A_INFO_CTA_PAIR] == 0 and v[m.MXA2A_INFO_TAIL_SPLIT] == 1


def test_smallest_problem():
    """2 x 128 x 256 x 256: one tile; the fused grid covers the copy tasks
    (2 steps x 2 segments x 2 chunks of 32 rows = 8), the unfused one the tile."""
    v = preview((2, 128, 128, 256, 64, 2))
    assert v[m.MXA2A_INFO_ITEMS] == 1 and v[m.MXA2A_INFO_GRID_UNFUSED] == 1
    assert v[m.MXA2A_INFO_GRID_FUSED] == 8 and v[m.MXA2A_INFO_SPLITS] == 1


def test_split_never_exceeds_the_ctas():
    """A forced split of 8 on a grid of 4 single CTAs is cut to 4 (a tile's
    splits wait for each other, so each needs its own CTA)."""
    v = preview(R8_8192, [(m.MXA2A_OPT_CTA_PAIR, 0), (m.MXA2A_OPT_GRID, 4), (m.MXA2A_OPT_SPLIT_K, 8)])
    assert v[m.MXA2A_INFO_SPLITS] == 4 and v[m.MXA2A_INFO_SPLITS_UNFUSED] == 4
    assert v[m.MXA2A_INFO_TAIL_SPLIT] == 1   # no tail split under a uniform split


@pytest.mark.parametrize("shape,opts,want", [
    # the GPU tests' tail shape: 4 m x 2 n = 8 tiles on 6 CTAs -> 2 left, split in two
    ((2, 448, 4096, 400, 64, 4), [(m.MXA2A_OPT_GRID, 6), (m.MXA2A_OPT_SPLIT_K, 1)], (2, 6 + 2 * 2)),
    # R odd: no tail split (32 single-CTA tiles)
    ((3, 1024, 3072, 1024, 128, 4), [(m.MXA2A_OPT_CTA_PAIR, 0), (m.MXA2A_OPT_GRID, 6), (m.MXA2A_OPT_SPLIT_K, 1)],
     (1, 32)),
    # the same on automatic pairs: the ring's 2 pair rows x 4 = 8 pair tiles >= 2 x 3 pairs -> 16 pair items
    ((3, 1024, 3072, 1024, 128, 4), [(m.MXA2A_OPT_GRID, 6), (m.MXA2A_OPT_SPLIT_K, 1)], (1, 16)),
    # K = 4096: no tail split
    ((2, 448, 2048, 400, 64, 4), [(m.MXA2A_OPT_GRID, 6), (m.MXA2A_OPT_SPLIT_K, 1)], (1, 8)),
    # last round more than half the grid (8 tiles on 5: 3 left): no tail split
    ((2, 512, 4096, 400, 64, 4), [(m.MXA2A_OPT_GRID, 5), (m.MXA2A_OPT_SPLIT_K, 1)], (1, 8)),
])
def test_tail_split_rule(shape, opts, want):
    v = preview(shape, opts)
    assert (v[m.MXA2A_INFO_TAIL_SPLIT], v[m.MXA2A_INFO_ITEMS]) == want


def test_preview_rejects_bad_input():
    with pytest.raises(m.Mxa2aError) as e:
        preview((2, 100, 128, 256, 64, 2))
    assert e.value.code == m.MXA2A_ERR_INVALID_SHAPE
    with pytest.raises(m.Mxa2aError) as e:
        preview(R8_8192, sm_count=0)
    assert e.value.code == m.MXA2A_ERR_INVALID_OPTION
    with pytest.raises(m.Mxa2aError) as e:
        preview(R8_8192, [(m.MXA2A_OPT_CTA_PAIR, 3)])
    assert e.value.code == m.MXA2A_ERR_INVALID_OPTION
    with pytest.raises(m.Mxa2aError) as e:   # a run option, not a planner one
        preview(R8_8192, [(m.MXA2A_OPT_TIMEOUT_NS, 10 ** 9)])
    assert e.value.code == m.MXA2A_ERR_INVALID_OPTION
    with pytest.raises(m.Mxa2aError) as e:
        m.plan_preview(*R8_8192, keys=[m.MXA2A_INFO_WORKSPACE_BYTES], **GB300)
    assert e.value.code == m.MXA2A_ERR_INVALID_OPTION
