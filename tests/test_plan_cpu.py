"""Host scheduling logic, checked on the CPU through igc_plan_gemm against values
derived by hand from the documented rules (no GPU):

- tile width: the candidate with the smallest (rounds of tiles over the CTA pairs,
  a last round of column halves counting one half) x width / efficiency, widths
  {256, 224, 128} with efficiencies {1, 0.97, 0.87} (integer paths {256, 128});
- the last round is split into column halves when at most half of the pairs
  would be busy in it;
- 64-deep stages for fp16 / bf16 GEMMs of at most two rounds that fill at least a
  quarter of the pairs, with K >= 2048;
- panels of the first two units per pair are prefetched when both operands fit in
  64 MiB, of the first unit otherwise."""

import pytest

import implicit_gemm_conv_tcgen05_gb300 as igc

F16, BF16, S8 = igc.PLAN_GEMM_F16, igc.PLAN_GEMM_BF16, igc.PLAN_GEMM_S8


def plan(op, M, N, K, clusters=76):
    return igc.igc_plan_gemm(op, M, N, K, clusters)


def test_fp16_4096_cubed():
    # 16 x 16 = 256 tiles of 256 = 3 * 76 + 28; 2 * 28 <= 76: the last 28 tiles are
    # split into 56 halves; 256 > 2 * 76 tiles: 128-deep; 2 * 32 MiB operands
    assert plan(F16, 4096, 4096, 4096) == dict(
        tile_width=256, stage_k=128, tiles_m=16, tiles_n=16, tail_start=228, units=284,
        ctas=152, prefetch_units=2)


def test_fp16_8192_cubed_and_int8():
    # 1024 tiles = 13 * 76 + 36; 72 <= 76: split; operands 256 MiB: one unit prefetched
    want = dict(tile_width=256, stage_k=128, tiles_m=32, tiles_n=32, tail_start=988,
                units=1060, ctas=152, prefetch_units=1)
    assert plan(F16, 8192, 8192, 8192) == want
    # int8: widths 256 (13.5 rounds x 256 = 3456) or 128 (2048 tiles = 26 * 76 + 72,
    # 144 > 76: 27 rounds x 128 / 0.87 = 3972); never 64-deep
    assert plan(S8, 8192, 8192, 8192) == want


def test_skinny_takes_224_wide_64_deep():
    # widths: 256 -> 64 tiles, one round, cost 256; 224 -> 74 tiles, one round,
    # 224 / 0.97 = 230.9; 128 -> 128 tiles = 76 + 52 (104 > 76: a whole round),
    # 2 x 128 / 0.87 = 294.3.  74 tiles <= 152 and 4 * 74 >= 76, K >= 2048: 64-deep;
    # 74 % 76 = 74 and 148 > 76: no split
    assert plan(F16, 512, 8192, 8192) == dict(
        tile_width=224, stage_k=64, tiles_m=2, tiles_n=37, tail_start=74, units=74,
        ctas=148, prefetch_units=1)
    # 2048 rows: 8 x 32 = 256 tiles of 256 (3.5 rounds, cost 896) against 8 x 37 = 296
    # of 224 (296 = 3 * 76 + 68, 136 > 76: 4 rounds, 923.7): 256 wide, 128-deep
    p = plan(BF16, 2048, 8192, 8192)
    assert (p["tile_width"], p["stage_k"], p["tail_start"], p["units"]) == (256, 128, 228, 284)


def test_small_configurations():
    # 256^3: 256 wide -> 1 tile (half round, 128); 224 -> 2 tiles (112 / 0.97 = 115.5);
    # 128 -> 2 tiles (64 / 0.87 = 73.6).  2 tiles: split into 4 halves on 4 pairs
    assert plan(F16, 256, 256, 256) == dict(
        tile_width=128, stage_k=128, tiles_m=1, tiles_n=2, tail_start=0, units=4, ctas=8,
        prefetch_units=2)
    # int8 1024^3: 256 -> 16 tiles (128), 128 -> 32 tiles (64 / 0.87 = 73.6): 128 wide;
    # 2 * 32 <= 76: 64 halves
    assert plan(S8, 1024, 1024, 1024) == dict(
        tile_width=128, stage_k=128, tiles_m=4, tiles_n=8, tail_start=0, units=64, ctas=128,
        prefetch_units=2)
    # four tiles fill less than a quarter of the pairs: 128-deep although K >= 2048
    assert plan(F16, 512, 512, 2048)["stage_k"] == 128


def test_round_count_depends_on_pairs():
    # 8 pairs: 256 tiles are 32 whole rounds, nothing split
    p = plan(F16, 4096, 4096, 4096, clusters=8)
    assert (p["tail_start"], p["units"], p["ctas"]) == (256, 256, 16)
    # 200 pairs: 256 tiles = 200 + 56 and 2 * 56 <= 200: the 56 are split into 112 halves
    p = plan(F16, 4096, 4096, 4096, clusters=200)
    assert (p["tail_start"], p["units"], p["ctas"]) == (200, 312, 400)


def test_overrides_apply_and_integer_paths_ignore_224_and_depth():
    old_w = igc.igc_set_tile_width(224)
    old_d = igc.igc_set_stage_depth(64)
    try:
        p = plan(F16, 4096, 4096, 4096)
        assert (p["tile_width"], p["stage_k"], p["tiles_n"]) == (224, 64, 19)
        p = plan(S8, 4096, 4096, 4096)
        assert (p["tile_width"], p["stage_k"]) == (256, 128)
    finally:
        igc.igc_set_tile_width(old_w)
        igc.igc_set_stage_depth(old_d)
    igc.igc_set_stage_depth(128)
    try:
        assert plan(F16, 512, 8192, 8192)["stage_k"] == 128
    finally:
        igc.igc_set_stage_depth(0)


def test_invalid_queries_raise():
    for args in [(7, 64, 64, 64), (F16, 0, 64, 64), (F16, 64, 64, 0), (F16, 1 << 31, 64, 64)]:
        with pytest.raises(igc.IGCError):
            plan(*args)
