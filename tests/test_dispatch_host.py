"""Host logic of the automatic kernel choice, on any machine: the time model's
choice for a 152-SM GB300 (fp8mm_describe_model_choice needs no device).

Each expectation is a configuration measured fastest on GB300 for the shape
(CUDA-graph replays), so a change to the dispatch that moves one of them has
to come with new measurements.
"""
from __future__ import annotations

import pytest

import fp8_scaled_gemm_gb300 as fm

SMS = 152


def _choice(M, N, K, batch=1, sms=SMS):
    return fm.fp8mm_describe_model_choice(M, N, K, sms, batch)


@pytest.mark.parametrize("shape,expected", [
    # the benchmark workload: 2-SM pairs, stream-K over the last partial
    # wave plus one, tile groups of 16 rows at K = 8192
    ((8192, 8192, 8192), "pair tile_n=256 split=1 tiles=32x32 units=912 grid=152 stream_k_tiles=112 group=16"),
    # shallow K with many tiles: the 1-SM 256-wide kernel, 16 epilogue warps at K <= 512
    ((8191, 8193, 32), "tile tile_n=256 split=1 tiles=64x33 units=2112 grid=152 epilogue_warps=16"),
    ((16384, 8192, 1024), "tile tile_n=256 split=1 tiles=128x32 units=4096 grid=152"),
    # skinny M: cluster split-K, and the row-tile split for 32 < M <= 128
    ((16, 4096, 4096), "swapk tile_n=16 split=4 tiles=32x1 units=32 grid=128"),
    ((1, 8192, 8192), "swapk tile_n=16 split=4 tiles=64x1 units=64 grid=256"),
    ((16, 14336, 4096), "swapk tile_n=16 split=2 tiles=112x1 units=112 grid=224"),
    ((128, 4096, 4096), "swapk tile_n=32 split=2 tiles=32x4 units=128 grid=256"),
    ((128, 2048, 4096), "swapk tile_n=32 split=4 tiles=16x4 units=64 grid=256"),
    ((128, 14336, 4096), "swap tile_n=128 split=1 tiles=112x1 units=112 grid=112"),
    ((128, 4096, 14336), "swapk tile_n=128 split=4 tiles=32x1 units=32 grid=128"),
    # mid-size: stream-K where it pays, the unsplit pair launch where it does not
    ((3000, 5000, 4112), "pair tile_n=256 split=1 tiles=12x20 units=152 grid=152 stream_k_tiles=88 group=28"),
    ((2304, 3072, 12288), "pair tile_n=256 split=1 tiles=9x12 units=0 grid=152 stream_k_tiles=108"),
    ((4096, 4096, 4096), "pair tile_n=256 split=1 tiles=16x16 units=256 grid=152 group=32"),
    ((1024, 4096, 4096), "pair tile_n=256 split=1 tiles=4x16 units=64 grid=128 group=32"),
])
def test_model_choice_of_measured_shapes(shape, expected):
    assert _choice(*shape) == expected


@pytest.mark.parametrize("M", [33, 48, 64, 96, 100, 128])
@pytest.mark.parametrize("N,K", [(1024, 2048), (2048, 4096), (4096, 8192), (8192, 2048)])
def test_row_tile_split_rule(M, N, K):
    """32 < M <= 128, 1024 <= N <= 8192, 2048 <= K <= 8192: 32-wide tiles
    over ceil(M / 32) row tiles, clusters of 4 when they fit one wave of two
    CTAs per SM, else of 2 up to K = 4096, else the model's own choice."""
    c = _choice(M, N, K)
    nt, mt = -(-N // 128), -(-M // 32)
    if nt * mt * 4 <= 2 * SMS:
        assert c.startswith("swapk tile_n=32 split=4 "), c
    elif K <= 4096 and nt * mt * 2 <= 2 * SMS:
        assert c.startswith("swapk tile_n=32 split=2 "), c
    else:
        assert "tile_n=32 " not in c, c


@pytest.mark.parametrize("shape", [(32, 4096, 4096), (16, 2048, 4096), (128, 16384, 4096),
                                   (128, 4096, 16384), (128, 512, 4096), (64, 4096, 1024)])
def test_row_tile_split_stays_inside_its_range(shape):
    c = _choice(*shape)
    assert not (c.startswith("swapk tile_n=32 ") and shape[0] > 32), c


def test_batched_products_take_no_row_tile_split():
    c = _choice(128, 4096, 4096, batch=2)
    assert "tile_n=32 " not in c, c


@pytest.mark.parametrize("K,group", [(4096, 32), (8192, 16), (14336, 8)])
def test_tile_group_follows_the_l2_budget(K, group):
    # g = 32 MiB / (256 * K) rounded down to a multiple of 4, clamped to [4, 32]
    c = _choice(16384, 14336, K)
    assert c.startswith("pair "), c
    if group == 8:
        assert "group=" not in c, c
    else:
        assert f"group={group}" in c, c


def test_invalid_shapes_and_devices():
    assert _choice(0, 16, 16) == "no-op or invalid shape"
    assert _choice(16, 16, 8) == "no-op or invalid shape"
    assert _choice(16, 16, 16, batch=0) == "no-op or invalid shape"
    assert _choice(16, 16, 16, sms=1) == "no-op or invalid shape"


def test_grid_follows_the_sm_count():
    # a smaller device: the pair grid is its SM count (rounded to pairs)
    c = _choice(8192, 8192, 8192, sms=132)
    assert c.startswith("pair ") and "grid=132" in c, c


# ------------------------------------------------------------ quantiser ---

def _qplan(R, C, mode, sms=SMS):
    return fm.fp8mm_describe_quant_plan(R, C, mode, sms)


@pytest.mark.parametrize("C,team", [(8, "4x1 chunks=1"), (64, "8x1 chunks=1"), (128, "16x1 chunks=1"),
                                    (256, "32x1 chunks=1"), (512, "32x1 chunks=2"), (1024, "32x1 chunks=4"),
                                    (2048, "32x2 chunks=4"), (4096, "32x4 chunks=4"), (8192, "32x8 chunks=4"),
                                    (16384, "32x8 chunks=8"), (32768, "32x8 chunks=16")])
def test_row_wise_team_covers_the_row(C, team):
    """The smallest measured team whose chunks cover the row (C / 8 groups of
    8 bf16): lanes x warps threads x chunks groups >= C / 8."""
    plan = _qplan(1000, C, 1)
    assert plan == f"rows team={team}", plan
    lanes, rest = team.split("x")
    warps, chunks = rest.split(" chunks=")
    assert int(lanes) * int(warps) * int(chunks) >= C // 8


def test_row_wise_long_rows_take_the_two_pass_kernel():
    assert _qplan(10, 32776, 1) == "rows long"


@pytest.mark.parametrize("R,C,plan", [
    (16, 4096, "tensor two-launch"),                 # 128 KB: under 1 MB
    (64, 4096, "tensor two-launch"),                 # 512 KB
    (128, 4096, "tensor one-launch grid=16 tmem=0 keep=0"),    # 1 MB: 64 KB per CTA
    (16384, 1024, "tensor one-launch grid=152 tmem=0 keep=1510"),
])
def test_per_tensor_form(R, C, plan):
    assert _qplan(R, C, 0) == plan


@pytest.mark.parametrize("R,C", [(8192, 8192), (16384, 8192), (4096, 14336)])
def test_per_tensor_large_tensors_hold_a_part_in_tensor_memory(R, C):
    plan = _qplan(R, C, 0)
    assert plan.startswith("tensor one-launch grid=152 tmem=1 "), plan
    total = R * C // 8
    per_cta = -(-total // 152)
    keep = int(plan.split("keep=")[1])
    # the rest after 12288 groups in shared memory and 16384 in tensor memory,
    # capped at 96 MB of L2 over the grid
    assert keep == min(max(0, per_cta - 12288 - 16384), (96 << 20) // 16 // 152)


def test_quant_plan_rejects_bad_arguments():
    for args in [(0, 8, 0), (8, 0, 0), (8, 12, 0), (8, 8, 2)]:
        assert _qplan(*args) == "no-op or invalid shape"
    assert _qplan(8, 8, 0, sms=0) == "no-op or invalid shape"
