"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Small cases compare every output element; they span several tiles with a
ragged tail in M, N and K. The configurations of the benchmark workloads are
run at full size and compared on sampled rows and columns (every tile edge
plus random indices), which the oracle computes one by one.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from tests._parity import bf16_bits, compare, run_and_compare, to_device

pytestmark = pytest.mark.gpu

TILE, SWAP, PAIR, SWAPK, SWAPPAIR = 1, 2, 3, 4, 5


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _assert_ok(stats, label):
    assert stats["violations"] == 0, f"{label}: {stats}"


# ------------------------------------------------------------ small, full ---

KERNELS = [(TILE, 128), (TILE, 256), (SWAP, 16), (SWAP, 32), (SWAP, 64), (SWAP, 128),
           (PAIR, 128), (PAIR, 256), (SWAPPAIR, 16), (SWAPPAIR, 32), (SWAPPAIR, 64), (SWAPPAIR, 128)]


@pytest.mark.parametrize("variant,tile_n", KERNELS)
@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("split", [1, 3])
def test_every_kernel_on_a_ragged_shape(variant, tile_n, mode, split):
    _need_gpu()
    # M, N, K all ragged: 2+ tiles in each direction and a K tail of 16. For
    # PAIR the last 256-row tile leaves the odd CTA's rows entirely out of
    # range, and the last column tile leaves the odd CTA's Bt half empty.
    M, N, K = 300, 520, 400
    stats, _, _ = run_and_compare(M, N, K, mode, seed=11, with_bias=(split == 3),
                                  variant=variant, tile_n=tile_n,
                                  split_k=(1 if variant == SWAPPAIR else split))
    _assert_ok(stats, f"v{variant} n{tile_n} mode{mode} split{split}")


@pytest.mark.parametrize("shape", [
    (256, 256, 256),            # the small per-tensor configuration (seed 0)
    (1, 1, 16), (1, 7, 32), (7, 1, 48), (127, 129, 144), (129, 127, 16),
    (255, 257, 128), (16, 77, 64),  # N odd: scalar stores
    (64, 4096, 1024),
])
@pytest.mark.parametrize("mode", [0, 1])
def test_auto_choice_edge_shapes(shape, mode):
    _need_gpu()
    M, N, K = shape
    stats, _, _ = run_and_compare(M, N, K, mode, seed=0, with_bias=(mode == 1))
    _assert_ok(stats, f"{shape} mode{mode}")


@pytest.mark.parametrize("shape", [(129, 300, 256), (512, 512, 1024), (1000, 777, 48)])
def test_pair_kernel_shapes(shape):
    _need_gpu()
    M, N, K = shape
    for tile_n in (128, 256):
        stats, _, _ = run_and_compare(M, N, K, 1, seed=4, with_bias=True, variant=PAIR,
                                      tile_n=tile_n, split_k=1)
        _assert_ok(stats, f"pair{tile_n} {shape}")


@pytest.mark.parametrize("split", [2, 3, 5, 8])
@pytest.mark.parametrize("tile_n", [128, 256])
def test_pair_kernel_split_k(split, tile_n):
    _need_gpu()
    # ragged M, N and K (K blocks not divisible by the split), bias, both modes
    for mode in (0, 1):
        stats, _, _ = run_and_compare(300, 520, 1296, mode, seed=24 + split, with_bias=(mode == 1),
                                      variant=PAIR, tile_n=tile_n, split_k=split)
        _assert_ok(stats, f"pair{tile_n} split{split} mode{mode}")


def test_pair_split_k_is_deterministic_and_reuses_counters():
    _need_gpu()
    import fp8_scaled_gemm_gb300 as fm
    from fp8_scaled_gemm_gb300.inputs import make_inputs
    inp = make_inputs(512, 1024, 4096, 1, seed=31, with_bias=True)
    A, Bt, sa, sb, bias = to_device(inp)
    outs = [bf16_bits(fm.fp8_scaled_mm_config(A, Bt.t(), sa, sb, 1, bias=bias, variant=PAIR, tile_n=256,
                                              split_k=4)) for _ in range(3)]
    assert fm.fp8mm_device_status() == 0
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[1], outs[2])
    _assert_ok(compare(outs[0], inp), "pair split4")


@pytest.mark.parametrize("tile_n", [16, 32, 64, 128])
@pytest.mark.parametrize("cs", [2, 4, 8])
def test_cluster_k_kernel(tile_n, cs):
    _need_gpu()
    # ragged M, N and K; K blocks not divisible by the cluster size
    M, N, K = min(tile_n, 100) - 3, 300, 1296
    for mode, bias in ((0, False), (1, True)):
        stats, _, _ = run_and_compare(M, N, K, mode, seed=21, with_bias=bias, variant=SWAPK,
                                      tile_n=tile_n, split_k=cs)
        _assert_ok(stats, f"swapk n{tile_n} cs{cs} mode{mode}")


@pytest.mark.parametrize("tile_n", [16, 32, 64, 128])
def test_swap_pair_kernel(tile_n):
    _need_gpu()
    # ragged M and N: the last 256-row pair tile leaves the odd CTA with
    # N rows 384..511 out of range; K tail of 16
    M, N, K = max(1, tile_n - 5), 600, 784
    for mode, bias in ((0, False), (1, True)):
        stats, _, _ = run_and_compare(M, N, K, mode, seed=23, with_bias=bias, variant=SWAPPAIR,
                                      tile_n=tile_n, split_k=0)
        _assert_ok(stats, f"swappair n{tile_n} mode{mode}")


def test_cluster_k_with_fewer_k_blocks_than_ctas():
    _need_gpu()
    # K = 272 is 3 K blocks over a cluster of 8: five CTAs have no K block
    stats, _, _ = run_and_compare(20, 260, 272, 1, seed=22, with_bias=True, variant=SWAPK,
                                  tile_n=32, split_k=8)
    _assert_ok(stats, "swapk empty slices")


def test_cluster_k_is_deterministic():
    _need_gpu()
    import fp8_scaled_gemm_gb300 as fm
    from fp8_scaled_gemm_gb300.inputs import make_inputs
    inp = make_inputs(16, 4096, 4096, 1, seed=6, with_bias=True)
    A, Bt, sa, sb, bias = to_device(inp)
    outs = [bf16_bits(fm.fp8_scaled_mm_config(A, Bt.t(), sa, sb, 1, bias=bias, variant=SWAPK,
                                              tile_n=16, split_k=8)) for _ in range(3)]
    assert fm.fp8mm_device_status() == 0
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[1], outs[2])
    _assert_ok(compare(outs[0], inp), "swapk det")


def test_empty_problems_leave_out_untouched():
    _need_gpu()
    import fp8_scaled_gemm_gb300 as fm
    A = torch.zeros(0, 32, dtype=torch.float8_e4m3fn, device="cuda")
    Bt = torch.zeros(8, 32, dtype=torch.float8_e4m3fn, device="cuda")
    one = torch.ones(1, device="cuda")
    out = torch.empty(0, 8, dtype=torch.bfloat16, device="cuda")
    fm.fp8_scaled_mm(A, Bt.t(), one, one, 0, out=out)
    torch.cuda.synchronize()


def test_split_k_is_deterministic_and_workspace_is_reusable():
    _need_gpu()
    import fp8_scaled_gemm_gb300 as fm
    from fp8_scaled_gemm_gb300.inputs import make_inputs
    inp = make_inputs(48, 1000, 2048, 1, seed=5, with_bias=True)
    A, Bt, sa, sb, bias = to_device(inp)
    outs = []
    for _ in range(3):
        o = fm.fp8_scaled_mm_config(A, Bt.t(), sa, sb, 1, bias=bias, variant=SWAP, tile_n=64,
                                    split_k=7)
        outs.append(bf16_bits(o))
    assert fm.fp8mm_device_status() == 0
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[1], outs[2])
    _assert_ok(compare(outs[0], inp), "split7")


def test_host_entry_matches_device_entry():
    _need_gpu()
    import fp8_scaled_gemm_gb300 as fm
    from fp8_scaled_gemm_gb300.inputs import make_inputs
    inp = make_inputs(200, 333, 160, 1, seed=9, with_bias=True)
    A, Bt, sa, sb, bias = to_device(inp)
    dev = bf16_bits(fm.fp8_scaled_mm(A, Bt.t(), sa, sb, 1, bias=bias))
    host = fm.fp8_scaled_mm_host(inp.a_q.pin_memory(), inp.bt_q.pin_memory().t(),
                                 inp.scale_a, inp.scale_b, 1, bias=inp.bias)
    assert np.array_equal(dev, bf16_bits(host))
    _assert_ok(compare(dev, inp), "host/device")


def test_host_entry_in_several_chunks():
    _need_gpu()
    import fp8_scaled_gemm_gb300 as fm
    from fp8_scaled_gemm_gb300.inputs import make_inputs
    # 3000 rows: three 1024-row chunks (the last one ragged), row-wise + bias
    inp = make_inputs(3000, 1000, 528, 1, seed=12, with_bias=True)
    host = fm.fp8_scaled_mm_host(inp.a_q.pin_memory(), inp.bt_q.pin_memory().t(),
                                 inp.scale_a.pin_memory(), inp.scale_b.pin_memory(), 1,
                                 bias=inp.bias.pin_memory())
    _assert_ok(compare(bf16_bits(host), inp), "host chunks")
    # a second call reuses the staging buffers and the pipeline
    host2 = fm.fp8_scaled_mm_host(inp.a_q, inp.bt_q.t(), inp.scale_a, inp.scale_b, 1, bias=inp.bias)
    assert np.array_equal(bf16_bits(host), bf16_bits(host2))


# ------------------------------------------------- other element types ------

TYPES = [("e5m2", "e5m2", "bf16"), ("e4m3", "e5m2", "fp16"), ("e5m2", "e4m3", "fp16"),
         ("e4m3", "e4m3", "fp32"), ("e4m3", "e4m3", "e4m3"), ("e5m2", "e4m3", "e4m3")]


@pytest.mark.parametrize("variant,tile_n,split", [
    (TILE, 128, 1), (TILE, 256, 2), (SWAP, 16, 1), (SWAP, 64, 3), (PAIR, 256, 0),
    (SWAPK, 16, 4), (SWAPK, 128, 2), (SWAPPAIR, 32, 0)])
@pytest.mark.parametrize("types", TYPES)
def test_other_element_types_every_kernel(variant, tile_n, split, types):
    _need_gpu()
    at, bt, ot = types
    M = 300 if variant in (TILE, PAIR) else min(tile_n, 100) - 3
    stats, _, _ = run_and_compare(M, 520, 400, 1, seed=41, with_bias=True, variant=variant,
                                  tile_n=tile_n, split_k=split, a_dtype=at, b_dtype=bt, out_dtype=ot)
    _assert_ok(stats, f"v{variant} n{tile_n} {types}")


@pytest.mark.parametrize("types", TYPES)
def test_other_element_types_auto_full_size_sampled(types):
    _need_gpu()
    at, bt, ot = types
    stats, _, _ = run_and_compare(8192, 8192, 8192, 0, 42, False, sample=True, n_random=32,
                                  a_dtype=at, b_dtype=bt, out_dtype=ot)
    _assert_ok(stats, f"8192^3 {types}")
    stats, _, _ = run_and_compare(16, 4096, 4096, 1, 42, True, sample=True, n_random=32,
                                  a_dtype=at, b_dtype=bt, out_dtype=ot)
    _assert_ok(stats, f"16x4096x4096 {types}")


# ------------------------------------------------- full-size, sampled -------

BENCH_SHAPES = [
    (8192, 8192, 8192, 0, 42, False),   # per-tensor, the headline shape
    (8192, 8192, 8192, 1, 42, False),   # row-wise, the headline shape
    (3000, 5000, 4112, 1, 42, True),    # tails in M, N, K + bias
    (16384, 8192, 1024, 1, 42, True),
    (1, 8192, 8192, 1, 42, True),
    (8191, 8193, 32, 1, 42, True),      # N odd, K = 32
]

SWEEP = [(m, n, k) for m in (16, 128, 1024, 4096, 16384)
         for (n, k) in ((4096, 4096), (14336, 4096), (4096, 14336))]


@pytest.mark.parametrize("M,N,K,mode,seed,bias", BENCH_SHAPES)
def test_full_size_configs_sampled(M, N, K, mode, seed, bias):
    _need_gpu()
    stats, _, _ = run_and_compare(M, N, K, mode, seed, bias, sample=True)
    _assert_ok(stats, f"{(M, N, K)} mode{mode}")


@pytest.mark.parametrize("M,N,K", SWEEP)
def test_rowwise_sweep_sampled(M, N, K):
    _need_gpu()
    stats, _, _ = run_and_compare(M, N, K, 1, 42, False, sample=True, n_random=32)
    _assert_ok(stats, f"sweep {(M, N, K)}")


def test_host_entry_in_blocks():
    _need_gpu()
    import fp8_scaled_gemm_gb300 as fm
    from fp8_scaled_gemm_gb300.inputs import make_inputs
    # 3300 x 3100: 3 x 3 blocks of the growing-square schedule (chunks of
    # 1280, 1024 and 996 / 796 rows), ragged in both directions; row-wise
    # scales and bias are sliced per block
    for mode, bias in ((1, True), (0, False)):
        inp = make_inputs(3300, 3100, 528, mode, seed=13, with_bias=bias)
        host = fm.fp8_scaled_mm_host(inp.a_q.pin_memory(), inp.bt_q.pin_memory().t(),
                                     inp.scale_a.pin_memory(), inp.scale_b.pin_memory(), mode,
                                     bias=None if inp.bias is None else inp.bias.pin_memory())
        _assert_ok(compare(bf16_bits(host), inp), f"host blocks mode{mode}")


# ------------------------------------------------------------- stream-K -----

@pytest.mark.parametrize("mode", [0, 1])
def test_pair_stream_k_ragged(mode):
    _need_gpu()
    # 2 x 11 pair tiles (fewer than the pairs) with 33 K blocks (a K tail of
    # 16): every tile's K blocks are spread over several pairs, and each tile
    # is finished by the pair holding its first K block
    stats, _, _ = run_and_compare(300, 2600, 4112, mode, seed=61, with_bias=(mode == 1), variant=PAIR,
                                  tile_n=256, split_k=-1)
    _assert_ok(stats, f"stream-K ragged mode{mode}")


def test_pair_stream_k_between_one_and_two_waves():
    _need_gpu()
    # 9 x 10 = 90 pair tiles: all of them in the stream-K region
    stats, _, _ = run_and_compare(2304, 2560, 1296, 1, seed=62, with_bias=True, variant=PAIR, tile_n=256,
                                  split_k=-1, sample=True, n_random=48)
    _assert_ok(stats, "stream-K 90 tiles")


@pytest.mark.parametrize("tile_n", [256, 128])
def test_pair_stream_k_partial_through_ring(tile_n):
    _need_gpu()
    # 7 x 11 (tile_n 256) or 7 x 22 (128) pair tiles, 5 K blocks with a tail
    # of 16: more tiles than pairs, so every pair's stream-K range covers at
    # least a whole tile and an owner adds exactly one partial, which its
    # producer copies into the drained operand ring; full-output compare
    stats, _, _ = run_and_compare(1700, 2700, 528, 1, seed=65, with_bias=True, variant=PAIR, tile_n=tile_n,
                                  split_k=-1)
    _assert_ok(stats, f"stream-K ring tile_n={tile_n}")


def test_pair_stream_k_is_deterministic():
    _need_gpu()
    import fp8_scaled_gemm_gb300 as fm
    from fp8_scaled_gemm_gb300.inputs import make_inputs
    inp = make_inputs(512, 3072, 4096, 1, seed=63, with_bias=True)
    A, Bt, sa, sb, bias = to_device(inp)
    outs = [bf16_bits(fm.fp8_scaled_mm_config(A, Bt.t(), sa, sb, 1, bias=bias, variant=PAIR, tile_n=256,
                                              split_k=-1)) for _ in range(3)]
    assert fm.fp8mm_device_status() == 0
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[1], outs[2])
    _assert_ok(compare(outs[0], inp), "stream-K det")


@pytest.mark.parametrize("at,ot", [("e5m2", "fp16"), ("e4m3", "fp32"), ("e4m3", "e4m3")])
def test_pair_stream_k_other_types(at, ot):
    _need_gpu()
    # 300 x 2600 has fewer tiles than pairs (partials read through L2);
    # 2304 x 3072 has more (one partial, copied into the ring)
    for M, N, K in ((300, 2600, 4112), (2304, 3072, 2048)):
        stats, _, _ = run_and_compare(M, N, K, 1, seed=64, with_bias=True, variant=PAIR, tile_n=256,
                                      split_k=-1, a_dtype=at, out_dtype=ot, sample=M > 1000)
        _assert_ok(stats, f"stream-K {(M, N, K)} {at}/{ot}")


@pytest.mark.parametrize("ot", ["fp32", "e4m3"])
@pytest.mark.parametrize("N", [4099, 4104, 4112])
def test_fp32_and_e4m3_outputs_unaligned_rows(ot, N):
    """Rows that are not 16-byte aligned take element stores; aligned ones 16-byte stores."""
    _need_gpu()
    for variant, tile_n, split in ((TILE, 256, 1), (PAIR, 256, 1), (TILE, 128, 2), (SWAP, 32, 1)):
        M = 37 if variant == SWAP else 300
        stats, _, _ = run_and_compare(M, N, 160, 1, seed=65, with_bias=True, variant=variant,
                                      tile_n=tile_n, split_k=split, out_dtype=ot)
        _assert_ok(stats, f"{ot} N={N} v{variant}")


def test_e4m3_output_saturates_like_the_oracle():
    """Large scales push most outputs past 448: both sides saturate."""
    _need_gpu()
    from fp8_scaled_gemm_gb300.inputs import make_inputs
    inp = make_inputs(256, 384, 512, 0, seed=66, out_dtype="e4m3")
    inp.scale_a = inp.scale_a * 64
    stats, out, _ = run_and_compare(256, 384, 512, 0, 66, False, inp=inp)
    _assert_ok(stats, "e4m3 saturation")
    codes = out.view(torch.uint8).cpu().numpy()
    assert ((codes & 0x7F) == 0x7E).mean() > 0.2     # many saturated
    assert not ((codes & 0x7F) == 0x7F).any()        # no NaN


# M above 32 with 16 to 32 column tiles: the automatic choice splits M into
# 32-row tiles over clusters of 4 (or 2), ragged M included.
@pytest.mark.parametrize("shape,choice", [
    ((128, 2048, 4096), "swapk tile_n=32 split=4"),
    ((128, 4096, 4096), "swapk tile_n=32 split=2"),
    ((100, 2056, 2048), "swapk tile_n=32 split=4"),
    ((48, 4096, 8192), "swapk tile_n=32 split=4"),
    ((64, 8192, 2048), "swapk tile_n=32 split=2"),
    ((128, 1024, 4096), "swapk tile_n=32 split=4"),
])
@pytest.mark.parametrize("mode", [0, 1])
def test_auto_row_split_skinny(shape, choice, mode):
    _need_gpu()
    import fp8_scaled_gemm_gb300 as fm
    M, N, K = shape
    assert fm.fp8mm_describe_choice(M, N, K, mode).startswith(choice)
    stats, _, _ = run_and_compare(M, N, K, mode, seed=12, with_bias=(mode == 1))
    _assert_ok(stats, f"{shape} mode{mode}")
