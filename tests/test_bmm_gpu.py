"""GPU parity of the batched scaled matmul (3-D tensor maps) against the
oracle, item by item, for every kernel family; and bit-identity with the
single-matrix entry point run on each item with the same kernel."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from fp8_scaled_gemm_gb300.inputs import make_inputs
from tests._parity import bf16_bits, compare, out_bits, unwritten_out

pytestmark = pytest.mark.gpu

TILE, SWAP, PAIR, SWAPK, SWAPPAIR = 1, 2, 3, 4, 5


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def make_batch(nb, M, N, K, mode, seed, bias, a_dtype="e4m3", b_dtype="e4m3", out_dtype="bf16"):
    """nb input sets of one shape (seeds seed..seed+nb-1); the bias of the
    first is shared by every item."""
    items = [make_inputs(M, N, K, mode, seed + i, with_bias=bias, a_dtype=a_dtype, b_dtype=b_dtype,
                         out_dtype=out_dtype) for i in range(nb)]
    shared_bias = items[0].bias
    for it in items:
        it.bias = shared_bias
    return items


def run_batch(items, mode, variant=0, tile_n=0, split_k=0):
    import fp8_scaled_gemm_gb300 as fm
    A = torch.stack([it.a_q for it in items]).cuda()
    Bt = torch.stack([it.bt_q for it in items]).cuda()
    sa = torch.cat([it.scale_a for it in items]).cuda()
    sb = torch.cat([it.scale_b for it in items]).cuda()
    bias = None if items[0].bias is None else items[0].bias.cuda()
    nb, M, N = len(items), items[0].M, items[0].N
    out = unwritten_out((nb, M, N), items[0].out_dtype)
    fm.fp8_scaled_bmm(A, Bt.transpose(1, 2), sa, sb, mode, bias=bias, out=out, variant=variant,
                      tile_n=tile_n, split_k=split_k)
    assert fm.fp8mm_device_status() == 0, fm.fp8mm_last_error()
    return out


def check_items(out, items):
    for i, it in enumerate(items):
        stats = compare(out_bits(out[i]), it)
        assert stats["violations"] == 0, f"item {i}: {stats}"


KERNELS = [(TILE, 128, 1), (TILE, 256, 1), (TILE, 128, 3), (SWAP, 16, 1), (SWAP, 64, 2), (SWAP, 128, 1),
           (PAIR, 128, 1), (PAIR, 256, 1), (PAIR, 256, 3), (PAIR, 256, -1), (SWAPK, 16, 4), (SWAPK, 128, 2),
           (SWAPPAIR, 32, 0)]


@pytest.mark.parametrize("variant,tile_n,split", KERNELS)
@pytest.mark.parametrize("mode", [0, 1])
def test_every_kernel_batched(variant, tile_n, split, mode):
    _need_gpu()
    # ragged M, N and K: an item's last tiles reach past its own rows, which
    # must read as zeros (not the next item's rows) and must not be written
    M = 300 if variant in (TILE, PAIR) else min(tile_n, 100) - 3
    items = make_batch(3, M, 520, 400, mode, seed=50 + mode, bias=(mode == 1))
    out = run_batch(items, mode, variant, tile_n, split)
    check_items(out, items)


@pytest.mark.parametrize("shape", [(8, 256, 256, 256), (64, 16, 512, 256), (4, 1024, 1024, 1024),
                                   (5, 129, 130, 144), (2, 1, 8192, 1024)])
@pytest.mark.parametrize("mode", [0, 1])
def test_auto_choice_batched(shape, mode):
    _need_gpu()
    nb, M, N, K = shape
    items = make_batch(nb, M, N, K, mode, seed=60, bias=True)
    out = run_batch(items, mode)
    check_items(out, items)


def test_batched_equals_single_calls_with_the_same_kernel():
    _need_gpu()
    import fp8_scaled_gemm_gb300 as fm
    items = make_batch(4, 300, 520, 400, 1, seed=70, bias=True)
    for variant, tile_n, split in ((TILE, 256, 1), (PAIR, 256, 1), (PAIR, 256, 4), (SWAP, 64, 3)):
        M = 300 if variant != SWAP else 60
        its = make_batch(4, M, 520, 400, 1, seed=70, bias=True)
        out = run_batch(its, 1, variant, tile_n, split)
        for i, it in enumerate(its):
            single = fm.fp8_scaled_mm_config(it.a_q.cuda(), it.bt_q.cuda().t(), it.scale_a.cuda(),
                                             it.scale_b.cuda(), 1, bias=it.bias.cuda(), variant=variant,
                                             tile_n=tile_n, split_k=split)
            assert np.array_equal(bf16_bits(out[i]), bf16_bits(single)), (variant, i)
    del items


def test_batched_other_types():
    _need_gpu()
    items = make_batch(3, 200, 300, 256, 1, seed=80, bias=True, a_dtype="e5m2", out_dtype="fp16")
    check_items(run_batch(items, 1), items)


def test_batched_full_size_sampled():
    _need_gpu()
    from tests._parity import sample_indices
    # 4 items of 2048 x 2048 x 2048, row-wise: the pair kernel over the batch
    items = make_batch(4, 2048, 2048, 2048, 1, seed=90, bias=False)
    out = run_batch(items, 1)
    rows = sample_indices(2048, 128, 16, 1)
    cols = sample_indices(2048, 128, 16, 2)
    for i, it in enumerate(items):
        stats = compare(bf16_bits(out[i])[np.ix_(rows, cols)], it, rows, cols)
        assert stats["violations"] == 0, f"item {i}: {stats}"


@pytest.mark.parametrize("variant,tile_n,split", [(TILE, 256, 1), (PAIR, 256, 1), (PAIR, 256, -1),
                                                  (TILE, 128, 3), (SWAP, 32, 1), (SWAPK, 64, 2)])
@pytest.mark.parametrize("out_dtype", ["fp32", "e4m3"])
def test_bmm_fp32_and_e4m3_outputs(variant, tile_n, split, out_dtype):
    """Items sit back to back in an output of 4- or 1-byte elements."""
    _need_gpu()
    M = 200 if variant in (TILE, PAIR) else 40
    items = make_batch(3, M, 264, 1040, 1, 70, True, out_dtype=out_dtype)
    check_items(run_batch(items, 1, variant=variant, tile_n=tile_n, split_k=split), items)
