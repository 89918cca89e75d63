"""Failure detection on the GPU without a fault: a bounded wait runs out.

The test hook makes CTA 0's TMA producer stop after a few K blocks, so its
MMA thread waits for a barrier that nothing completes. With a short wait
budget (2^22 clock cycles, about 2 ms) the kernel must record
FP8MM_ERR_TIMEOUT in the device status word, release its tensor memory and
return; the host reads the status, and the next launches in the same
context must be correct (including split-K, whose arrival counters the
status read resets).
"""
from __future__ import annotations

import pytest
import torch

from fp8_scaled_gemm_gb300.inputs import make_inputs
from tests._parity import compare, bf16_bits, run_and_compare, to_device

pytestmark = pytest.mark.gpu

TILE, SWAP, PAIR = 1, 2, 3
SHORT = 1 << 22


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("variant,tile_n,split", [(TILE, 128, 1), (SWAP, 32, 3)])
def test_wait_runs_out_and_the_context_survives(variant, tile_n, split):
    _need_gpu()
    import fp8_scaled_gemm_gb300 as fm

    M, N, K = (300, 520, 1024) if variant == TILE else (20, 1000, 2048)
    inp = make_inputs(M, N, K, 1, seed=31, with_bias=True)
    A, Bt, sa, sb, bias = to_device(inp)
    assert fm.fp8mm_device_status() == 0
    fm.fp8mm_debug_inject(stop_after_kblocks=2, wait_limit_cycles=SHORT)
    try:
        fm.fp8_scaled_mm_config(A, Bt.t(), sa, sb, 1, bias=bias, variant=variant, tile_n=tile_n,
                                split_k=split)
        status = fm.fp8mm_device_status()
    finally:
        fm.fp8mm_debug_inject(-1, 0)
    assert status == -7, f"expected FP8MM_ERR_TIMEOUT, got {status}"
    assert "ran out" in fm.fp8mm_last_error()
    # status word cleared; the same kernel is correct again, twice
    assert fm.fp8mm_device_status() == 0
    for _ in range(2):
        stats, _, _ = run_and_compare(M, N, K, 1, 31, True, variant=variant, tile_n=tile_n,
                                      split_k=split, inp=inp)
        assert stats["violations"] == 0, stats
    assert fm.fp8mm_device_status() == 0


def test_auto_path_unaffected_after_a_timeout():
    _need_gpu()
    import fp8_scaled_gemm_gb300 as fm
    stats, _, _ = run_and_compare(1024, 1024, 512, 0, 5, False)
    assert stats["violations"] == 0, stats


def test_stream_k_flag_wait_runs_out_and_the_context_survives():
    _need_gpu()
    import fp8_scaled_gemm_gb300 as fm

    # 9 x 10 pair tiles, 11 K blocks: every tile is split between two pairs;
    # pair 1's range starts inside tile 1, which pair 0 finishes
    M, N, K = 2304, 2560, 1296
    inp = make_inputs(M, N, K, 1, seed=33, with_bias=True)
    A, Bt, sa, sb, bias = to_device(inp)
    assert fm.fp8mm_device_status() == 0
    # test hook: pair 1's partials are never flagged; pair 0's wait gives up
    fm.fp8mm_debug_inject(stop_after_kblocks=0, wait_limit_cycles=SHORT)
    try:
        fm.fp8_scaled_mm_config(A, Bt.t(), sa, sb, 1, bias=bias, variant=PAIR, tile_n=256, split_k=-1)
        status = fm.fp8mm_device_status()
    finally:
        fm.fp8mm_debug_inject(-1, 0)
    assert status == -7, f"expected FP8MM_ERR_TIMEOUT, got {status}"
    # the status read cleared the flags: the same launch is exact again, twice
    for _ in range(2):
        stats, _, _ = run_and_compare(M, N, K, 1, 33, True, variant=PAIR, tile_n=256, split_k=-1, inp=inp,
                                      sample=True, n_random=32)
        assert stats["violations"] == 0, stats
    assert fm.fp8mm_device_status() == 0


def test_per_tensor_grid_wait_runs_out_and_the_context_survives():
    """CTA 0 of the one-launch per-tensor quantisation withholds its share of
    the grid-wide amax (test hook): every CTA's bounded wait runs out, the
    status word says so, and the next calls are correct."""
    _need_gpu()
    import numpy as np
    import oracle
    import fp8_scaled_gemm_gb300 as fm
    from fp8_scaled_gemm_gb300.inputs import bf16_matrix

    x = bf16_matrix(4096, 4096, seed=34)
    xd = x.cuda()
    assert fm.fp8mm_device_status() == 0
    fm.fp8mm_debug_inject(-1, SHORT)
    fm.fp8mm_debug_quant(2)
    try:
        fm.fp8_quantize(xd, 0)
        status = fm.fp8mm_device_status()
    finally:
        fm.fp8mm_debug_quant(0)
        fm.fp8mm_debug_inject(-1, 0)
    assert status == -7, f"expected FP8MM_ERR_TIMEOUT, got {status}"
    assert "ran out" in fm.fp8mm_last_error()
    assert fm.fp8mm_device_status() == 0
    q_ref, s_ref = oracle.quantize(x.view(torch.int16).numpy().view(np.uint16), 0, 0)
    for _ in range(2):
        q, s = fm.fp8_quantize(xd, 0)
        torch.cuda.synchronize()
        assert np.array_equal(q.view(torch.uint8).cpu().numpy(), q_ref)
        assert s.cpu().numpy().view(np.uint32)[0] == s_ref.view(np.uint32)[0]
    assert fm.fp8mm_device_status() == 0
