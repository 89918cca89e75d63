"""GPU parity for operands that hold NaN and infinity codes.

The quantisation recipe never produces these codes (it clamps to the
format's finite range), so the benchmark inputs hold none. The definition
still fixes the result: the exact dot product propagates IEEE NaN and
infinity, scaling and bias keep them, and the output conversion maps them to
the output type's NaN / infinity. Positions of NaN must agree exactly, and
infinities in position and sign; every other element is held to the usual
tolerance.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from fp8_scaled_gemm_gb300.inputs import make_inputs
from tests._parity import bf16_bits, to_device

pytestmark = pytest.mark.gpu

TILE, SWAP, PAIR, SWAPK = 1, 2, 3, 4


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _run(inp, mode, variant, tile_n, split):
    import fp8_scaled_gemm_gb300 as fm
    A, Bt, sa, sb, bias = to_device(inp)
    M, N = inp.a_q.shape[0], inp.bt_q.shape[0]
    odt = torch.bfloat16 if inp.out_type == 0 else torch.float16
    out = torch.zeros((M, N), dtype=odt, device="cuda")
    fm.fp8_scaled_mm_ex(A, Bt.t(), sa, sb, mode, bias=bias, out=out, variant=variant, tile_n=tile_n,
                        split_k=split)
    assert fm.fp8mm_device_status() == 0
    return bf16_bits(out)


def _check(gpu_bits, inp):
    ref_bits, _, absum = oracle.scaled_mm(inp.a_u8(), inp.bt_u8(), inp.sa_np(), inp.sb_np(), inp.scale_mode,
                                          bias=inp.bias_u16(), **inp.oracle_types())
    gpu = oracle.out_to_f64(gpu_bits, inp.out_type)
    ref = oracle.out_to_f64(ref_bits, inp.out_type)
    assert np.isnan(ref).any(), "the case must produce NaN outputs"
    assert np.array_equal(np.isnan(gpu), np.isnan(ref)), "NaN positions differ"
    assert np.array_equal(np.isinf(gpu), np.isinf(ref)), "infinity positions differ"
    inf = np.isinf(ref)
    assert np.array_equal(np.sign(gpu[inf]), np.sign(ref[inf])), "infinity signs differ"
    fin = np.isfinite(ref)
    tol = oracle.tolerance(ref_bits, absum, inp.out_type)
    assert np.all(np.abs(gpu[fin] - ref[fin]) <= tol[fin]), "finite outputs out of tolerance"


@pytest.mark.parametrize("variant,tile_n,split", [(0, 0, 0), (TILE, 128, 2), (PAIR, 256, 1), (PAIR, 256, -1)])
def test_nan_codes_in_e4m3_operands(variant, tile_n, split):
    _need_gpu()
    M, N, K = (300, 2600, 4112) if split == -1 else (300, 520, 1040)
    inp = make_inputs(M, N, K, 1, seed=101, with_bias=True)
    a = inp.a_q.view(torch.uint8)
    bt = inp.bt_q.view(torch.uint8)
    a[7, 5] = 0x7F           # NaN: row 7 of out is NaN
    a[150, K - 1] = 0xFF     # NaN in the K tail
    bt[33, 64] = 0x7F        # NaN: column 33 of out is NaN
    _check(_run(inp, 1, variant, tile_n, split), inp)


@pytest.mark.parametrize("variant,tile_n,split", [(0, 0, 0), (SWAP, 32, 1), (SWAPK, 32, 4)])
def test_infinities_and_nans_in_e5m2_operands_skinny(variant, tile_n, split):
    _need_gpu()
    M, N, K = 24, 1000, 2048
    inp = make_inputs(M, N, K, 1, seed=102, with_bias=True, a_dtype="e5m2", b_dtype="e5m2")
    a = inp.a_q.view(torch.uint8)
    bt = inp.bt_q.view(torch.uint8)
    a[3, 10] = 0x7C          # +inf: row 3 is +-inf where nothing cancels it
    a[5, 11] = 0xFC          # -inf
    a[5, 12] = 0x7C          # +inf in the same row: inf - inf is NaN wherever both meet nonzero codes
    bt[900, 100] = 0x7E      # NaN: column 900
    bt[17, :] = 0x00         # column 17 all zero: inf x 0 = NaN in rows 3 and 5
    _check(_run(inp, 1, variant, tile_n, split), inp)
