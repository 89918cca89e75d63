"""GPU parity of the four operand layouts (A row- or column-major, B row- or
column-major) against the oracle, which reads the same codes in the TN form
(the layout only changes where each code sits in memory)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from fp8_scaled_gemm_gb300.inputs import make_inputs
from tests._parity import bf16_bits, compare, sample_indices

pytestmark = pytest.mark.gpu


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def run_layout(inp, a_col: bool, b_row: bool, mode: int, **kw):
    import fp8_scaled_gemm_gb300 as fm
    A = inp.a_q.cuda()                       # [M, K] row-major
    Bt = inp.bt_q.cuda()                     # [N, K] row-major = B column-major
    A_arg = A.t().contiguous().t() if a_col else A          # same values, M contiguous
    B_arg = Bt.t().contiguous() if b_row else Bt.t()        # [K, N]: row-major, or column-major view
    out = fm.fp8_scaled_mm_layout(A_arg, B_arg, inp.scale_a.cuda(), inp.scale_b.cuda(), mode,
                                  bias=None if inp.bias is None else inp.bias.cuda(), **kw)
    assert fm.fp8mm_device_status() == 0
    return out


LAYOUTS = [(False, False), (True, False), (False, True), (True, True)]


@pytest.mark.parametrize("a_col,b_row", LAYOUTS)
@pytest.mark.parametrize("shape", [(300, 520, 400), (256, 256, 256), (17, 1000, 96), (1, 40, 16), (129, 7, 48)])
@pytest.mark.parametrize("mode", [0, 1])
def test_layouts_full_output(a_col, b_row, shape, mode):
    _need_gpu()
    M, N, K = shape
    inp = make_inputs(M, N, K, mode, seed=100 + M, with_bias=(mode == 1))
    out = run_layout(inp, a_col, b_row, mode)
    stats = compare(bf16_bits(out), inp)
    assert stats["violations"] == 0, (a_col, b_row, shape, stats)


@pytest.mark.parametrize("a_col,b_row", LAYOUTS[1:])
def test_layouts_equal_the_tn_result(a_col, b_row):
    _need_gpu()
    # the transposed copy feeds the same kernel, so the bits match the TN call
    inp = make_inputs(1000, 777, 528, 1, seed=7, with_bias=True)
    tn = run_layout(inp, False, False, 1)
    other = run_layout(inp, a_col, b_row, 1)
    assert np.array_equal(bf16_bits(tn), bf16_bits(other))


def test_layouts_full_size_sampled():
    _need_gpu()
    inp = make_inputs(4096, 4096, 4096, 1, seed=42, with_bias=False)
    out = run_layout(inp, True, True, 1)
    rows = sample_indices(4096, 128, 32, 1)
    cols = sample_indices(4096, 128, 32, 2)
    stats = compare(bf16_bits(out)[np.ix_(rows, cols)], inp, rows, cols)
    assert stats["violations"] == 0, stats


def test_layout_other_types():
    _need_gpu()
    inp = make_inputs(300, 520, 400, 1, seed=9, with_bias=True, a_dtype="e5m2", b_dtype="e4m3",
                      out_dtype="fp16")
    out = run_layout(inp, True, True, 1, out_dtype=torch.float16)
    stats = compare(bf16_bits(out), inp)
    assert stats["violations"] == 0, stats
