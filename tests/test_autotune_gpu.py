"""Shape-keyed autotuning on the GPU: a tuned choice is taken by automatic
kernel choice for exactly its shape and types, keeps parity with the oracle,
and survives save / clear / load."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from fp8_scaled_gemm_gb300.inputs import make_inputs
from tests._parity import run_and_compare

pytestmark = pytest.mark.gpu


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.fixture(autouse=True)
def _clean_table():
    if torch.cuda.is_available():
        import fp8_scaled_gemm_gb300 as fm
        fm.fp8mm_autotune_clear()
        yield
        fm.fp8mm_autotune_clear()
    else:
        yield


@pytest.mark.parametrize("shape,mode", [((512, 3072, 12288), 1), ((16, 4096, 4096), 1), ((300, 520, 400), 0),
                                        ((1, 8192, 1024), 1)])
def test_tuned_choice_is_used_and_keeps_parity(shape, mode):
    _need_gpu()
    import fp8_scaled_gemm_gb300 as fm
    M, N, K = shape
    builtin = fm.fp8mm_describe_choice(M, N, K, mode)
    neighbour = fm.fp8mm_describe_choice(M, N + 16, K, mode)
    chosen = fm.fp8mm_autotune(M, N, K, mode)
    assert fm.fp8mm_autotune_count() == 1
    assert fm.fp8mm_describe_choice(M, N, K, mode) == chosen
    assert chosen.split()[0] in ("tile", "swap", "pair", "swapk", "swappair")
    # a neighbouring shape keeps the built-in choice
    assert fm.fp8mm_describe_choice(M, N + 16, K, mode) == neighbour
    stats, _, _ = run_and_compare(M, N, K, mode, seed=5, with_bias=True, sample=(M * N > 2 ** 20))
    assert stats["violations"] == 0, (chosen, builtin, stats)
    fm.fp8mm_autotune_clear()
    assert fm.fp8mm_describe_choice(M, N, K, mode) == builtin


def test_tuned_choices_survive_save_clear_load(tmp_path):
    _need_gpu()
    import fp8_scaled_gemm_gb300 as fm
    a = fm.fp8mm_autotune(768, 2048, 8192, 1)
    b = fm.fp8mm_autotune(128, 4096, 4096, 0)
    path = tmp_path / "tuned.txt"
    assert fm.fp8mm_autotune_save(str(path)) == 2
    fm.fp8mm_autotune_clear()
    assert fm.fp8mm_autotune_count() == 0
    assert fm.fp8mm_autotune_load(str(path)) == 2
    assert fm.fp8mm_describe_choice(768, 2048, 8192, 1) == a
    assert fm.fp8mm_describe_choice(128, 4096, 4096, 0) == b


def test_tuning_other_types_and_batches():
    _need_gpu()
    import fp8_scaled_gemm_gb300 as fm
    fm.fp8mm_autotune(300, 520, 1024, 1, a_dtype=torch.float8_e5m2, out_dtype=torch.float16)
    stats, _, _ = run_and_compare(300, 520, 1024, 1, seed=6, with_bias=True, a_dtype="e5m2", out_dtype="fp16")
    assert stats["violations"] == 0, stats
    fm.fp8mm_autotune(1024, 1024, 1024, 1, batch=4)
    from tests.test_bmm_gpu import check_items, make_batch, run_batch
    items = make_batch(4, 1024, 1024, 1024, 1, seed=7, bias=True)
    check_items(run_batch(items, 1), items)
