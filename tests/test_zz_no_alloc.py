"""The allocation-free entry point, fp8_scaled_mm_noalloc, on the GPU.

Some callers cannot allocate device memory while they run (code inside a
memory pool it does not own, or a runtime whose memory was split up front),
and fp8_scaled_mm may cudaMalloc its split-K workspace on first use. The
allocation-free entry point keeps that scratch in a fixed array inside the
library instead. These tests call it through the C ABI twice in a row on
problems whose kernel choice uses split-K (so the scratch array is really
used, and reused with the previous call's contents still in it) and compare
its output with fp8_scaled_mm's within the parity tolerance of the other GPU
tests. Problems for which fp8_scaled_mm picks stream-K (the 8192^3 benchmark
shape among them) take a whole-tile schedule here; those cases are checked
against the oracle element by element (on sampled rows and columns at
8192^3) and for unwritten elements over the whole output. This file is
collected last on purpose.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from fp8_scaled_gemm_gb300.inputs import make_inputs
from tests._parity import bf16_bits, compare, sample_indices, to_device

pytestmark = pytest.mark.gpu


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("M,N,K,mode,with_bias", [
    (200, 300, 16384, 1, True),    # very few tiles and deep K: split-K
    (300, 520, 8192, 0, False),    # split-K, ragged M and N
])
def test_noalloc_matches_fp8_scaled_mm_on_two_calls(M, N, K, mode, with_bias):
    _need_gpu()
    import fp8_scaled_gemm_gb300 as fm

    choice = fm.fp8mm_describe_choice(M, N, K, mode)
    assert "split=1 " not in choice, f"expected a split-K choice, got {choice}"
    inp = make_inputs(M, N, K, mode, seed=3, with_bias=with_bias)
    A, Bt, sa, sb, bias = to_device(inp)
    ref_out = fm.fp8_scaled_mm(A, Bt.t(), sa, sb, mode, bias=bias)
    assert fm.fp8mm_device_status() == 0
    ref_bits = bf16_bits(ref_out)
    # the per-element tolerance of the parity tests, around the existing entry's output
    _, _, absum = oracle.scaled_mm(inp.a_u8(), inp.bt_u8(), inp.sa_np(), inp.sb_np(), mode,
                                   bias=inp.bias_u16())
    tol = oracle.tolerance(ref_bits, absum)
    ref = oracle.bf16_to_f64(ref_bits)

    # both outputs exist before the calls, so any change in free device
    # memory across the two calls would come from the entry point itself
    outs = [torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    for out in outs:
        fm.fp8_scaled_mm_noalloc(A, Bt.t(), sa, sb, mode, bias=bias, out=out)
    torch.cuda.synchronize()
    free_after = torch.cuda.mem_get_info()[0]
    for call, out in enumerate(outs):
        got = oracle.bf16_to_f64(bf16_bits(out))
        bad = int((~(np.abs(got - ref) <= tol)).sum())
        assert bad == 0, f"call {call}: {bad} elements outside the tolerance"
    assert free_after == free_before


@pytest.mark.parametrize("M,N,K,mode,with_bias,sample", [
    (8192, 8192, 8192, 0, False, True),    # the benchmark shape, per-tensor
    (3000, 5000, 4112, 1, True, True),     # ragged tiles and K tail, row-wise + bias
])
def test_noalloc_on_stream_k_shapes_matches_the_oracle(M, N, K, mode, with_bias, sample):
    _need_gpu()
    import fp8_scaled_gemm_gb300 as fm

    choice = fm.fp8mm_describe_choice(M, N, K, mode)
    assert "stream_k_tiles" in choice, f"expected fp8_scaled_mm to pick stream-K, got {choice}"
    inp = make_inputs(M, N, K, mode, seed=42, with_bias=with_bias)
    A, Bt, sa, sb, bias = to_device(inp)
    ref_out = fm.fp8_scaled_mm(A, Bt.t(), sa, sb, mode, bias=bias)
    assert fm.fp8mm_device_status() == 0
    rows = sample_indices(M, 128, 96, 11) if sample else None
    cols = sample_indices(N, 128, 96, 12) if sample else None

    outs = [torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    for out in outs:
        fm.fp8_scaled_mm_noalloc(A, Bt.t(), sa, sb, mode, bias=bias, out=out)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free_before
    ref_bits = bf16_bits(ref_out)
    for call, out in enumerate(outs):
        # every element written (the inputs give finite results), on the whole output
        unwritten = int(torch.isnan(out).sum().item())
        assert unwritten == 0, f"call {call}: {unwritten} elements never written"
        bits = bf16_bits(out)
        if sample:
            bits = bits[np.ix_(rows, cols)]
        st = compare(bits, inp, rows, cols)
        assert st["violations"] == 0, f"call {call} vs oracle: {st}"
    # and against fp8_scaled_mm's stream-K result on the same grid
    got = bf16_bits(outs[1])
    if sample:
        got, ref_bits = got[np.ix_(rows, cols)], ref_bits[np.ix_(rows, cols)]
    _, _, absum = oracle.scaled_mm(inp.a_u8(), inp.bt_u8(), inp.sa_np(), inp.sb_np(), mode,
                                   bias=inp.bias_u16(), rows=rows, cols=cols)
    tol = oracle.tolerance(ref_bits, absum)
    diff = np.abs(oracle.bf16_to_f64(got) - oracle.bf16_to_f64(ref_bits))
    assert int((~(diff <= tol)).sum()) == 0


def _scratch_bytes(choice: str) -> int:
    """Split-K partial bytes of a kernel choice string ("pair tile_n=.. split=.. tiles=PxQ ...")."""
    if not choice.startswith(("tile", "swap ", "pair")):
        return 0   # the cluster kernels reduce in distributed shared memory
    f = dict(kv.split("=") for kv in choice.split()[1:])
    p, q = (int(x) for x in f["tiles"].split("x"))
    split = int(f["split"])
    rows = 256 if choice.startswith("pair") else 128
    return 0 if split == 1 else p * q * split * rows * int(f["tile_n"]) * 4


def test_noalloc_rejects_problems_beyond_the_static_scratch():
    _need_gpu()
    import fp8_scaled_gemm_gb300 as fm

    # deep K and few output tiles: the kernel choice splits K, and its fp32
    # partial tiles need more than the 16 MiB array (the first such shape)
    for M, N, K in ((512, 4352, 65536), (640, 2560, 65536), (256, 8192, 65536), (512, 8192, 65536)):
        need = _scratch_bytes(fm.fp8mm_describe_choice(M, N, K, 1))
        if need > 16 * 2 ** 20:
            break
    else:
        pytest.skip("this device's SM count gives smaller splits for the probe shapes")
    A = torch.zeros(M, K, dtype=torch.float8_e4m3fn, device="cuda")
    Bt = torch.zeros(N, K, dtype=torch.float8_e4m3fn, device="cuda")
    sa = torch.ones(M, device="cuda")
    sb = torch.ones(N, device="cuda")
    out = torch.zeros(M, N, dtype=torch.bfloat16, device="cuda")
    assert _scratch_bytes(fm.fp8mm_describe_choice(M, N, K, 1)) == need
    with pytest.raises(fm.Fp8mmError) as ei:
        fm.fp8_scaled_mm_noalloc(A, Bt.t(), sa, sb, 1, out=out)
    assert ei.value.status == -2
    assert "static scratch" in str(ei.value)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out).item() == 0   # nothing was launched
