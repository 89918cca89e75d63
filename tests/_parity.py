"""Parity helpers: run the CUDA path through the C ABI and compare it with the
oracle element by element, on the full output or on sampled rows/columns.

Tolerance (per element): |gpu - ref| <= 2^-7 |ref| + 2^-20 * S_ij * sum_k |a_ik b_kj|
with ``ref`` the bf16-rounded oracle value (one bf16 ulp for a rounding
boundary crossed by fp32 accumulation, plus the fp32 accumulation error).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from fp8_scaled_gemm_gb300.inputs import ScaledMMInputs, make_inputs


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def out_bits(t: torch.Tensor) -> np.ndarray:
    """Bit patterns of an output tensor of any output dtype (uint16 for
    bf16 / fp16, uint32 for fp32, uint8 for e4m3fn)."""
    t = t.contiguous()
    if t.dtype == torch.float32:
        return t.view(torch.int32).cpu().numpy().view(np.uint32)
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).cpu().numpy()
    return bf16_bits(t)


def unwritten_out(shape, dtype, device="cuda") -> torch.Tensor:
    """An output buffer pre-filled with NaN (0x7F for e4m3fn), so that an
    element the kernel never writes fails the comparison."""
    if dtype == torch.float8_e4m3fn:
        return torch.full(shape, 0x7F, dtype=torch.uint8, device=device).view(dtype)
    return torch.full(shape, float("nan"), dtype=dtype, device=device)


def sample_indices(n: int, tile: int, n_random: int, seed: int) -> np.ndarray:
    """Tile-edge indices (first/last of every tile, the last index) plus random ones."""
    idx = {0, n - 1}
    for t in range(0, n, tile):
        for d in (-1, 0, 1):
            if 0 <= t + d < n:
                idx.add(t + d)
    rng = np.random.default_rng(seed)
    if n_random > 0:
        idx.update(int(i) for i in rng.integers(0, n, size=n_random))
    return np.array(sorted(idx), dtype=np.int64)


def to_device(inp: ScaledMMInputs, device="cuda"):
    A = inp.a_q.to(device)
    Bt = inp.bt_q.to(device)
    sa = inp.scale_a.to(device)
    sb = inp.scale_b.to(device)
    bias = None if inp.bias is None else inp.bias.to(device)
    return A, Bt, sa, sb, bias


def compare(gpu_bits: np.ndarray, inp: ScaledMMInputs, rows=None, cols=None, threads: int = 0):
    """Compare GPU output bits (already restricted to rows x cols) with the oracle."""
    ref_bits, _, absum = oracle.scaled_mm(
        inp.a_u8(), inp.bt_u8(), inp.sa_np(), inp.sb_np(), inp.scale_mode,
        bias=inp.bias_u16(), rows=rows, cols=cols, threads=threads, **inp.oracle_types())
    gpu = oracle.out_to_f64(gpu_bits, inp.out_type)
    ref = oracle.out_to_f64(ref_bits, inp.out_type)
    tol = oracle.tolerance(ref_bits, absum, inp.out_type)
    err = np.abs(gpu - ref)
    bad = ~(err <= tol)          # NaN in gpu counts as bad
    ratio = np.where(tol > 0, err / np.where(tol > 0, tol, 1), np.where(err > 0, np.inf, 0))
    worst = np.unravel_index(int(np.nanargmax(ratio)), ratio.shape) if ratio.size else (0, 0)
    return {
        "violations": int(bad.sum()),
        "checked": int(bad.size),
        "max_ratio": float(np.nanmax(ratio)) if ratio.size else 0.0,
        "worst": tuple(int(x) for x in worst),
        "exact_frac": float((gpu_bits == ref_bits).mean()) if ratio.size else 1.0,
    }


def run_and_compare(M, N, K, mode, seed, with_bias, variant=0, tile_n=0, split_k=0,
                    sample=False, n_random=64, inp=None, a_dtype="e4m3", b_dtype="e4m3",
                    out_dtype="bf16"):
    import fp8_scaled_gemm_gb300 as fm
    if inp is None:
        inp = make_inputs(M, N, K, mode, seed, with_bias=with_bias, a_dtype=a_dtype,
                          b_dtype=b_dtype, out_dtype=out_dtype)
    A, Bt, sa, sb, bias = to_device(inp)
    out = unwritten_out((M, N), inp.out_dtype)
    if (inp.a_type, inp.b_type, inp.out_type) == (0, 0, 0):
        fm.fp8_scaled_mm_config(A, Bt.t(), sa, sb, mode, bias=bias, out=out,
                                variant=variant, tile_n=tile_n, split_k=split_k)
    else:
        fm.fp8_scaled_mm_ex(A, Bt.t(), sa, sb, mode, bias=bias, out=out,
                            variant=variant, tile_n=tile_n, split_k=split_k)
    status = fm.fp8mm_device_status()
    assert status == 0, f"device status {status}: {fm.fp8mm_last_error()}"
    bits = out_bits(out)
    rows = cols = None
    if sample:
        rows = sample_indices(M, 128, n_random, seed + 1)
        cols = sample_indices(N, 128, n_random, seed + 2)
        bits = bits[np.ix_(rows, cols)]
    stats = compare(bits, inp, rows, cols)
    return stats, out, inp
