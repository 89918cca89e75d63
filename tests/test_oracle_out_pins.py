"""Pins for the oracle's fp32 and e4m3 OUTPUT types (no GPU).

The pages cast the fp32 accumulator to the output's dtype (gist
"matmul_fp8.py", `matmul_fp8_kernel`, "Cast the accumulator to output dtype
(fp8)"; `benchmark()` takes the output dtype as an argument). Readings:

  * fp32 output: one round-to-nearest-even step from the exact value (fp64
    in the oracle); subnormals kept; 2^128 - 2^103 and above overflow to inf.
  * e4m3fn output: one round-to-nearest-even step, saturating: every value
    that rounds above 448, and +-inf, gives +-448; NaN gives 0x7F. (The
    hardware conversion such a cast lowers to saturates; PyTorch's plain
    ``.to(float8_e4m3fn)`` turns values of 464 and more into NaN instead.)
  * bias: fp32 for an fp32 output, bf16 for an e4m3 output.

What pins them, other than the oracle itself:
  * exact rational round-to-nearest-even (``fractions``) at every midpoint
    between adjacent e4m3 values and one fp64 ulp either side, and at fp32
    midpoints, subnormals and the overflow threshold;
  * numpy's float64 -> float32 conversion on a million random doubles, and
    PyTorch's CPU float32 -> float8_e4m3fn cast on every fp32 input where its
    non-saturating rule agrees (|x| < 464);
  * the saturation region and NaN, value by value;
  * exact rational brute force of the whole scaled matmul on tiny shapes;
  * planted mistakes (truncation, ties away, an fp32 step in between, a
    non-saturating overflow) fail these pins.
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from tests.test_oracle_pins import (finite_codes, finite_e5m2, frac_round, torch_e4m3_decode,
                                    torch_e5m2_decode)


# ------------------------------------------------------- exact references ---

def frac_to_f32_bits(x: Fraction) -> int:
    v = frac_round(x, 24, -126)
    if abs(v) >= Fraction(2) ** 128:
        return (0x80000000 if x < 0 else 0) | 0x7F800000
    f = np.array([float(v)], dtype=np.float32)
    assert Fraction(float(f[0])) == v          # v is an fp32 value
    return int(f.view(np.uint32)[0]) | (0x80000000 if (x < 0 and v == 0) else 0)


E4M3_VALUES = torch_e4m3_decode(np.arange(256))


def frac_to_e4m3_sat(x: Fraction) -> int:
    """Exact RNE to e4m3 (p = 4, emin = -6), then saturation at 448."""
    v = frac_round(x, 4, -6)
    sign = 0x80 if x < 0 else 0
    if abs(v) > 448:
        return sign | 0x7E
    if v == 0:
        return sign
    # the code whose value is v (a finite e4m3 value by construction)
    hits = np.flatnonzero(E4M3_VALUES == float(v))
    assert hits.size == 1
    return int(hits[0])


# -------------------------------------------------------------------- fp32 ---

def test_f32_rne_vs_exact_rational_at_midpoints():
    rng = np.random.default_rng(21)
    bits = rng.integers(0x00000001, 0x7F7FFFFF, size=4000, dtype=np.int64).astype(np.uint32)
    lo = bits.view(np.float32).astype(np.float64)
    hi = (bits + np.uint32(1)).view(np.float32).astype(np.float64)
    mids = (lo + hi) / 2                                   # exact in fp64
    xs = np.concatenate([mids, np.nextafter(mids, 0), np.nextafter(mids, np.inf), -mids])
    ours = oracle.f32_rne(xs)
    for x, o in zip(xs, ours):
        assert int(o) == frac_to_f32_bits(Fraction(float(x))), x


def test_f32_rne_matches_numpy_on_random_doubles():
    rng = np.random.default_rng(22)
    n = 1_000_000
    xs = np.ldexp(rng.random(n) + 1.0, rng.integers(-160, 130, size=n)) * np.where(rng.random(n) < 0.5, -1, 1)
    with np.errstate(over="ignore"):
        theirs = xs.astype(np.float32).view(np.uint32)
    ours = np.empty(n, np.uint32)
    step = 100_000
    for i in range(0, n, step):
        ours[i:i + step] = oracle.f32_rne(xs[i:i + step])
    assert np.array_equal(ours, theirs)


def test_f32_rne_specials():
    big = float(np.finfo(np.float32).max)
    tie_above = big + 2.0 ** 103                           # 2^128 - 2^103
    assert int(oracle.f32_rne(big)) == 0x7F7FFFFF
    assert int(oracle.f32_rne(math.nextafter(tie_above, 0))) == 0x7F7FFFFF
    assert int(oracle.f32_rne(tie_above)) == 0x7F800000
    assert int(oracle.f32_rne(-tie_above)) == 0xFF800000
    assert int(oracle.f32_rne(2.0 ** -149)) == 0x00000001
    assert int(oracle.f32_rne(2.0 ** -150)) == 0x00000000      # tie -> even (0)
    assert int(oracle.f32_rne(3 * 2.0 ** -150)) == 0x00000002  # tie -> even (2)
    assert int(oracle.f32_rne(1 + 2.0 ** -24)) == 0x3F800000   # tie -> even
    assert int(oracle.f32_rne(1 + 2.0 ** -24 + 2.0 ** -50)) == 0x3F800001   # one rounding from fp64
    assert int(oracle.f32_rne(-0.0)) == 0x80000000
    assert int(oracle.f32_rne(float("inf"))) == 0x7F800000
    assert (int(oracle.f32_rne(float("nan"))) & 0x7FFFFFFF) > 0x7F800000


# -------------------------------------------------------------------- e4m3 ---

def _e4m3_midpoints():
    """Every midpoint between adjacent non-negative finite e4m3 values, plus
    the midpoint 464 between 448 and the next value the format would have."""
    vals = np.unique(E4M3_VALUES[np.isfinite(E4M3_VALUES) & (E4M3_VALUES >= 0)])
    mids = list((vals[:-1] + vals[1:]) / 2) + [464.0]
    return np.array(mids)


def test_e4m3_sat_vs_exact_rational_at_every_midpoint():
    mids = _e4m3_midpoints()
    xs = np.concatenate([mids, np.nextafter(mids, 0), np.nextafter(mids, np.inf)])
    xs = np.concatenate([xs, -xs])
    ours = oracle.e4m3_sat(xs)
    for x, o in zip(xs, ours):
        assert int(o) == frac_to_e4m3_sat(Fraction(float(x))), x


def test_e4m3_sat_round_trips_every_finite_code():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    assert np.array_equal(oracle.e4m3_sat(E4M3_VALUES[codes]), codes)


def test_e4m3_sat_matches_torch_where_torch_does_not_overflow():
    rng = np.random.default_rng(23)
    bits = rng.integers(0, 2 ** 32, size=200_000, dtype=np.uint64).astype(np.uint32)
    f32 = bits.view(np.float32)
    f32 = f32[np.isfinite(f32) & (np.abs(f32) < 464)]
    # and every fp32 value near the e4m3 midpoints
    mids = _e4m3_midpoints().astype(np.float32)
    near = np.concatenate([mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(np.inf))])
    f32 = np.concatenate([f32, near[np.abs(near) < 464], -near[np.abs(near) < 464]])
    ours = oracle.e4m3_sat(f32.astype(np.float64))
    theirs = torch.from_numpy(f32.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, theirs)


def test_e4m3_sat_saturation_and_nan():
    for x in (448.0, 448.5, 463.999, 464.0, 480.0, 1e6, 1e300, float("inf")):
        assert int(oracle.e4m3_sat(x)) == 0x7E, x
        assert int(oracle.e4m3_sat(-x)) == 0xFE, x
    assert int(oracle.e4m3_sat(float("nan"))) == 0x7F
    assert int(oracle.e4m3_sat(-float("nan"))) == 0x7F
    assert int(oracle.e4m3_sat(0.0)) == 0x00 and int(oracle.e4m3_sat(-0.0)) == 0x80
    assert int(oracle.e4m3_sat(2.0 ** -10)) == 0x00             # tie -> even (0)
    assert int(oracle.e4m3_sat(3 * 2.0 ** -10)) == 0x02         # tie -> even (2)
    assert int(oracle.e4m3_sat(2.0 ** -6 - 2.0 ** -10)) == 0x08  # tie -> even: the smallest normal
    assert int(oracle.e4m3_sat(1.0625)) == 0x38                 # tie -> even (1.0)
    assert int(oracle.e4m3_sat(1.0625 + 2.0 ** -40)) == 0x39    # one rounding from fp64


# ------------------------------------------------- whole product, exactly ---

def exact_out(A, Bt, at, bt, sa, sb, mode, bias_vals, out_type):
    dec = {0: torch_e4m3_decode, 1: torch_e5m2_decode}
    Ad, Bd = dec[at](A), dec[bt](Bt)
    M, K = Ad.shape
    N = Bd.shape[0]
    out = np.zeros((M, N), dtype=oracle.OUT_BITS[out_type])
    for i in range(M):
        for j in range(N):
            dot = sum((Fraction(float(Ad[i, k])) * Fraction(float(Bd[j, k])) for k in range(K)),
                      Fraction(0))
            S = Fraction(float(sa[0 if mode == 0 else i])) * Fraction(float(sb[0 if mode == 0 else j]))
            v = dot * S + (Fraction(float(bias_vals[j])) if bias_vals is not None else 0)
            out[i, j] = frac_to_f32_bits(v) if out_type == oracle.F32 else frac_to_e4m3_sat(v)
    return out


def _bias(rng, n, out_type):
    """Bias bit patterns of the output type's bias dtype, and their values."""
    if out_type == oracle.F32:
        v = (rng.standard_normal(n) * 0.1).astype(np.float32)
        return v.view(np.uint32), v.astype(np.float64)
    t = (torch.from_numpy(rng.standard_normal(n)) * 0.1).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16), t.to(torch.float64).numpy()


@pytest.mark.parametrize("out_type", [oracle.F32, oracle.E4M3_OUT])
@pytest.mark.parametrize("at,bt", [(0, 0), (1, 0)])
@pytest.mark.parametrize("mode", [0, 1])
def test_brute_force_fp32_and_e4m3_outputs(out_type, at, bt, mode):
    rng = np.random.default_rng(300 + 10 * out_type + 2 * at + mode)
    M, N, K = 5, 6, 13
    gen = {0: lambda s: finite_codes(rng, s), 1: lambda s: finite_e5m2(rng, s)}
    A, Bt = gen[at]((M, K)), gen[bt]((N, K))
    # e4m3 outputs: scales that put results across the format's range,
    # including saturation; fp32: scales as the recipe gives them
    lo, hi = (2.0 ** -12, 2.0 ** -6) if out_type == oracle.E4M3_OUT else (2.0 ** -10, 2.0 ** -8)
    if at == 1:
        lo, hi = lo * 2.0 ** -7, hi * 2.0 ** -7
    n_sa, n_sb = (1, 1) if mode == 0 else (M, N)
    sa = np.exp2(rng.uniform(np.log2(lo), np.log2(hi), n_sa)).astype(np.float32)
    sb = np.exp2(rng.uniform(np.log2(lo), np.log2(hi), n_sb)).astype(np.float32)
    bias_bits, bias_vals = _bias(rng, N, out_type)
    out, _, _ = oracle.scaled_mm(A, Bt, sa, sb, mode, bias=bias_bits, a_type=at, b_type=bt,
                                 out_type=out_type)
    assert out.dtype == oracle.OUT_BITS[out_type]
    assert np.array_equal(out, exact_out(A, Bt, at, bt, sa, sb, mode, bias_vals, out_type))


def test_e4m3_output_saturates_in_the_product():
    # all-448 operands, K = 16: dot = 16 * 448^2 = 3211264; S = 2^-10 -> 3136 > 448
    A = np.full((2, 16), 0x7E, np.uint8)
    Bt = np.full((3, 16), 0x7E, np.uint8)
    Bt[1] ^= 0x80                                   # a negative column
    out, ref64, _ = oracle.scaled_mm(A, Bt, [2.0 ** -5], [2.0 ** -5], 0, out_type=oracle.E4M3_OUT)
    assert ref64[0, 0] == 3136.0
    assert out.tolist() == [[0x7E, 0xFE, 0x7E]] * 2


def test_fp32_output_closed_form():
    # all-ones, K = 4096, scales 1 and bias 0.5 (fp32): 4096.5 exactly
    A = np.full((3, 4096), 0x38, np.uint8)
    Bt = np.full((2, 4096), 0x38, np.uint8)
    bias = np.float32([0.5, -0.25]).view(np.uint32)
    out, _, _ = oracle.scaled_mm(A, Bt, [1.0], [1.0], 0, bias=bias, out_type=oracle.F32)
    assert oracle.f32_to_f64(out).tolist() == [[4096.5, 4095.75]] * 3


def test_output_pins_catch_planted_mistakes():
    """Planted roundings must fail the exact references above."""
    mids = _e4m3_midpoints()
    xs = np.concatenate([mids, np.nextafter(mids, np.inf)])
    truth = [frac_to_e4m3_sat(Fraction(float(x))) for x in xs]
    vals = np.unique(E4M3_VALUES[np.isfinite(E4M3_VALUES) & (E4M3_VALUES >= 0)])

    def code_of(v):
        return 0x7E if v > 448 else int(np.flatnonzero(E4M3_VALUES == v)[0])

    def trunc(x):
        return code_of(vals[vals <= x].max())

    def ties_away(x):
        below, above = vals[vals <= x].max(), (vals[vals >= x].min() if x <= 448 else 480.0)
        return code_of(above if (x - below) >= (above - x) else below)

    def no_saturation(x):                       # 464 and up would be NaN
        return 0x7F if x >= 464 else truth[list(xs).index(x)]

    for name, fn in {"truncation": trunc, "ties away": ties_away, "NaN on overflow": no_saturation}.items():
        assert [fn(float(x)) for x in xs] != truth, name
    # an fp32 step before rounding to e4m3 (double rounding): a value just above
    # an e4m3 midpoint that fp32 rounds onto the midpoint
    x = 1.0625 + 2.0 ** -40
    assert frac_to_e4m3_sat(Fraction(x)) == 0x39
    assert int(oracle.e4m3_sat(float(np.float32(x)))) == 0x38     # what the fp32 step would give
    # fp32: truncation instead of RNE
    assert frac_to_f32_bits(Fraction(1 + 3 * 2.0 ** -24)) == 0x3F800002 != 0x3F800001
