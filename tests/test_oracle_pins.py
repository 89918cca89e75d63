"""Pins for the CPU oracle (no GPU).

Each test ties the oracle to something other than itself: torch's own float8
and bf16 conversions (independent implementations), exact rational brute force
with Python's ``fractions``, closed forms whose results are exactly
representable, the fp64-exactness invariant on the 2^-18 grid, and the one
value the pages fix (the largest e4m3fn value, 448: gist "matmul_fp8.py",
``benchmark()``, ``quant_max = torch.finfo(dtype).max``).

The last test plants mistakes in calls to the oracle and checks that the
brute-force pin fails for each one.
"""
from __future__ import annotations

import math
import os
import struct
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- helpers ---

def torch_e4m3_decode(codes) -> np.ndarray:
    t = torch.as_tensor(np.asarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def frac_to_bf16_bits(x: Fraction) -> int:
    """Exact rational -> bf16 RNE by integer arithmetic (independent method)."""
    if x == 0:
        return 0
    sign = 0x8000 if x < 0 else 0
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -126)
    q = a / (Fraction(2) ** (e - 7))
    n = q.numerator // q.denominator
    rem = q - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    v = n * Fraction(2) ** (e - 7)
    if v >= Fraction(2) ** 128:
        return sign | 0x7F80
    (w,) = struct.unpack(">I", struct.pack(">f", float(v)))
    assert float(v) == v  # v is a bf16 value, hence exact in fp32
    assert w & 0xFFFF == 0
    return sign | (w >> 16)


def exact_scaled_mm(A, Bt, sa, sb, mode, bias_bits):
    """Brute force: exact rational sum, scale and bias, then exact RNE."""
    Ad = torch_e4m3_decode(A)
    Bd = torch_e4m3_decode(Bt)
    M, K = Ad.shape
    N = Bd.shape[0]
    out = np.zeros((M, N), dtype=np.uint16)
    bias_vals = None
    if bias_bits is not None:
        bias_vals = torch.from_numpy(np.asarray(bias_bits, np.uint16).view(np.int16)) \
            .view(torch.bfloat16).to(torch.float64).numpy()
    for i in range(M):
        for j in range(N):
            dot = sum((Fraction(float(Ad[i, k])) * Fraction(float(Bd[j, k])) for k in range(K)),
                      Fraction(0))
            if mode == 0:
                S = Fraction(float(sa[0])) * Fraction(float(sb[0]))
            else:
                S = Fraction(float(sa[i])) * Fraction(float(sb[j]))
            v = dot * S
            if bias_vals is not None:
                v += Fraction(float(bias_vals[j]))
            out[i, j] = frac_to_bf16_bits(v)
    return out


def finite_codes(rng, shape, allow_subnormal=True):
    """Random e4m3 codes without the two NaN codes."""
    c = rng.integers(0, 256, size=shape, dtype=np.int64)
    c = np.where((c & 0x7F) == 0x7F, c - 1, c)
    if not allow_subnormal:
        c = np.where(((c >> 3) & 0xF) == 0, c | 0x08, c)
    return c.astype(np.uint8)


def bf16_bits_of(values) -> np.ndarray:
    """torch's fp64 -> bf16 for values known to be exactly representable."""
    t = torch.as_tensor(np.asarray(values, dtype=np.float64)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


# ------------------------------------------------------------ e4m3 table ---

def test_e4m3_all_256_codes_match_torch():
    ours = oracle.e4m3_table()
    theirs = torch_e4m3_decode(np.arange(256))
    nan_ours = np.isnan(ours)
    assert np.array_equal(nan_ours, np.isnan(theirs))
    assert np.array_equal(ours[~nan_ours], theirs[~nan_ours])
    assert np.array_equal(np.signbit(ours[~nan_ours]), np.signbit(theirs[~nan_ours]))


def test_e4m3_landmarks():
    t = oracle.e4m3_table()
    assert list(np.flatnonzero(np.isnan(t))) == [0x7F, 0xFF]
    assert np.nanmax(t) == 448.0 == torch.finfo(torch.float8_e4m3fn).max
    assert np.nanmin(t) == -448.0
    assert not np.isinf(t).any()
    assert t[0x38] == 1.0
    assert t[0x01] == 2.0 ** -9           # smallest subnormal
    assert t[0x07] == 7 * 2.0 ** -9       # largest subnormal
    assert t[0x08] == 2.0 ** -6           # smallest normal
    assert t[0x80] == 0.0 and math.copysign(1.0, t[0x80]) == -1.0
    # every finite value is a multiple of 2^-9 (the exactness argument)
    fin = t[~np.isnan(t)]
    assert np.all(fin * 2 ** 9 == np.round(fin * 2 ** 9))


def test_e4m3_golden_fixture():
    path = os.path.join(GOLDEN, "e4m3_landmarks.txt")
    t = oracle.e4m3_table()
    n = 0
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            code_s, val_s = line.split()
            code = int(code_s, 16)
            if val_s == "nan":
                assert math.isnan(t[code])
            else:
                v = float.fromhex(val_s) if val_s.startswith(("0x", "-0x")) else float(val_s)
                assert t[code] == v and math.copysign(1, t[code]) == math.copysign(1, v), hex(code)
            n += 1
    assert n >= 10


# ------------------------------------------------------------ bf16 RNE ------

def test_bf16_rne_matches_torch_on_fp32_values():
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 2 ** 32, size=400_000, dtype=np.uint64).astype(np.uint32)
    f32 = bits.view(np.float32)
    f32 = f32[~np.isnan(f32)]
    ours = oracle.bf16_rne(f32.astype(np.float64))
    theirs = torch.from_numpy(f32.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, theirs)


def test_bf16_rne_single_rounding_from_fp64():
    # Values whose fp64 -> fp32 -> bf16 path rounds twice and lands elsewhere.
    cases = [
        1 + 2 ** -8 + 2 ** -40,          # above the tie: up
        1 + 2 ** -8 - 2 ** -40,          # below the tie: down
        1 + 3 * 2 ** -8 - 2 ** -45,      # below the tie at an odd neighbour
        -(1 + 2 ** -8 + 2 ** -40),
        448 * 448 * 3 + 2 ** -30,
    ]
    for x in cases:
        assert int(oracle.bf16_rne(x)) == frac_to_bf16_bits(Fraction(x)), x
    assert int(oracle.bf16_rne(1 + 2 ** -8 + 2 ** -40)) == 0x3F81
    assert int(oracle.bf16_rne(1 + 2 ** -8)) == 0x3F80      # exact tie: to even
    assert int(oracle.bf16_rne(1 + 3 * 2 ** -8)) == 0x3F82  # exact tie: to even (up)


def test_bf16_rne_vs_exact_rational_random():
    rng = np.random.default_rng(2)
    mant = rng.random(3000) + 1.0
    expo = rng.integers(-140, 129, size=3000)
    sign = np.where(rng.random(3000) < 0.5, -1.0, 1.0)
    xs = sign * np.ldexp(mant, expo)
    ours = oracle.bf16_rne(xs)
    for x, o in zip(xs, ours):
        assert int(o) == frac_to_bf16_bits(Fraction(float(x))), x


def test_bf16_rne_specials():
    big = 2.0 ** 127 * (2 - 2 ** -8)           # exact tie above max bf16 -> inf
    assert int(oracle.bf16_rne(big)) == 0x7F80
    assert int(oracle.bf16_rne(2.0 ** 127 * (2 - 2 ** -7))) == 0x7F7F  # max bf16
    assert int(oracle.bf16_rne(-big)) == 0xFF80
    assert int(oracle.bf16_rne(float("inf"))) == 0x7F80
    assert int(oracle.bf16_rne(float("-inf"))) == 0xFF80
    assert int(oracle.bf16_rne(float("nan"))) & 0x7FFF > 0x7F80
    assert int(oracle.bf16_rne(2.0 ** -133)) == 0x0001           # min subnormal
    assert int(oracle.bf16_rne(2.0 ** -134)) == 0x0000           # tie -> even (0)
    assert int(oracle.bf16_rne(2.0 ** -134 * 1.0001)) == 0x0001
    assert int(oracle.bf16_rne(3 * 2.0 ** -134)) == 0x0002        # tie -> even (2)
    assert int(oracle.bf16_rne(-0.0)) == 0x8000
    assert int(oracle.bf16_rne(0.0)) == 0x0000
    assert oracle.bf16_to_f64(np.uint16(0x3F80)) == 1.0


# ------------------------------------------------------------ closed forms --

def test_identity_B():
    rng = np.random.default_rng(3)
    K = N = 64
    M = 48
    A = finite_codes(rng, (M, K))
    Bt = np.zeros((N, K), np.uint8)
    Bt[np.arange(N), np.arange(K)] = 0x38            # 1.0
    out, ref, _ = oracle.scaled_mm(A, Bt, [0.5], [3.0], 0)
    # <= 5 significant bits: exact in bf16; "+ 0.0" because an exact zero sum is +0
    expect = torch_e4m3_decode(A) * 1.5 + 0.0
    assert np.array_equal(ref, expect)
    assert np.array_equal(out, bf16_bits_of(expect))


def test_diagonal_B_rowwise():
    rng = np.random.default_rng(4)
    M, N = 40, 32
    K = N
    A = finite_codes(rng, (M, K), allow_subnormal=False)
    d = finite_codes(rng, (N,), allow_subnormal=False)
    Bt = np.zeros((N, K), np.uint8)
    Bt[np.arange(N), np.arange(K)] = d
    sa = np.ldexp(1.0, rng.integers(-6, 6, size=M)).astype(np.float32)
    sb = np.ldexp(1.0, rng.integers(-6, 6, size=N)).astype(np.float32)
    out, ref, absum = oracle.scaled_mm(A, Bt, sa, sb, 1)
    expect = torch_e4m3_decode(A) * torch_e4m3_decode(d)[None, :] * sa[:, None].astype(np.float64) \
        * sb[None, :].astype(np.float64) + 0.0
    assert np.array_equal(ref, expect)
    assert np.array_equal(absum, np.abs(expect))
    # a product of two 4-bit significands has <= 8 bits: exact in bf16
    assert np.array_equal(out, bf16_bits_of(expect))


@pytest.mark.parametrize("K", [16, 4096])
def test_all_ones(K):
    M, N = 8, 24
    A = np.full((M, K), 0x38, np.uint8)
    Bt = np.full((N, K), 0x38, np.uint8)
    out, ref, absum = oracle.scaled_mm(A, Bt, [2.0 ** -3], [2.0 ** -5], 0)
    assert np.all(ref == K * 2.0 ** -8)
    assert np.all(absum == K * 2.0 ** -8)
    assert np.all(out == bf16_bits_of([K * 2.0 ** -8])[0])
    out1, _, _ = oracle.scaled_mm(A, Bt, [1.0], [1.0], 0)
    assert np.all(out1 == bf16_bits_of([float(K)])[0])


def test_all_448_and_sign():
    K = 16
    A = np.full((3, K), 0x7E, np.uint8)          # +448
    Bt = np.full((5, K), 0xFE, np.uint8)         # -448
    out, ref, absum = oracle.scaled_mm(A, Bt, [1.0], [1.0], 0)
    assert np.all(ref == -K * 448.0 ** 2)
    assert np.all(absum == K * 448.0 ** 2)
    assert np.all(out == bf16_bits_of([-K * 448.0 ** 2])[0])


def test_bias_only_when_A_is_zero():
    rng = np.random.default_rng(5)
    M, N, K = 6, 20, 32
    A = np.zeros((M, K), np.uint8)
    Bt = finite_codes(rng, (N, K))
    bias = torch.randn(N, dtype=torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    out, _, _ = oracle.scaled_mm(A, Bt, [1.5], [2.0], 0, bias=bias)
    assert np.array_equal(out, np.broadcast_to(bias, (M, N)))


def test_rowwise_scales_hit_the_intended_rows_and_columns():
    M, N, K = 5, 7, 16
    A = np.full((M, K), 0x38, np.uint8)
    Bt = np.full((N, K), 0x38, np.uint8)
    sa = np.ones(M, np.float32)
    sb = np.ones(N, np.float32)
    sa[2] = 4.0
    sb[5] = 0.25
    out, ref, _ = oracle.scaled_mm(A, Bt, sa, sb, 1)
    expect = np.full((M, N), float(K))
    expect[2, :] *= 4.0
    expect[:, 5] *= 0.25
    assert np.array_equal(ref, expect)
    assert np.array_equal(out, bf16_bits_of(expect))


# ------------------------------------------------------------ brute force ---

@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("with_bias", [False, True])
@pytest.mark.parametrize("shape", [(1, 1, 1), (3, 5, 7), (8, 6, 16), (5, 8, 33)])
def test_brute_force_exact_rational(mode, with_bias, shape):
    M, N, K = shape
    rng = np.random.default_rng(hash((mode, with_bias, shape)) % 2 ** 32)
    A = finite_codes(rng, (M, K))
    Bt = finite_codes(rng, (N, K))
    if mode == 0:
        sa = np.array([rng.random() + 0.01], np.float32)
        sb = np.array([rng.random() * 3 + 0.01], np.float32)
    else:
        sa = (rng.random(M) + 0.01).astype(np.float32)
        sb = (rng.random(N) * 3 + 0.01).astype(np.float32)
    bias = None
    if with_bias:
        bias = torch.randn(N, dtype=torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    out, _, _ = oracle.scaled_mm(A, Bt, sa, sb, mode, bias=bias)
    expect = exact_scaled_mm(A, Bt, sa, sb, mode, bias)
    assert np.array_equal(out, expect)


def test_grid_selection_matches_full_output():
    rng = np.random.default_rng(6)
    M, N, K = 37, 29, 48
    A = finite_codes(rng, (M, K))
    Bt = finite_codes(rng, (N, K))
    sa = (rng.random(M) + 0.1).astype(np.float32)
    sb = (rng.random(N) + 0.1).astype(np.float32)
    bias = torch.randn(N, dtype=torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    full, fref, fabs_ = oracle.scaled_mm(A, Bt, sa, sb, 1, bias=bias)
    rows = np.array([0, 36, 5, 5, 17])
    cols = np.array([28, 0, 3])
    sub, sref, sabs = oracle.scaled_mm(A, Bt, sa, sb, 1, bias=bias, rows=rows, cols=cols)
    assert np.array_equal(sub, full[np.ix_(rows, cols)])
    assert np.array_equal(sref, fref[np.ix_(rows, cols)])
    assert np.array_equal(sabs, fabs_[np.ix_(rows, cols)])


# ------------------------------------------------------------ exactness -----

def test_fp64_dot_is_exact_on_the_2pow_minus18_grid():
    rng = np.random.default_rng(7)
    K = 16384
    A = finite_codes(rng, (2, K))
    Bt = finite_codes(rng, (3, K))
    A[1, :] = 0x7E
    Bt[2, :] = 0xFE
    _, ref, absum = oracle.scaled_mm(A, Bt, [1.0], [1.0], 0)
    ai = np.round(torch_e4m3_decode(A) * 2 ** 9).astype(np.int64)
    bi = np.round(torch_e4m3_decode(Bt) * 2 ** 9).astype(np.int64)
    for i in range(2):
        for j in range(3):
            exact = int(np.dot(ai[i], bi[j]))
            assert ref[i, j] == exact / 2 ** 18
            assert absum[i, j] == int(np.abs(ai[i] * bi[j]).sum()) / 2 ** 18


def test_nan_code_propagates():
    A = np.full((2, 16), 0x38, np.uint8)
    Bt = np.full((2, 16), 0x38, np.uint8)
    A[0, 3] = 0x7F
    out, _, _ = oracle.scaled_mm(A, Bt, [1.0], [1.0], 0)
    assert (int(out[0, 0]) & 0x7FFF) > 0x7F80 and (int(out[0, 1]) & 0x7FFF) > 0x7F80
    assert int(out[1, 0]) == 0x4180  # 16.0


# ------------------------------------------------------------ planted bugs --

def test_pins_catch_planted_mistakes():
    """Mistakes planted in calls to the oracle must fail the brute-force pin."""
    rng = np.random.default_rng(8)
    M, N, K = 4, 4, 16
    A = finite_codes(rng, (M, K), allow_subnormal=False)
    Bt = finite_codes(rng, (N, K), allow_subnormal=False)
    # scales small enough that the outputs are O(1), so the bias is visible
    sa = np.array([0.5, 1.0, 2.0, 4.0], np.float32) * np.float32(2.0 ** -9)
    sb = np.array([3.0, 0.25, 1.0, 8.0], np.float32) * np.float32(2.0 ** -9)
    bias = torch.randn(N, dtype=torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    truth = exact_scaled_mm(A, Bt, sa, sb, 1, bias)
    good, _, _ = oracle.scaled_mm(A, Bt, sa, sb, 1, bias=bias)
    assert np.array_equal(good, truth)
    planted = {
        "transposed operands": lambda: oracle.scaled_mm(Bt, A, sa, sb, 1, bias=bias)[0].T,
        "scales swapped": lambda: oracle.scaled_mm(A, Bt, sb, sa, 1, bias=bias)[0],
        "bias dropped": lambda: oracle.scaled_mm(A, Bt, sa, sb, 1)[0],
        "k index reversed on one side": lambda: oracle.scaled_mm(A[:, ::-1], Bt, sa, sb, 1, bias=bias)[0],
        "sign flipped": lambda: oracle.scaled_mm(A ^ 0x80, Bt, sa, sb, 1, bias=bias)[0],
        "last k dropped": lambda: oracle.scaled_mm(A[:, :-1], Bt[:, :-1], sa, sb, 1, bias=bias)[0],
    }
    for name, fn in planted.items():
        assert not np.array_equal(fn(), truth), name


# ------------------------------------------------ other dtypes (e5m2, fp16) --

def torch_e5m2_decode(codes) -> np.ndarray:
    t = torch.as_tensor(np.asarray(codes, dtype=np.uint8)).view(torch.float8_e5m2)
    return t.to(torch.float64).numpy()


def frac_round(x: Fraction, p: int, emin: int) -> Fraction:
    """Exact RNE of a rational to p significand bits, exponent floor emin."""
    if x == 0:
        return Fraction(0)
    sign = -1 if x < 0 else 1
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, emin)
    quantum = Fraction(2) ** (e - (p - 1))
    q = a / quantum
    n = q.numerator // q.denominator
    rem = q - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return sign * n * quantum


def frac_to_f16_bits(x: Fraction) -> int:
    v = frac_round(x, 11, -14)
    if abs(v) >= 65520:
        return (0x8000 if x < 0 else 0) | 0x7C00
    h = np.array([float(v)], dtype=np.float16)
    assert Fraction(float(h[0])) == v
    return int(h.view(np.uint16)[0]) | (0x8000 if (x < 0 and v == 0) else 0)


def test_e5m2_all_256_codes_match_torch():
    ours = oracle.e5m2_table()
    theirs = torch_e5m2_decode(np.arange(256))
    nan = np.isnan(ours)
    assert np.array_equal(nan, np.isnan(theirs))
    assert np.array_equal(ours[~nan], theirs[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(theirs[~nan]))


def test_e5m2_landmarks():
    t = oracle.e5m2_table()
    assert t[0x7B] == 57344.0 == torch.finfo(torch.float8_e5m2).max
    assert t[0x7C] == float("inf") and t[0xFC] == float("-inf")
    assert list(np.flatnonzero(np.isnan(t))) == [0x7D, 0x7E, 0x7F, 0xFD, 0xFE, 0xFF]
    assert t[0x3C] == 1.0
    assert t[0x01] == 2.0 ** -16 and t[0x04] == 2.0 ** -14
    fin = t[np.isfinite(t)]
    assert np.all(fin * 2 ** 16 == np.round(fin * 2 ** 16))


def test_f16_rne_matches_torch_on_fp32_values():
    rng = np.random.default_rng(11)
    bits = rng.integers(0, 2 ** 32, size=300_000, dtype=np.uint64).astype(np.uint32)
    f32 = bits.view(np.float32)
    f32 = f32[~np.isnan(f32)]
    ours = oracle.f16_rne(f32.astype(np.float64))
    theirs = torch.from_numpy(f32.copy()).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, theirs)


def test_f16_rne_vs_exact_rational_random_fp64():
    rng = np.random.default_rng(12)
    mant = rng.random(3000) + 1.0
    expo = rng.integers(-27, 17, size=3000)
    sign = np.where(rng.random(3000) < 0.5, -1.0, 1.0)
    xs = sign * np.ldexp(mant, expo)
    ours = oracle.f16_rne(xs)
    for x, o in zip(xs, ours):
        assert int(o) == frac_to_f16_bits(Fraction(float(x))), x


def test_f16_rne_specials():
    assert int(oracle.f16_rne(65504.0)) == 0x7BFF
    assert int(oracle.f16_rne(65519.99)) == 0x7BFF
    assert int(oracle.f16_rne(65520.0)) == 0x7C00          # tie above max -> inf
    assert int(oracle.f16_rne(-70000.0)) == 0xFC00
    assert int(oracle.f16_rne(2.0 ** -24)) == 0x0001        # min subnormal
    assert int(oracle.f16_rne(2.0 ** -25)) == 0x0000        # tie -> even (0)
    assert int(oracle.f16_rne(3 * 2.0 ** -25)) == 0x0002    # tie -> even (2)
    assert int(oracle.f16_rne(2.0 ** -14 * (1 - 2 ** -12))) == 0x0400   # rounds up into the normals
    assert int(oracle.f16_rne(1 + 2 ** -11)) == 0x3C00      # tie -> even
    assert int(oracle.f16_rne(1 + 2 ** -11 + 2 ** -40)) == 0x3C01   # single rounding from fp64
    assert int(oracle.f16_rne(-0.0)) == 0x8000


def exact_typed(A, Bt, at, bt, sa, sb, mode, bias_bits, out_type):
    dec = {0: torch_e4m3_decode, 1: torch_e5m2_decode}
    Ad, Bd = dec[at](A), dec[bt](Bt)
    M, K = Ad.shape
    N = Bd.shape[0]
    out = np.zeros((M, N), dtype=np.uint16)
    bv = None
    if bias_bits is not None:
        bv = oracle.out_to_f64(bias_bits, out_type)
    for i in range(M):
        for j in range(N):
            dot = sum((Fraction(float(Ad[i, k])) * Fraction(float(Bd[j, k])) for k in range(K)),
                      Fraction(0))
            S = Fraction(float(sa[0 if mode == 0 else i])) * Fraction(float(sb[0 if mode == 0 else j]))
            v = dot * S + (Fraction(float(bv[j])) if bv is not None else 0)
            out[i, j] = frac_to_bf16_bits(v) if out_type == 0 else frac_to_f16_bits(v)
    return out


def finite_e5m2(rng, shape):
    c = rng.integers(0, 256, size=shape, dtype=np.int64)
    c = np.where((c & 0x7C) == 0x7C, c & 0xF3, c)     # no inf / NaN exponent
    return c.astype(np.uint8)


@pytest.mark.parametrize("at,bt", [(1, 1), (0, 1), (1, 0)])
@pytest.mark.parametrize("out_type", [0, 1])
def test_brute_force_other_dtypes(at, bt, out_type):
    rng = np.random.default_rng(100 * at + 10 * bt + out_type)
    M, N, K = 4, 5, 9
    gen = {0: lambda s: finite_codes(rng, s), 1: lambda s: finite_e5m2(rng, s)}
    A, Bt = gen[at]((M, K)), gen[bt]((N, K))
    # scales keep fp16 results in range for e5m2 magnitudes
    sa = (rng.random(M) * 2 ** -12 + 2 ** -14).astype(np.float32)
    sb = (rng.random(N) * 2 ** -12 + 2 ** -14).astype(np.float32)
    bias = (torch.randn(N) * 0.1).to(torch.bfloat16 if out_type == 0 else torch.float16) \
        .view(torch.int16).numpy().view(np.uint16)
    out, _, _ = oracle.scaled_mm(A, Bt, sa, sb, 1, bias=bias, a_type=at, b_type=bt, out_type=out_type)
    assert np.array_equal(out, exact_typed(A, Bt, at, bt, sa, sb, 1, bias, out_type))


def test_fp16_output_bias_only():
    rng = np.random.default_rng(13)
    A = np.zeros((3, 16), np.uint8)
    Bt = finite_e5m2(rng, (7, 16))
    bias = (torch.randn(7) * 3).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    out, _, _ = oracle.scaled_mm(A, Bt, [2.0], [3.0], 0, bias=bias, b_type=1, out_type=1)
    assert np.array_equal(out, np.broadcast_to(bias, (3, 7)))
