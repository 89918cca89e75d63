"""Pins for the oracle's quantisation step (bf16 -> fp8 codes + fp32 scales).

The recipe is that of the gist "matmul_fp8.py", `get_scale` and
`benchmark()`: amax over the tensor or each row, scale = amax / qmax,
codes = fp8(clamp(x / scale, -qmax, qmax)), in fp32. The oracle is pinned to:

- exact rational round-to-nearest-even at every midpoint between adjacent
  fp8 values (and one fp32 ulp either side), written here from the format's
  definition with fractions.Fraction;
- PyTorch's own CPU conversion fp32 -> float8_e4m3fn / float8_e5m2 and its
  CPU fp32 division (an independent implementation of the same recipe);
- invariants: round trip of every finite code, the amax element maps to
  +-qmax, the reconstruction error bound, and the degenerate rows (zeros,
  NaN, inf).
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

E4M3_MAX, E5M2_MAX = 448.0, 57344.0


# ------------------------------------------------- independent references ---

def exact_rne_code(v: Fraction, q_type: int) -> int:
    """fp8 code of the rational v, round to nearest even, |v| <= qmax."""
    mbits, bias, min_exp = (3, 7, -6) if q_type == oracle.E4M3 else (2, 15, -14)
    sign = 0x80 if v < 0 else 0
    a = abs(v)
    if a == 0:
        return sign
    e = min_exp
    while a >= Fraction(2) ** (e + 1):
        e += 1
    quantum = Fraction(2) ** (e - mbits)            # spacing in [2^e, 2^(e+1)) or subnormals
    n = a / quantum
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    if fl == 2 ** (mbits + 1):                      # carried into the next binade
        fl //= 2
        e += 1
    if fl < 2 ** mbits:                             # subnormal
        assert e == min_exp
        return sign | fl
    return sign | ((e + bias) << mbits) | (fl - 2 ** mbits)


def torch_codes(v32: np.ndarray, q_type: int) -> np.ndarray:
    dt = torch.float8_e4m3fn if q_type == oracle.E4M3 else torch.float8_e5m2
    return torch.from_numpy(np.ascontiguousarray(v32, dtype=np.float32)).to(dt).view(torch.uint8).numpy()


def torch_recipe(x_bits: np.ndarray, mode: int, q_type: int):
    """The recipe in PyTorch CPU ops, as the gist writes it."""
    x = torch.from_numpy(x_bits.view(np.int16).copy()).view(torch.bfloat16)
    dt = torch.float8_e4m3fn if q_type == oracle.E4M3 else torch.float8_e5m2
    qmax = torch.finfo(dt).max
    if mode == 0:
        amax = x.abs().max().to(torch.float32).view(1, 1)
    else:
        amax = x.abs().amax(dim=1, keepdim=True).to(torch.float32)
    scale = amax / qmax
    codes = (x / scale).clamp(-qmax, qmax).to(dt).view(torch.uint8).numpy()
    return codes, scale.reshape(-1).numpy()


def fp8_values(q_type: int) -> np.ndarray:
    table = oracle.e4m3_table() if q_type == oracle.E4M3 else oracle.e5m2_table()
    return table


def finite_codes(q_type: int):
    vals = fp8_values(q_type)
    return [c for c in range(256) if np.isfinite(vals[c])]


def bf16_of(values) -> np.ndarray:
    return oracle.bf16_rne(np.asarray(values, dtype=np.float64))


# ------------------------------------------------------------- encoders ---

@pytest.mark.parametrize("q_type", [oracle.E4M3, oracle.E5M2])
def test_encode_round_trips_every_finite_code(q_type):
    vals = fp8_values(q_type)
    codes = np.array(finite_codes(q_type), dtype=np.int64)
    got = oracle.encode(vals[codes].astype(np.float32), q_type)
    assert np.array_equal(got.astype(np.int64), codes)


@pytest.mark.parametrize("q_type", [oracle.E4M3, oracle.E5M2])
def test_encode_matches_exact_rounding_at_every_midpoint(q_type):
    vals = fp8_values(q_type)
    qmax = E4M3_MAX if q_type == oracle.E4M3 else E5M2_MAX
    pos = sorted({float(vals[c]) for c in finite_codes(q_type) if vals[c] >= 0})
    probes = []
    for lo, hi in zip(pos[:-1], pos[1:]):
        mid = np.float32((lo + hi) / 2)             # exact: few significant bits
        for v in (np.nextafter(mid, np.float32(-1)), mid, np.nextafter(mid, np.float32(1e9)),
                  np.float32(lo), np.float32(hi)):
            probes.extend([v, -v])
    probes = np.array(probes, dtype=np.float32)
    probes = probes[np.abs(probes) <= qmax]
    got = oracle.encode(probes, q_type)
    want = np.array([exact_rne_code(Fraction(float(v)), q_type) | (0x80 if np.signbit(v) else 0)
                     for v in probes], dtype=np.uint8)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("q_type", [oracle.E4M3, oracle.E5M2])
def test_encode_matches_torch_conversion(q_type):
    qmax = E4M3_MAX if q_type == oracle.E4M3 else E5M2_MAX
    rng = np.random.default_rng(7)
    v = np.concatenate([
        rng.uniform(-qmax, qmax, 20000),
        rng.standard_normal(20000) * rng.choice([1e-6, 1e-3, 0.1, 1.0, 10.0], 20000),
        np.ldexp(rng.uniform(1, 2, 4000), rng.integers(-30, 9, 4000)) * rng.choice([-1, 1], 4000),
        [0.0, -0.0, qmax, -qmax],
    ]).astype(np.float32)
    v = v[np.abs(v) <= qmax]
    assert np.array_equal(oracle.encode(v, q_type), torch_codes(v, q_type))


def test_encode_specials():
    for q_type in (oracle.E4M3, oracle.E5M2):
        assert oracle.encode([np.nan], q_type)[0] == 0x7F
        assert oracle.encode([-np.nan], q_type)[0] == 0x7F   # one NaN code
        assert oracle.encode([-0.0], q_type)[0] == 0x80
        assert oracle.encode([0.0], q_type)[0] == 0x00
    assert oracle.encode([np.inf], oracle.E5M2)[0] == 0x7C
    # smallest subnormals and the ties below them
    assert oracle.encode([2.0 ** -9, 2.0 ** -10, 1.5 * 2.0 ** -9], oracle.E4M3).tolist() == [1, 0, 2]
    assert oracle.encode([2.0 ** -16, 2.0 ** -17, 1.5 * 2.0 ** -16], oracle.E5M2).tolist() == [1, 0, 2]


def test_planted_rounding_mistakes_fail_the_midpoint_pin():
    # 1.6875 lies halfway between 1.625 (mantissa 5, odd) and 1.75 (mantissa 6,
    # even): round-to-nearest-even gives 1.75, truncation 1.625, and rounding
    # ties away from zero agrees only by luck of parity elsewhere.
    v = Fraction(27, 16)
    assert oracle.encode([float(v)], oracle.E4M3)[0] == exact_rne_code(v, oracle.E4M3) == 0x3E

    def truncating(x):
        e = int(np.floor(np.log2(x)))
        return 0x38 + (e << 3) + int(x / 2.0 ** (e - 3)) - 8

    def ties_away(x):
        e = int(np.floor(np.log2(x)))
        return 0x38 + (e << 3) + int(np.floor(x / 2.0 ** (e - 3) + 0.5)) - 8

    ties = [Fraction(17 + 2 * k, 16) for k in range(8)]      # every midpoint in [1, 2)
    want = [exact_rne_code(t, oracle.E4M3) for t in ties]
    assert oracle.encode([float(t) for t in ties], oracle.E4M3).tolist() == want
    assert [truncating(float(t)) for t in ties] != want
    assert [ties_away(float(t)) for t in ties] != want


# ------------------------------------------------------------- quantize ---

def random_bf16(R, C, seed, wide=False):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(R, C, generator=g, dtype=torch.float32)
    if wide:
        x = x * torch.exp2(torch.randint(-40, 40, (R, 1), generator=g).float())
        x = x * torch.exp2(torch.randint(-12, 1, (R, C), generator=g).float())
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("q_type", [oracle.E4M3, oracle.E5M2])
@pytest.mark.parametrize("wide", [False, True])
def test_quantize_matches_the_torch_recipe(mode, q_type, wide):
    x = random_bf16(97, 333, seed=3 + mode + 2 * q_type, wide=wide)
    q, s = oracle.quantize(x, mode, q_type)
    tq, ts = torch_recipe(x, mode, q_type)
    assert np.array_equal(s.view(np.uint32), ts.view(np.uint32))
    assert np.array_equal(q, tq)


def exhaustive_significands(amax_exps=(0,), with_neg=True):
    """Rows whose amax runs over all 128 bf16 significands (at each exponent
    given), each holding every bf16 value below its amax down to 2^-24 times it."""
    rows = []
    for e in amax_exps:
        for m in range(128):
            amax = (1 + m / 128) * 2.0 ** e
            vals = [amax]
            for d in range(0, 25):
                vals.extend((1 + k / 128) * 2.0 ** (e - d) for k in range(128))
            vals = [v for v in vals if v <= amax]
            vals = vals + [-v for v in vals] if with_neg else vals
            rows.append(vals)
    C = max(len(r) for r in rows)
    C = (C + 15) // 16 * 16
    out = np.zeros((len(rows), C), dtype=np.float64)
    for i, r in enumerate(rows):
        out[i, :len(r)] = r
    return bf16_of(out)


@pytest.mark.parametrize("q_type", [oracle.E4M3, oracle.E5M2])
def test_quantize_exhaustive_significands_match_torch(q_type):
    x = exhaustive_significands(amax_exps=(0, -100, -130, 120))
    q, s = oracle.quantize(x, 1, q_type)
    tq, ts = torch_recipe(x, 1, q_type)
    assert np.array_equal(s.view(np.uint32), ts.view(np.uint32))
    assert np.array_equal(q, tq)


@pytest.mark.parametrize("q_type", [oracle.E4M3, oracle.E5M2])
def test_quantize_invariants(q_type):
    qmax = E4M3_MAX if q_type == oracle.E4M3 else E5M2_MAX
    x = random_bf16(64, 512, seed=5)
    xf = oracle.bf16_to_f64(x)
    q, s = oracle.quantize(x, 1, q_type)
    vals = fp8_values(q_type)
    # the scale is amax / qmax in fp32, and the amax element maps to +-qmax
    amax = np.abs(xf).max(axis=1)
    assert np.array_equal(s, (amax.astype(np.float32) / np.float32(qmax)).astype(np.float32))
    j = np.abs(xf).argmax(axis=1)
    assert np.all(np.abs(vals[q[np.arange(64), j]]) == qmax)
    # reconstruction: |dec(q) s - x| <= half an fp8 spacing at |x / s| (times s), plus fp32 rounding
    v = xf / s[:, None].astype(np.float64)
    mb, sub = (3, 2.0 ** -9) if q_type == oracle.E4M3 else (2, 2.0 ** -16)
    spacing = np.maximum(2.0 ** (np.floor(np.log2(np.maximum(np.abs(v), 1e-30))) - mb), sub)
    err = np.abs(vals[q] - v)
    assert np.all(err <= spacing / 2 * (1 + 2.0 ** -20) + np.abs(v) * 2.0 ** -23)
    # per-tensor: one scale from the global amax
    q0, s0 = oracle.quantize(x, 0, q_type)
    assert s0.shape == (1,) and s0[0] == np.float32(np.abs(xf).max()) / np.float32(qmax)


def test_quantize_degenerate_rows():
    x = np.zeros((4, 32), dtype=np.float64)
    x[1, 3] = np.nan
    x[2, 5] = np.inf
    x[2, 6] = 3.0
    x[3, :] = -0.0
    xb = bf16_of(x)
    q, s = oracle.quantize(xb, 1, oracle.E4M3)
    assert s[0] == 0 and np.all(q[0] == 0)                 # zeros -> zero codes, zero scale
    assert np.isnan(s[1]) and np.all(q[1] == 0x7F)         # a NaN spreads through its row's scale
    assert np.isinf(s[2]) and q[2, 5] == 0x7F and q[2, 6] == 0 and q[2, 0] == 0   # inf/inf, 3/inf
    assert s[3] == 0 and np.all(q[3] == 0x80)              # -0 keeps its sign
    qt, st = oracle.quantize(xb, 0, oracle.E4M3)
    assert np.isnan(st[0]) and np.all(qt == 0x7F)


def test_quantize_rejects_bad_arguments():
    with pytest.raises(ValueError):
        oracle.quantize(np.zeros(8, dtype=np.uint16), 0)
    with pytest.raises(RuntimeError):
        oracle.quantize(np.zeros((2, 8), dtype=np.uint16), 2)
