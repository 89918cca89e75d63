"""Pins for ``oracle.tolerance`` and for the ``absum`` term it takes (no GPU).

The parity bound every GPU test applies is

    |gpu - ref| <= 2^-7 |ref| + 2^-20 * S_ij * sum_k |a_ik b_kj|      (bf16 out)
    |gpu - ref| <= 2^-10 |ref| + 2^-20 * S_ij * sum_k |a_ik b_kj| + 2^-24   (fp16 out)

with ``ref`` the rounded oracle value. The bf16 form is the one the project
fixes for the FP8 scaled matmul (one unit in the last place of the output for
a rounding boundary crossed by the fp32 sums, plus the fp32 accumulation
error near cancellation); the fp16 form is its reading for an fp16 output
(fp16 keeps 10 fraction bits instead of 7; 2^-24 is the spacing of fp16's
subnormals, which a relative term cannot cover near zero).

What pins it, other than retyping the formula:
  * literals worked out by hand, per term and per output type;
  * a property of the output formats, checked on every normal bf16 value and
    every fp16 value from 2^-4 to the largest finite one, with ``absum = 0``: the next representable value
    above and below ``ref`` is admitted, and values two steps above or three
    steps below are not (the relative term is at least one unit in the last
    place and under two);
  * a hand-worked ``absum`` = S * sum |a b| on named e4m3 codes, per-tensor
    and row-wise (a dropped S_ij, a signed sum or a missing factor fails);
  * ``tests/_parity.compare`` on an input whose bound is exactly one bf16
    step: the value at the bound passes, one step beyond it fails;
  * planted slips in a copy of the bound (2^-8, 2^-17, the fp16 branch for
    bf16, S_ij dropped from absum) fail these pins.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from fp8_scaled_gemm_gb300.inputs import from_codes


def _bits(values, dtype) -> np.ndarray:
    """Bit patterns of values that are exact in ``dtype`` (torch conversion)."""
    t = torch.as_tensor(np.asarray(values, dtype=np.float64)).to(dtype)
    return t.view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------- hand-worked literals ---

@pytest.mark.parametrize("ref,absum,want", [
    (1.0, 0.0, 0.0078125),                   # 2^-7 * 1
    (0.0, 1048576.0, 1.0),                   # 2^-20 * 2^20
    (-3.0, 0.0, 0.0234375),                  # 2^-7 * |-3| = 3/128
    (1.0, 3145728.0, 3.0078125),             # 2^-7 + 2^-20 * 3 * 2^20
    (448.0, 0.0, 3.5),                       # 448 / 128
    (-0.0, 0.0, 0.0),                        # exact zero admits nothing
])
def test_bf16_bound_literals(ref, absum, want):
    got = oracle.tolerance(_bits([ref], torch.bfloat16), np.array([absum]), oracle.BF16)
    assert got.dtype == np.float64
    assert got[0] == want


@pytest.mark.parametrize("ref,absum,want", [
    (1.0, 0.0, 0.000976622104644775390625),  # 2^-10 + 2^-24
    (0.0, 0.0, 5.9604644775390625e-08),      # 2^-24: one fp16 subnormal step
    (-2.0, 1048576.0, 1.001953184604644775390625),   # 2 * 2^-10 + 1 + 2^-24
    (65504.0, 0.0, 63.96875005960464477539),          # 65504 / 1024 + 2^-24
])
def test_fp16_bound_literals(ref, absum, want):
    got = oracle.tolerance(_bits([ref], torch.float16), np.array([absum]), oracle.F16)
    assert got[0] == pytest.approx(want, rel=0, abs=1e-20)


# ------------------------------------------ format property (exhaustive) ---

_FMT = {"bf16": oracle.BF16, "fp16": oracle.F16, "fp32": oracle.F32, "e4m3": oracle.E4M3_OUT}


def _neighbours(bits: np.ndarray, fmt: str, step: int) -> np.ndarray:
    """Value ``step`` representable values away from each pattern (the sign
    bit is the top bit, so +step moves away from zero on either sign)."""
    return (bits.astype(np.int64) + step).astype(bits.dtype)


def _check_ulp_property(fmt: str, bits: np.ndarray, tol_fn=oracle.tolerance):
    """absum = 0: +1 and -1 steps admitted, +2 and -3 steps refused."""
    out_type = _FMT[fmt]

    def dec(b):
        return oracle.out_to_f64(b, out_type)
    ref = dec(bits)
    tol = tol_fn(bits, np.zeros(bits.shape), out_type)
    for step, admitted in ((1, True), (-1, True), (2, False), (-3, False)):
        nb = _neighbours(bits, fmt, step)
        v = dec(nb)
        ok = np.isfinite(v)
        inside = np.abs(v[ok] - ref[ok]) <= tol[ok]
        if admitted:
            assert inside.all(), (fmt, step, int((~inside).sum()))
        else:
            assert not inside.any(), (fmt, step, int(inside.sum()))


def _positive_normals(fmt: str) -> np.ndarray:
    # bf16: exponent field 1..254 (0x0080 .. 0x7F7F); three steps below the
    # smallest normal stay in the subnormals, so start three steps higher.
    # fp16: from 2^-4 (0x2C00) to the largest finite value (0x7BFF); below
    # 2^-4 the 2^-24 term is no longer small against two steps of the format
    # (it is pinned by the literals above instead).
    lo, hi = (0x0083, 0x7F7F) if fmt == "bf16" else (0x2C00, 0x7BFF)
    return np.arange(lo, hi + 1, dtype=np.uint16)


@pytest.mark.parametrize("fmt", ["bf16", "fp16"])
def test_bound_admits_one_step_and_refuses_two_on_every_value(fmt):
    bits = _positive_normals(fmt)
    _check_ulp_property(fmt, bits)
    _check_ulp_property(fmt, bits | np.uint16(0x8000))  # negative values mirror it


def test_bound_one_step_property_fp32_and_e4m3_outputs():
    # e4m3: every code from 2^-2 (0x28) up; below it the 2^-9 term is no
    # longer small against two steps. fp32: a million normal values from
    # 2^-100 up (the 2^-149 term is negligible there).
    e4 = np.arange(0x28, 0x7F, dtype=np.uint8)
    _check_ulp_property("e4m3", e4)
    _check_ulp_property("e4m3", e4 | np.uint8(0x80))
    rng = np.random.default_rng(5)
    f32 = rng.integers(0x0D800000, 0x7F7FFFFD, size=1_000_000, dtype=np.int64).astype(np.uint32)
    _check_ulp_property("fp32", f32)
    _check_ulp_property("fp32", f32 | np.uint32(0x80000000))


@pytest.mark.parametrize("out_type,ref_bits,absum,want", [
    (oracle.F32, np.uint32(0x3F800000), 0.0, 2.0 ** -23 + 2.0 ** -149),      # ref 1.0
    (oracle.F32, np.uint32(0x00000000), 1048576.0, 1.0 + 2.0 ** -149),      # ref 0
    (oracle.E4M3_OUT, np.uint8(0x38), 0.0, 0.126953125),                   # ref 1.0: 1/8 + 1/512
    (oracle.E4M3_OUT, np.uint8(0xFE), 0.0, 56.001953125),                  # ref -448: 56 + 1/512
    (oracle.E4M3_OUT, np.uint8(0x00), 0.0, 0.001953125),                   # ref 0: 2^-9
])
def test_fp32_and_e4m3_bound_literals(out_type, ref_bits, absum, want):
    got = oracle.tolerance(np.array([ref_bits]), np.array([absum]), out_type)
    assert got[0] == want


# ----------------------------------------------------- absum, hand-worked ---

# e4m3 codes (sign | 4 exponent bits, bias 7 | 3 fraction bits):
#   0x38 = 1.0, 0xC0 = -2.0, 0x30 = 0.5, 0x7E = 448, 0x44 = 3.0, 0x48 = 4.0
_A = np.array([[0x38, 0xC0, 0x30, 0x7E]], dtype=np.uint8)          # [1, -2, 0.5, 448]
_BT = np.array([[0x44, 0x48, 0xC0, 0x38],                          # [3, 4, -2, 1]
                [0x38, 0x38, 0x38, 0x38]], dtype=np.uint8)         # [1, 1, 1, 1]


def test_absum_per_tensor_hand_worked():
    # row 0 . col 0: 3 - 8 - 1 + 448 = 442, sum |.| = 3 + 8 + 1 + 448 = 460
    # row 0 . col 1: 1 - 2 + 0.5 + 448 = 447.5, sum |.| = 451.5
    # S = 0.5 * 0.25 = 0.125
    _, ref64, absum = oracle.scaled_mm(_A, _BT, np.float32([0.5]), np.float32([0.25]), 0)
    assert ref64.tolist() == [[55.25, 55.9375]]
    assert absum.tolist() == [[57.5, 56.4375]]


def test_absum_rowwise_hand_worked():
    # S_00 = 2 * 0.125, S_01 = 2 * 8
    _, ref64, absum = oracle.scaled_mm(_A, _BT, np.float32([2.0]), np.float32([0.125, 8.0]), 1)
    assert ref64.tolist() == [[110.5, 7160.0]]
    assert absum.tolist() == [[115.0, 7224.0]]


# -------------------------------------- the comparison helper at the bound ---

def test_compare_passes_at_the_bound_and_fails_one_step_beyond():
    from tests._parity import compare

    # A = 0 gives absum = 0 exactly and ref = bias; bias 1.0 makes the bound
    # exactly 2^-7, one bf16 step above 1.0 and two steps below it.
    A = np.zeros((1, 16), np.uint8)
    Bt = np.full((2, 16), 0x38, np.uint8)
    bias = _bits([1.0, -1.0], torch.bfloat16)
    inp = from_codes(A, Bt, [1.0], [1.0], 0, bias_u16=bias)
    ref = np.array([[0x3F80, 0xBF80]], np.uint16)
    assert compare(ref, inp)["violations"] == 0
    at = np.array([[0x3F81, 0xBF7E]], np.uint16)       # 1 + 2^-7, -(1 - 2^-7): exactly at the bound
    assert compare(at, inp)["violations"] == 0
    beyond = np.array([[0x3F82, 0xBF7D]], np.uint16)   # one more step: outside
    assert compare(beyond, inp)["violations"] == 2
    nan = np.array([[0x7FC0, 0xBF80]], np.uint16)      # NaN never passes
    assert compare(nan, inp)["violations"] == 1


# --------------------------------------------------------- planted slips ---

def _planted(rel_bf16=2.0 ** -7, rel_f16=2.0 ** -10, abs_w=2.0 ** -20, f16_for_bf16=False):
    def tol(ref_bits, absum, out_type=oracle.BF16):
        ot = oracle.F16 if (f16_for_bf16 and out_type == oracle.BF16) else out_type
        ref = oracle.out_to_f64(ref_bits, out_type)
        if ot == oracle.BF16:
            return np.abs(ref) * rel_bf16 + np.asarray(absum) * abs_w
        return np.abs(ref) * rel_f16 + np.asarray(absum) * abs_w + 2.0 ** -24
    return tol


def test_pins_catch_planted_slips():
    def literal_ok(tol):
        return (tol(_bits([1.0], torch.bfloat16), np.array([0.0]))[0] == 0.0078125 and
                tol(_bits([0.0], torch.bfloat16), np.array([1048576.0]))[0] == 1.0)

    def property_ok(tol):
        try:
            _check_ulp_property("bf16", _positive_normals("bf16"), tol)
            return True
        except AssertionError:
            return False

    assert literal_ok(oracle.tolerance) and property_ok(oracle.tolerance)
    slips = {
        "2^-8 relative": _planted(rel_bf16=2.0 ** -8),
        "2^-6 relative": _planted(rel_bf16=2.0 ** -6),
        "2^-17 absolute": _planted(abs_w=2.0 ** -17),
        "fp16 branch for bf16": _planted(f16_for_bf16=True),
    }
    for name, tol in slips.items():
        assert not (literal_ok(tol) and property_ok(tol)), name
    # S_ij dropped from absum: the hand-worked absum is S * 460, not 460
    _, _, absum = oracle.scaled_mm(_A, _BT, np.float32([0.5]), np.float32([0.25]), 0)
    assert absum[0, 0] != 460.0 and absum[0, 0] == 0.125 * 460
