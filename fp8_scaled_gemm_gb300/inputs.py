"""Seeded synthetic inputs for the FP8 scaled matrix multiply.

This module is shared by the CUDA path's tests and benchmark and by the
oracle's tests; it holds none of the matrix multiply's arithmetic, only the
input recipe the pages use to make FP8 operands from bf16 data:

  * ``a = randn(M, K)``, ``b = randn(K, N)`` in bf16 from one seeded generator
    (gist "matmul_fp8.py", ``benchmark()``: ``torch.manual_seed(42)``,
    ``init_dtype = torch.bfloat16``);
  * scale = amax / 448, per tensor (``|x|.max()``) or per row
    (``|x|.amax(dim=1)``), B's scale taken over ``b.t()`` so that it has one
    value per column of B (same page, ``get_scale`` and ``benchmark()``);
  * ``x_q = (x / scale).clamp(-448, 448).to(float8_e4m3fn)`` (same page);
  * B made column-major, i.e. stored as Bt[N, K] row-major (same page,
    ``b.to(dtype).t().contiguous().t()``);
  * the optional bias is ``randn(N) * 0.1`` in bf16, drawn from the same
    generator right after ``b`` (the pages fix no distribution for it), then
    held in the bias dtype of the output type: fp16 for an fp16 output, fp32
    for an fp32 output, bf16 for bf16 and e4m3fn outputs.

Generation runs on the CPU so the bytes depend only on (shape, seed, mode).
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import torch

E4M3_MAX = 448.0  # torch.finfo(torch.float8_e4m3fn).max
FP8 = {"e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}
OUT_TYPES = {"bf16": 0, "fp16": 1, "fp32": 2, "e4m3": 3}
OUT_DTYPES = {0: torch.bfloat16, 1: torch.float16, 2: torch.float32, 3: torch.float8_e4m3fn}
BIAS_DTYPES = {0: torch.bfloat16, 1: torch.float16, 2: torch.float32, 3: torch.bfloat16}


@dataclass
class ScaledMMInputs:
    M: int
    N: int
    K: int
    scale_mode: int                 # 0 per-tensor, 1 row-wise
    a_q: torch.Tensor               # float8_e4m3fn [M, K] row-major
    bt_q: torch.Tensor              # float8_e4m3fn [N, K] row-major (B column-major)
    scale_a: torch.Tensor           # float32 [1] or [M]
    scale_b: torch.Tensor           # float32 [1] or [N]
    bias: Optional[torch.Tensor]    # bfloat16 / float16 / float32 [N] or None
    a_type: int = 0                 # 0 e4m3fn, 1 e5m2
    b_type: int = 0
    out_type: int = 0               # 0 bf16, 1 fp16, 2 fp32, 3 e4m3fn

    # numpy views for the oracle (uint8 codes, float32 scales, uint16 bias bits)
    def a_u8(self):
        return self.a_q.view(torch.uint8).numpy()

    def bt_u8(self):
        return self.bt_q.view(torch.uint8).numpy()

    def sa_np(self):
        return self.scale_a.numpy()

    def sb_np(self):
        return self.scale_b.numpy()

    def bias_u16(self):
        """The bias bit patterns (uint16 for 16-bit bias dtypes, uint32 for fp32)."""
        if self.bias is None:
            return None
        if self.bias.dtype == torch.float32:
            return self.bias.view(torch.int32).numpy().view("uint32")
        return self.bias.view(torch.int16).numpy().view("uint16")

    @property
    def out_dtype(self) -> torch.dtype:
        return OUT_DTYPES[self.out_type]

    def oracle_types(self):
        """Keyword arguments of oracle.scaled_mm for this input set's types."""
        return {"a_type": self.a_type, "b_type": self.b_type, "out_type": self.out_type}

    @property
    def b_colmajor(self) -> torch.Tensor:
        """B[K, N] as the column-major view of ``bt_q``."""
        return self.bt_q.t()


def make_inputs(M: int, N: int, K: int, scale_mode: int, seed: int,
                with_bias: bool = False, a_dtype: str = "e4m3", b_dtype: str = "e4m3",
                out_dtype: str = "bf16") -> ScaledMMInputs:
    """The recipe above; ``a_dtype`` / ``b_dtype`` pick e4m3fn or e5m2 (scale
    = amax / finfo(dtype).max), ``out_dtype`` ("bf16", "fp16", "fp32",
    "e4m3") the output type, and with it the bias dtype."""
    if scale_mode not in (0, 1):
        raise ValueError("scale_mode must be 0 (per-tensor) or 1 (row-wise)")
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    a = torch.randn(M, K, dtype=torch.bfloat16, generator=g)
    b = torch.randn(K, N, dtype=torch.bfloat16, generator=g)
    bias = None
    if with_bias:
        bias = (torch.randn(N, dtype=torch.bfloat16, generator=g) * 0.1).contiguous()
        bias = bias.to(BIAS_DTYPES[OUT_TYPES[out_dtype]])
    ta, tb = FP8[a_dtype], FP8[b_dtype]
    qa, qb = torch.finfo(ta).max, torch.finfo(tb).max
    if scale_mode == 0:
        sa = a.abs().max().to(torch.float32).view(1, 1)
        sb = b.t().abs().max().to(torch.float32).view(1, 1)
    else:
        sa = a.abs().amax(dim=1, keepdim=True).to(torch.float32)           # [M, 1]
        sb = b.t().abs().amax(dim=1, keepdim=True).to(torch.float32)       # [N, 1]
        sb = sb.t().contiguous()                                           # [1, N]
    sa = sa / qa
    sb = sb / qb
    a_q = (a / sa).clamp(-qa, qa).to(ta)
    b_q = (b / sb).clamp(-qb, qb).to(tb)
    bt_q = b_q.t().contiguous()
    return ScaledMMInputs(
        M=M, N=N, K=K, scale_mode=scale_mode,
        a_q=a_q.contiguous(), bt_q=bt_q,
        scale_a=sa.reshape(-1).contiguous(), scale_b=sb.reshape(-1).contiguous(),
        bias=bias, a_type=0 if a_dtype == "e4m3" else 1, b_type=0 if b_dtype == "e4m3" else 1,
        out_type=OUT_TYPES[out_dtype])


def from_codes(A_u8, Bt_u8, scale_a, scale_b, scale_mode: int,
               bias_u16=None) -> ScaledMMInputs:
    """Wrap hand-made e4m3 codes (numpy uint8) as an input set."""
    import numpy as np
    A = torch.from_numpy(np.ascontiguousarray(A_u8, dtype=np.uint8)).view(torch.float8_e4m3fn)
    Bt = torch.from_numpy(np.ascontiguousarray(Bt_u8, dtype=np.uint8)).view(torch.float8_e4m3fn)
    sa = torch.as_tensor(np.asarray(scale_a, dtype=np.float32).reshape(-1)).contiguous()
    sb = torch.as_tensor(np.asarray(scale_b, dtype=np.float32).reshape(-1)).contiguous()
    bias = None
    if bias_u16 is not None:
        bias = torch.from_numpy(np.ascontiguousarray(bias_u16, dtype=np.uint16).view(np.int16)).view(torch.bfloat16)
    return ScaledMMInputs(M=A.shape[0], N=Bt.shape[0], K=A.shape[1], scale_mode=scale_mode,
                          a_q=A, bt_q=Bt, scale_a=sa, scale_b=sb, bias=bias)


# ------------------------------------------------ bf16 data to quantise ---
# Plain bf16 matrices for the quantisation step (no quantisation arithmetic
# here: the values are drawn or listed, then stored as bf16).

def bf16_matrix(R: int, C: int, seed: int, kind: str = "randn") -> torch.Tensor:
    """bf16 [R, C] on the CPU.

    ``randn``: the pages' operand data (``torch.randn`` in bf16).
    ``wide``: randn times a per-row power of two in [2^-40, 2^40] and a
    per-element power of two in [2^-12, 1], so rows differ in range and hold
    values far below their maximum.
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    if kind == "randn":
        return torch.randn(R, C, dtype=torch.bfloat16, generator=g)
    if kind == "wide":
        x = torch.randn(R, C, dtype=torch.float32, generator=g)
        x = x * torch.exp2(torch.randint(-40, 41, (R, 1), generator=g).float())
        x = x * torch.exp2(torch.randint(-12, 1, (R, C), generator=g).float())
        return x.to(torch.bfloat16)
    raise ValueError(f"unknown kind {kind!r}")


def bf16_significand_rows(amax_exps=(0,), depth: int = 25) -> torch.Tensor:
    """One row per (bf16 significand m, exponent e in amax_exps): the row's
    largest magnitude is (1 + m/128) 2^e, and it also holds every bf16 value
    (1 + k/128) 2^(e-d) below that, d = 0..depth-1, with both signs; rows are
    zero-padded to a common length that is a multiple of 16."""
    rows = []
    for e in amax_exps:
        for m in range(128):
            amax = (1 + m / 128) * 2.0 ** e
            vals = [amax] + [(1 + k / 128) * 2.0 ** (e - d) for d in range(depth) for k in range(128)]
            vals = [v for v in vals if v <= amax]
            rows.append(vals + [-v for v in vals])
    C = (max(len(r) for r in rows) + 15) // 16 * 16
    out = torch.zeros(len(rows), C, dtype=torch.float64)
    for i, r in enumerate(rows):
        out[i, :len(r)] = torch.tensor(r, dtype=torch.float64)
    return out.to(torch.float32).to(torch.bfloat16)


def bf16_special_rows(C: int = 64) -> torch.Tensor:
    """Rows for the degenerate cases: all +0; one NaN; +inf with finite
    values; all -0; -inf; bf16 subnormals only; values near the bf16
    maximum; values near the smallest normal; a randn row."""
    inf, nan = float("inf"), float("nan")
    x = torch.zeros(9, C, dtype=torch.float32)
    g = torch.Generator(device="cpu")
    g.manual_seed(1234)
    base = torch.randn(C, generator=g)
    x[1] = base
    x[1, C // 3] = nan
    x[2] = base
    x[2, 5] = inf
    x[3] = -0.0
    x[4] = base
    x[4, 7] = -inf
    x[5] = base * 2.0 ** -128          # bf16 subnormals
    x[6] = base.sign() * (3.0e38 - base.abs() * 1e37)
    x[7] = base * 2.0 ** -124
    x[8] = base
    return x.to(torch.bfloat16)
