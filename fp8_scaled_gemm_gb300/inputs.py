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
    generator right after ``b`` (the pages fix no distribution for it).

Generation runs on the CPU so the bytes depend only on (shape, seed, mode).
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import torch

E4M3_MAX = 448.0  # torch.finfo(torch.float8_e4m3fn).max
FP8 = {"e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}


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
    bias: Optional[torch.Tensor]    # bfloat16 / float16 [N] or None
    a_type: int = 0                 # 0 e4m3fn, 1 e5m2
    b_type: int = 0
    out_type: int = 0               # 0 bf16, 1 fp16

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
        if self.bias is None:
            return None
        return self.bias.view(torch.int16).numpy().view("uint16")

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
    = amax / finfo(dtype).max), ``out_dtype`` the bias dtype (bf16 or fp16)."""
    if scale_mode not in (0, 1):
        raise ValueError("scale_mode must be 0 (per-tensor) or 1 (row-wise)")
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    a = torch.randn(M, K, dtype=torch.bfloat16, generator=g)
    b = torch.randn(K, N, dtype=torch.bfloat16, generator=g)
    bias = None
    if with_bias:
        bias = (torch.randn(N, dtype=torch.bfloat16, generator=g) * 0.1).contiguous()
        if out_dtype == "fp16":
            bias = bias.to(torch.float16)
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
        out_type=0 if out_dtype == "bf16" else 1)


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
