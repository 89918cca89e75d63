"""Stray-write checks on the GPU: every output lives inside a larger buffer
filled with a byte pattern, and after a kernel variant has run, every byte
that is not an output element must still hold the pattern.

This stands in for a memory checker (which is not available here). It covers
the paths whose index arithmetic decides where stores land: TMA tensor stores
clipped at ragged edges, the plain-store paths for rows that are not 16-byte
aligned (odd N, an odd leading dimension, a misaligned base), the SWAP
kernels' column stores, the split-K and stream-K final stores, the fp32 and
e4m3 register stores, gaps between rows when the leading dimension exceeds N,
batched items back to back, and the host entry's copies into host memory.
The written elements are also compared with the oracle.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from fp8_scaled_gemm_gb300.inputs import OUT_DTYPES, make_inputs
from tests._parity import compare, out_bits, to_device

pytestmark = pytest.mark.gpu

TILE, SWAP, PAIR, SWAPK, SWAPPAIR = 1, 2, 3, 4, 5
PAD = 4096


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _pattern(n: int) -> torch.Tensor:
    i = torch.arange(n, dtype=torch.int64)
    return ((i * 131 + 7) & 0xFF).to(torch.uint8)


class Guarded:
    """A [rows, cols] output with row stride ld (elements) at byte offset
    PAD + misalign of a pattern-filled byte buffer."""

    def __init__(self, rows, cols, dtype, ld=None, misalign=0, device="cuda", batch=1):
        self.rows, self.cols, self.dtype = rows, cols, dtype
        self.ld = ld or cols
        self.esz = torch.empty(0, dtype=dtype).element_size()
        self.batch = batch
        self.off = PAD + misalign
        span = ((batch * rows - 1) * self.ld + cols) * self.esz
        self.total = self.off + span + PAD
        self.pattern = _pattern(self.total)
        self.buf = self.pattern.to(device) if device == "cuda" else self.pattern.clone().pin_memory()
        n_el = (batch * rows - 1) * self.ld + cols
        flat = self.buf[self.off:self.off + n_el * self.esz].view(dtype)
        if batch == 1:
            self.out = flat.as_strided((rows, cols), (self.ld, 1))
        else:
            self.out = flat.as_strided((batch, rows, cols), (rows * self.ld, self.ld, 1))

    def element_mask(self) -> np.ndarray:
        mask = np.zeros(self.total, dtype=bool)
        for r in range(self.batch * self.rows):
            a = self.off + r * self.ld * self.esz
            mask[a:a + self.cols * self.esz] = True
        return mask

    def stray_bytes(self) -> int:
        got = self.buf.cpu().numpy()
        keep = ~self.element_mask()
        return int((got[keep] != self.pattern.numpy()[keep]).sum())


def _run(M, N, K, mode, bias, variant, tile_n, split, out_dtype="bf16", ld=None, misalign=0, seed=80):
    import fp8_scaled_gemm_gb300 as fm
    inp = make_inputs(M, N, K, mode, seed, with_bias=bias, out_dtype=out_dtype)
    A, Bt, sa, sb, b = to_device(inp)
    g = Guarded(M, N, OUT_DTYPES[inp.out_type], ld=ld, misalign=misalign)
    if out_dtype == "bf16" and ld is None:
        fm.fp8_scaled_mm_config(A, Bt.t(), sa, sb, mode, bias=b, out=g.out, variant=variant, tile_n=tile_n,
                                split_k=split)
    else:
        fm.fp8_scaled_mm_ex(A, Bt.t(), sa, sb, mode, bias=b, out=g.out, variant=variant, tile_n=tile_n,
                            split_k=split)
    assert fm.fp8mm_device_status() == 0, fm.fp8mm_last_cuda_error()
    torch.cuda.synchronize()
    stray = g.stray_bytes()
    assert stray == 0, f"{stray} bytes outside the output changed"
    st = compare(out_bits(g.out), inp)
    assert st["violations"] == 0, st


# (variant, tile_n, split): every kernel family, with and without split-K
VARIANTS = [(0, 0, 0), (TILE, 128, 1), (TILE, 256, 1), (TILE, 128, 3), (SWAP, 16, 1), (SWAP, 64, 3),
            (SWAP, 128, 1), (PAIR, 128, 1), (PAIR, 256, 1), (PAIR, 256, 2), (SWAPK, 16, 2), (SWAPK, 64, 4),
            (SWAPK, 128, 8), (SWAPPAIR, 32, 0)]


@pytest.mark.parametrize("variant,tile_n,split", VARIANTS)
@pytest.mark.parametrize("N", [520, 523])          # TMA-store rows; odd N: plain stores
def test_no_stray_writes_ragged(variant, tile_n, split, N):
    _need_gpu()
    M = 300 if variant in (0, TILE, PAIR) else min(tile_n, 128) - 5
    _run(M, N, 400, 1, True, variant, tile_n, split)


@pytest.mark.parametrize("variant,tile_n,split", [(0, 0, 0), (TILE, 256, 1), (SWAP, 16, 1), (SWAPK, 16, 4)])
def test_no_stray_writes_single_row(variant, tile_n, split):
    _need_gpu()
    _run(1, 777, 512, 1, True, variant, tile_n, split)


@pytest.mark.parametrize("N,ld", [(520, 560), (520, 523), (523, 528)])   # 16-byte pitch and rows;
@pytest.mark.parametrize("variant,tile_n,split", [(TILE, 256, 1), (TILE, 128, 2), (PAIR, 256, 1),  # odd pitch;
                                                  (SWAP, 32, 1), (SWAPK, 64, 2)])                   # 16-byte pitch, odd rows
def test_no_stray_writes_between_rows(N, ld, variant, tile_n, split):
    """Leading dimension > N: the gap after every row stays untouched (a TMA
    store that ended a row of 523 elements in the middle of a 16-byte unit
    wrote the rest of that unit)."""
    _need_gpu()
    M = 300 if variant in (TILE, PAIR) else 50
    _run(M, N, 272, 1, True, variant, tile_n, split, out_dtype="fp16", ld=ld)


@pytest.mark.parametrize("variant,tile_n,split", [(TILE, 256, 1), (PAIR, 256, 1), (TILE, 128, 3)])
def test_no_stray_writes_misaligned_base(variant, tile_n, split):
    """A 4-byte aligned (not 16-byte aligned) output takes the plain stores."""
    _need_gpu()
    _run(300, 520, 400, 0, False, variant, tile_n, split, misalign=4)


@pytest.mark.parametrize("out_dtype", ["fp32", "e4m3"])
@pytest.mark.parametrize("variant,tile_n,split", [(TILE, 256, 1), (PAIR, 256, 1), (TILE, 128, 3),
                                                  (SWAP, 32, 1), (SWAPK, 16, 2), (SWAPPAIR, 64, 0)])
@pytest.mark.parametrize("ld_extra", [0, 5])
def test_no_stray_writes_fp32_and_e4m3(out_dtype, variant, tile_n, split, ld_extra):
    _need_gpu()
    M = 300 if variant in (TILE, PAIR) else 60
    _run(M, 523, 272, 1, True, variant, tile_n, split, out_dtype=out_dtype, ld=(523 + ld_extra) if ld_extra else None)


def test_no_stray_writes_stream_k():
    """Stream-K owners and contributors: fewer tiles than pairs (partials
    through L2) and more (one partial through the ring), odd N."""
    _need_gpu()
    _run(300, 523, 8192, 1, True, PAIR, 256, -1)
    _run(2304, 3075, 2048, 0, False, PAIR, 256, -1)


@pytest.mark.parametrize("N", [263, 264])   # plain stores; 16-byte rows (TMA stores of batch items)
def test_no_stray_writes_batched(N):
    _need_gpu()
    import fp8_scaled_gemm_gb300 as fm
    nb, M, K = 3, 200, 272
    items = [make_inputs(M, N, K, 1, 90 + i, with_bias=True) for i in range(nb)]
    for it in items:
        it.bias = items[0].bias
    A = torch.stack([it.a_q for it in items]).cuda()
    Bt = torch.stack([it.bt_q for it in items]).cuda()
    sa = torch.cat([it.scale_a for it in items]).cuda()
    sb = torch.cat([it.scale_b for it in items]).cuda()
    for variant, tile_n, split in ((TILE, 256, 1), (PAIR, 256, 1), (SWAP, 32, 1), (TILE, 128, 3), (SWAPK, 64, 2)):
        g = Guarded(M, N, torch.bfloat16, batch=nb)
        fm.fp8_scaled_bmm(A, Bt.transpose(1, 2), sa, sb, 1, bias=items[0].bias.cuda(), out=g.out,
                          variant=variant, tile_n=tile_n, split_k=split)
        assert fm.fp8mm_device_status() == 0
        torch.cuda.synchronize()
        assert g.stray_bytes() == 0, (variant, tile_n, split)
        for i, it in enumerate(items):
            assert compare(out_bits(g.out[i]), it)["violations"] == 0


def test_no_stray_writes_host_entry():
    """The host entry's device-to-host block copies land only on out's bytes."""
    _need_gpu()
    import fp8_scaled_gemm_gb300 as fm
    M, N, K = 2600, 2051, 512
    inp = make_inputs(M, N, K, 1, 95, with_bias=True)
    g = Guarded(M, N, torch.bfloat16, device="cpu")
    fm.fp8_scaled_mm_host(inp.a_q.pin_memory(), inp.bt_q.pin_memory().t(), inp.scale_a.pin_memory(),
                          inp.scale_b.pin_memory(), 1, bias=inp.bias.pin_memory(), out=g.out)
    got = g.buf.numpy()
    keep = ~g.element_mask()
    assert int((got[keep] != g.pattern.numpy()[keep]).sum()) == 0
    assert compare(out_bits(g.out), inp)["violations"] == 0
