"""GPU parity of the quantisation step (bf16 -> fp8 codes + fp32 scales)
through the C ABI, against the oracle: codes and scales bit for bit.

The codes are integers decided by fp32 arithmetic (one division and one
rounding per element), so both sides take the same fp32 steps and must agree
exactly; NaN scales compare as NaN.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from fp8_scaled_gemm_gb300.inputs import (bf16_matrix, bf16_significand_rows, bf16_special_rows,
                                          make_inputs)
from tests._parity import bf16_bits, compare

pytestmark = pytest.mark.gpu

DT = {0: torch.float8_e4m3fn, 1: torch.float8_e5m2}


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _bits(x: torch.Tensor) -> np.ndarray:
    return x.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _same_scales(got: np.ndarray, want: np.ndarray) -> bool:
    both_nan = np.isnan(got) & np.isnan(want)
    return bool(np.all(both_nan | (got.view(np.uint32) == want.view(np.uint32))))


def quantize_and_compare(x_cpu: torch.Tensor, mode: int, q_type: int):
    import fp8_scaled_gemm_gb300 as fm
    q, s = fm.fp8_quantize(x_cpu.cuda(), mode, DT[q_type])
    torch.cuda.synchronize()
    q_gpu = q.view(torch.uint8).cpu().numpy()
    s_gpu = s.cpu().numpy()
    q_ref, s_ref = oracle.quantize(_bits(x_cpu), mode, q_type)
    bad = np.argwhere(q_gpu != q_ref)
    assert _same_scales(s_gpu, s_ref), f"scales differ: {np.nonzero(s_gpu.view(np.uint32) != s_ref.view(np.uint32))}"
    assert bad.size == 0, (f"{len(bad)} codes differ; first {bad[:5].tolist()}: gpu "
                           f"{[int(q_gpu[tuple(i)]) for i in bad[:5]]} oracle {[int(q_ref[tuple(i)]) for i in bad[:5]]}")
    return q, s


# Row lengths that reach every team shape of the row-wise kernel (4, 8, 16,
# 32 lanes; 1, 2, 4, 8 warps; 1 to 16 groups per thread) and the two-pass
# kernel for rows longer than 32768.
ROW_LENGTHS = [8, 40, 64, 120, 256, 264, 512, 1000, 1024, 2048, 2056, 4096, 8192, 12288, 16384, 24576,
               32768, 32776, 65536]


@pytest.mark.parametrize("C", ROW_LENGTHS)
@pytest.mark.parametrize("mode", [0, 1])
def test_quantize_every_row_length(C, mode):
    _need_gpu()
    R = 37 if C >= 4096 else 301
    for q_type in (0, 1):
        quantize_and_compare(bf16_matrix(R, C, seed=C + mode, kind="wide"), mode, q_type)


@pytest.mark.parametrize("q_type", [0, 1])
@pytest.mark.parametrize("mode", [0, 1])
def test_quantize_every_reachable_significand_pair(q_type, mode):
    _need_gpu()
    # every bf16 row maximum (128 significands at 2^0, 2^-100, 2^-130 and
    # 2^120) against every bf16 value below it: all the (x, scale) pairs the
    # recipe can produce, up to powers of two, plus subnormal scales
    x = bf16_significand_rows((0, -100, -130, 120))
    quantize_and_compare(x, mode, q_type)


@pytest.mark.parametrize("q_type", [0, 1])
def test_quantize_edges_of_the_reciprocal_path(q_type):
    _need_gpu()
    # row maxima whose scales sit just inside and just outside the range the
    # reciprocal path takes ([2^-80, 2^100)), with values 60 binades below
    # the maximum, where that path's residual leaves the normal range
    x = bf16_significand_rows((-72, -71, -70, 107, 108), depth=60)
    quantize_and_compare(x, 1, q_type)


@pytest.mark.parametrize("q_type", [0, 1])
def test_quantize_degenerate_rows(q_type):
    _need_gpu()
    x = bf16_special_rows(64)
    q, s = quantize_and_compare(x, 1, q_type)
    s = s.cpu().numpy()
    assert s[0] == 0 and np.isnan(s[1]) and np.isinf(s[2]) and s[3] == 0 and np.isinf(s[4])
    # each degenerate row alone, per tensor
    for r in range(x.shape[0]):
        quantize_and_compare(x[r:r + 1].contiguous(), 0, q_type)


def test_quantize_many_rows_grid_stride():
    _need_gpu()
    # more rows than the grid has teams: 4-lane teams, 64 rows per CTA pass
    quantize_and_compare(bf16_matrix(700_000, 8, seed=3), 1, 0)
    # one-row-per-CTA teams with more rows than CTAs
    quantize_and_compare(bf16_matrix(10_000, 8192, seed=4), 1, 0)


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("q_type", [0, 1])
def test_quantize_full_size_operand(mode, q_type):
    _need_gpu()
    # the benchmark's operand: bf16 randn 8192 x 8192, compared in full
    quantize_and_compare(bf16_matrix(8192, 8192, seed=42), mode, q_type)


def test_per_tensor_back_to_back_calls_reuse_the_scratch():
    _need_gpu()
    import fp8_scaled_gemm_gb300 as fm
    xs = [bf16_matrix(999, 1024, seed=s, kind="wide") for s in range(4)]
    dev = [x.cuda() for x in xs]
    outs = [fm.fp8_quantize(d, 0) for d in dev]     # queued back to back on one stream
    torch.cuda.synchronize()
    for x, (q, s) in zip(xs, outs):
        q_ref, s_ref = oracle.quantize(_bits(x), 0, 0)
        assert np.array_equal(q.view(torch.uint8).cpu().numpy(), q_ref)
        assert _same_scales(s.cpu().numpy(), s_ref)


def test_quantize_matches_the_input_recipe_of_the_benchmark():
    _need_gpu()
    import fp8_scaled_gemm_gb300 as fm
    # the GEMM tests' operands come from the same recipe in PyTorch CPU ops
    inp = make_inputs(300, 520, 400, 1, seed=5)
    g = torch.Generator().manual_seed(5)
    a = torch.randn(300, 400, dtype=torch.bfloat16, generator=g)
    b = torch.randn(400, 520, dtype=torch.bfloat16, generator=g)
    qa, sa = fm.fp8_quantize(a.cuda(), 1)
    qb, sb = fm.fp8_quantize(b.t().contiguous().cuda(), 1)
    assert torch.equal(qa.cpu().view(torch.uint8), inp.a_q.view(torch.uint8))
    assert torch.equal(qb.cpu().view(torch.uint8), inp.bt_q.view(torch.uint8))
    assert torch.equal(sa.cpu(), inp.scale_a) and torch.equal(sb.cpu(), inp.scale_b)


# ------------------------------------------------- bf16 -> GEMM, end to end ---

def _bf16_path(M, N, K, mode, seed, bias, a_dtype=torch.float8_e4m3fn, b_dtype=torch.float8_e4m3fn,
               out_dtype=torch.bfloat16, sample=False):
    import fp8_scaled_gemm_gb300 as fm
    from fp8_scaled_gemm_gb300.inputs import from_codes
    from tests._parity import sample_indices
    a = bf16_matrix(M, K, seed)
    bt = bf16_matrix(N, K, seed + 1)
    bias_t = None
    if bias:
        bias_t = (bf16_matrix(1, N, seed + 2).reshape(-1) * 0.1).to(out_dtype)
    out, a_q, b_q, s_a, s_b = fm.fp8_scaled_mm_bf16(
        a.cuda(), bt.cuda().t(), mode, bias=None if bias_t is None else bias_t.cuda(),
        out_dtype=out_dtype, a_dtype=a_dtype, b_dtype=b_dtype, return_quantized=True)
    assert fm.fp8mm_device_status() == 0
    at, bt_type = {torch.float8_e4m3fn: 0, torch.float8_e5m2: 1}[a_dtype], \
        {torch.float8_e4m3fn: 0, torch.float8_e5m2: 1}[b_dtype]
    qa_ref, sa_ref = oracle.quantize(_bits(a), mode, at)
    qb_ref, sb_ref = oracle.quantize(_bits(bt), mode, bt_type)
    assert np.array_equal(a_q.view(torch.uint8).cpu().numpy(), qa_ref)
    assert np.array_equal(b_q.t().contiguous().view(torch.uint8).cpu().numpy(), qb_ref)
    assert _same_scales(s_a.cpu().numpy(), sa_ref) and _same_scales(s_b.cpu().numpy(), sb_ref)
    inp = from_codes(qa_ref, qb_ref, sa_ref, sb_ref, mode,
                     None if bias_t is None else _bits(bias_t))
    inp.a_type, inp.b_type = at, bt_type
    inp.out_type = 0 if out_dtype == torch.bfloat16 else 1
    bits = bf16_bits(out)
    rows = cols = None
    if sample:
        rows = sample_indices(M, 128, 32, seed + 3)
        cols = sample_indices(N, 128, 32, seed + 4)
        bits = bits[np.ix_(rows, cols)]
    stats = compare(bits, inp, rows, cols)
    assert stats["violations"] == 0, stats


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("shape", [(300, 520, 400), (1, 4096, 1024), (16, 14336, 4096), (129, 257, 16)])
def test_bf16_path_small(mode, shape):
    _need_gpu()
    _bf16_path(*shape, mode, seed=31, bias=(mode == 1))


def test_bf16_path_other_types():
    _need_gpu()
    _bf16_path(300, 520, 400, 1, 33, True, a_dtype=torch.float8_e5m2, out_dtype=torch.float16)
    _bf16_path(300, 520, 400, 0, 34, False, b_dtype=torch.float8_e5m2)


@pytest.mark.parametrize("mode", [0, 1])
def test_bf16_path_full_size_sampled(mode):
    _need_gpu()
    _bf16_path(8192, 8192, 8192, mode, seed=42, bias=False, sample=True)


# ------------------------------------------- per-tensor amax placement ---
# The per-tensor amax is a reduction over every CTA's share of the tensor and
# the scale reaches every element: the extreme value placed at the start, in
# the middle and in the last group must decide the scale, and every code must
# still match the oracle.

@pytest.mark.parametrize("where", ["first", "middle", "last"])
def test_per_tensor_amax_from_anywhere(where):
    _need_gpu()
    R, C = 8192, 4104
    x = bf16_matrix(R, C, seed=71)
    n = R * C
    pos = {"first": 3, "middle": n // 2 + 11, "last": n - 1}[where]
    x.view(-1)[pos] = -1000.0
    _, s = quantize_and_compare(x, 0, 0)
    assert float(s[0]) == float(np.float32(1000.0) / np.float32(448.0))


@pytest.mark.parametrize("where", ["first", "middle", "last"])
def test_per_tensor_nan_anywhere(where):
    _need_gpu()
    R, C = 8192, 4104
    x = bf16_matrix(R, C, seed=72)
    n = R * C
    pos = {"first": 0, "middle": n // 3, "last": n - 2}[where]
    x.view(-1)[pos] = float("nan")
    _, s = quantize_and_compare(x, 0, 1)
    assert np.isnan(s.cpu().numpy()[0])


def test_per_tensor_zero_and_odd_shapes():
    _need_gpu()
    # all +-0: zero scale, codes of +-0
    x = torch.zeros(2048, 1024, dtype=torch.bfloat16)
    x.view(-1)[1::3] = -0.0
    _, s = quantize_and_compare(x, 0, 0)
    assert float(s[0]) == 0.0
    quantize_and_compare(bf16_matrix(1, 1 << 20, seed=73, kind="wide"), 0, 0)
    quantize_and_compare(bf16_matrix(4001, 264, seed=74, kind="wide"), 0, 1)


def test_per_tensor_back_to_back_large_calls():
    _need_gpu()
    import fp8_scaled_gemm_gb300 as fm
    xs = [bf16_matrix(2048 + 8 * s, 1032, seed=80 + s, kind="wide") for s in range(5)]
    dev = [x.cuda() for x in xs]
    outs = [fm.fp8_quantize(d, 0, DT[s % 2]) for s, d in enumerate(dev)]   # queued on one stream
    torch.cuda.synchronize()
    assert fm.fp8mm_device_status() == 0
    for s, (x, (q, sc)) in enumerate(zip(xs, outs)):
        q_ref, s_ref = oracle.quantize(_bits(x), 0, s % 2)
        assert np.array_equal(q.view(torch.uint8).cpu().numpy(), q_ref)
        assert _same_scales(sc.cpu().numpy(), s_ref)


# ------------------------------------ per-tensor, one-launch partition ---
# The one-launch per-tensor kernel gives each CTA a contiguous run of 16-byte
# groups (8 bf16): run b is [total * b / grid, total * (b + 1) / grid) with
# grid = min(#SMs, ceil(total / 4096)). A CTA holds the first 12288 groups of
# its run in shared memory; when at least 8192 groups are left, the next
# 16384 go to tensor memory; it streams the rest. The extreme value is placed
# on both sides of those seams.

def _seams(total: int, sms: int):
    grid = max(1, min(sms, -(-total // 4096)))
    out = []
    for b in (0, grid // 2, grid - 1):
        g0, g1 = total * b // grid, total * (b + 1) // grid
        stash_end = g0 + min(g1 - g0, 12288)
        out += [g0, stash_end - 1, min(stash_end, g1 - 1), g1 - 1]
        if g1 - stash_end >= 8192:
            tm_end = min(g1, stash_end + 16384)
            out += [tm_end - 1, min(tm_end, g1 - 1)]
    return sorted(set(out))


@pytest.mark.parametrize("R,C", [(8192, 8192), (3000, 1000)])
def test_per_tensor_amax_on_run_seams(R, C):
    _need_gpu()
    import fp8_scaled_gemm_gb300 as fm
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    base = bf16_matrix(R, C, seed=75)
    dev = base.cuda()
    for k, grp in enumerate(_seams(R * C // 8, sms)):
        pos = grp * 8 + (k % 8)
        x = dev.clone()
        x.view(-1)[pos] = -600.0 - 4 * k          # bf16 steps are 4 apart here
        q, s = fm.fp8_quantize(x, 0)
        want = np.float32(600.0 + 4 * k) / np.float32(448.0)
        assert float(s.cpu()[0]) == float(want), (grp, pos)
        if k == 0:
            q_ref, s_ref = oracle.quantize(_bits(x.cpu()), 0, 0)
            assert np.array_equal(q.view(torch.uint8).cpu().numpy(), q_ref)


def test_per_tensor_larger_than_l2():
    _need_gpu()
    # 256 MB of bf16: more than the shared-memory runs and the L2 hold together
    quantize_and_compare(bf16_matrix(16384, 8192, seed=76), 0, 0)


def test_per_tensor_grid_sizes_alternate():
    _need_gpu()
    import fp8_scaled_gemm_gb300 as fm
    # one-CTA, partial and full grids queued back to back: the grid barrier's
    # counter and generation words must be left right for every grid size
    shapes = [(64, 8), (4096, 4096), (16, 1024), (1000, 136), (8192, 1024), (1, 8)]
    xs = [bf16_matrix(r, c, seed=90 + i, kind="wide") for i, (r, c) in enumerate(shapes)]
    outs = [fm.fp8_quantize(x.cuda(), 0, DT[i % 2]) for i, x in enumerate(xs)]
    torch.cuda.synchronize()
    assert fm.fp8mm_device_status() == 0
    for i, (x, (q, sc)) in enumerate(zip(xs, outs)):
        q_ref, s_ref = oracle.quantize(_bits(x), 0, i % 2)
        assert np.array_equal(q.view(torch.uint8).cpu().numpy(), q_ref), shapes[i]
        assert _same_scales(sc.cpu().numpy(), s_ref), shapes[i]


@pytest.mark.parametrize("R,C", [(8192, 4104), (3000, 1000), (1, 8)])
def test_per_tensor_two_launch_form(R, C):
    """The fallback for devices that cannot hold the one-launch grid at once
    (an amax kernel, then a convert kernel), forced by the test hook."""
    _need_gpu()
    import fp8_scaled_gemm_gb300 as fm
    fm.fp8mm_debug_quant(1)
    try:
        quantize_and_compare(bf16_matrix(R, C, seed=77, kind="wide"), 0, 1)
        quantize_and_compare(bf16_matrix(R, C, seed=78), 0, 0)
    finally:
        fm.fp8mm_debug_quant(0)
