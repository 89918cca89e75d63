"""CPU oracle for the FP8 scaled matrix multiply.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package. The product library
(``fp8_scaled_gemm_gb300``) never imports it and shares no code with it.

The arithmetic lives in ``fp8mm_oracle.c`` (plain C99 + OpenMP, fp64); this
module only compiles it with gcc and marshals numpy arrays through ctypes.
What it computes, with its sources on the pages:

    out[i, j] = round( sum_k dec(A[i, k]) * dec(Bt[j, k]) * S_ij + bias[j] )

(dec: e4m3fn or e5m2 codes; round: fp64 -> bf16, fp16 or fp32, one RNE
step, or fp64 -> e4m3fn, one RNE step saturating at +-448)

with ``S_ij = s_a * s_b`` (per-tensor) or ``s_a[i] * s_b[j]`` (row-wise):
gist "matmul_fp8.py" (FP8 Matmul), ``matmul_fp8_kernel`` scale epilogue;
PyTorch PR #125204 "fp8 row-scaling kernel for scaled_mm", Summary (row-wise
scale lengths M and N, TN layout); PyTorch PR #142045, Summary (bias).

Every function here is pinned against values fixed by the pages or by
mathematics: the matmul, the decoders and the output rounding by
``tests/test_oracle_pins.py`` (closed forms, exact rational brute force,
torch's independent float8/bf16 conversions), the quantiser by
``tests/test_oracle_quant_pins.py``, and ``tolerance`` with its ``absum``
input by ``tests/test_oracle_tolerance_pins.py`` (hand-worked literals, the
one-step property of the output formats, planted slips). No function is
unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp8mm_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libfp8mm_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/libfp8mm_oracle.so`` with gcc."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    fresh = (os.path.exists(_LIB_PATH)
             and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC))
    if fresh and not force:
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c99", "-O2", "-fopenmp", "-fPIC", "-shared",
           "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        c_i64p = ctypes.POINTER(ctypes.c_int64)
        lib.oracle_e4m3_to_f64.restype = ctypes.c_double
        lib.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_table.restype = None
        lib.oracle_e4m3_table.argtypes = [ctypes.c_void_p]
        lib.oracle_f64_to_bf16_rne.restype = ctypes.c_uint16
        lib.oracle_f64_to_bf16_rne.argtypes = [ctypes.c_double]
        lib.oracle_f64_to_bf16_array.restype = None
        lib.oracle_f64_to_bf16_array.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64]
        lib.oracle_bf16_to_f64.restype = ctypes.c_double
        lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_max_threads.restype = ctypes.c_int
        lib.oracle_max_threads.argtypes = []
        lib.oracle_e5m2_table.restype = None
        lib.oracle_e5m2_table.argtypes = [ctypes.c_void_p]
        lib.oracle_f64_to_f16_array.restype = None
        lib.oracle_f64_to_f16_array.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64]
        lib.oracle_f16_to_f64.restype = ctypes.c_double
        lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_f64_to_f32_rne.restype = ctypes.c_uint32
        lib.oracle_f64_to_f32_rne.argtypes = [ctypes.c_double]
        lib.oracle_f64_to_e4m3_sat.restype = ctypes.c_uint8
        lib.oracle_f64_to_e4m3_sat.argtypes = [ctypes.c_double]
        lib.oracle_scaled_mm_typed.restype = ctypes.c_int
        lib.oracle_scaled_mm_typed.argtypes = [
            ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int,
            ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
            ctypes.c_void_p, ctypes.c_int,
            c_i64p, ctypes.c_int64, c_i64p, ctypes.c_int64,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_int,
        ]
        lib.oracle_encode_e4m3.restype = ctypes.c_uint8
        lib.oracle_encode_e4m3.argtypes = [ctypes.c_float]
        lib.oracle_encode_e5m2.restype = ctypes.c_uint8
        lib.oracle_encode_e5m2.argtypes = [ctypes.c_float]
        lib.oracle_quantize.restype = ctypes.c_int
        lib.oracle_quantize.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
        lib.oracle_scaled_mm.restype = ctypes.c_int
        lib.oracle_scaled_mm.argtypes = [
            ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
            ctypes.c_void_p,
            c_i64p, ctypes.c_int64, c_i64p, ctypes.c_int64,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_int,
        ]
        _lib = lib
        return lib


def e4m3_table() -> np.ndarray:
    """The 256 e4m3fn code values as fp64 (NaN at 0x7F and 0xFF)."""
    t = np.empty(256, dtype=np.float64)
    _load().oracle_e4m3_table(t.ctypes.data)
    return t


def e4m3_to_f64(code: int) -> float:
    return float(_load().oracle_e4m3_to_f64(int(code)))


def bf16_rne(x) -> np.ndarray:
    """fp64 values -> bf16 bit patterns (uint16), one round-to-nearest-even."""
    arr = np.asarray(x, dtype=np.float64)
    xs = np.ascontiguousarray(arr.reshape(-1))
    out = np.empty(xs.shape, dtype=np.uint16)
    _load().oracle_f64_to_bf16_array(xs.ctypes.data, out.ctypes.data, xs.size)
    return out.reshape(arr.shape)


E4M3, E5M2 = 0, 1
BF16, F16, F32, E4M3_OUT = 0, 1, 2, 3
# numpy container of each output type's bit patterns, and of its bias
OUT_BITS = {BF16: np.uint16, F16: np.uint16, F32: np.uint32, E4M3_OUT: np.uint8}
BIAS_BITS = {BF16: np.uint16, F16: np.uint16, F32: np.uint32, E4M3_OUT: np.uint16}


def e5m2_table() -> np.ndarray:
    """The 256 e5m2 code values as fp64 (+-inf at 0x7C / 0xFC, NaN at 0x7D-0x7F, 0xFD-0xFF)."""
    t = np.empty(256, dtype=np.float64)
    _load().oracle_e5m2_table(t.ctypes.data)
    return t


def f16_rne(x) -> np.ndarray:
    """fp64 values -> IEEE binary16 bit patterns (uint16), one round-to-nearest-even."""
    arr = np.asarray(x, dtype=np.float64)
    xs = np.ascontiguousarray(arr.reshape(-1))
    out = np.empty(xs.shape, dtype=np.uint16)
    _load().oracle_f64_to_f16_array(xs.ctypes.data, out.ctypes.data, xs.size)
    return out.reshape(arr.shape)


def f16_to_f64(bits) -> np.ndarray:
    """binary16 bit patterns (uint16) -> fp64 values."""
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def f32_rne(x) -> np.ndarray:
    """fp64 values -> IEEE binary32 bit patterns (uint32), one round-to-nearest-even."""
    lib = _load()
    v = np.asarray(x, dtype=np.float64)
    flat = v.reshape(-1)
    return np.fromiter((lib.oracle_f64_to_f32_rne(float(a)) for a in flat), dtype=np.uint32,
                       count=flat.size).reshape(v.shape)


def e4m3_sat(x) -> np.ndarray:
    """fp64 values -> e4m3fn codes of an e4m3 output: one round-to-nearest-even,
    saturating at +-448 (also for +-inf); NaN -> 0x7F."""
    lib = _load()
    v = np.asarray(x, dtype=np.float64)
    flat = v.reshape(-1)
    return np.fromiter((lib.oracle_f64_to_e4m3_sat(float(a)) for a in flat), dtype=np.uint8,
                       count=flat.size).reshape(v.shape)


def f32_to_f64(bits) -> np.ndarray:
    """binary32 bit patterns (uint32) -> fp64 values."""
    return np.asarray(bits, dtype=np.uint32).view(np.float32).astype(np.float64)


def out_to_f64(bits, out_type: int) -> np.ndarray:
    """Output bit patterns of ``out_type`` -> fp64 values."""
    if out_type == BF16:
        return bf16_to_f64(bits)
    if out_type == F16:
        return f16_to_f64(bits)
    if out_type == F32:
        return f32_to_f64(bits)
    return e4m3_table()[np.asarray(bits, dtype=np.uint8)]


def bf16_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> fp64 values."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def scaled_mm(A, Bt, scale_a, scale_b, scale_mode: int, bias=None,
              rows=None, cols=None, threads: int = 0,
              a_type: int = E4M3, b_type: int = E4M3, out_type: int = BF16):
    """Oracle output on the grid ``rows x cols`` (all rows / columns if None).

    A: uint8 [M, K] fp8 codes (a_type 0 e4m3fn, 1 e5m2); Bt: uint8 [N, K]
    codes (B column-major, b_type likewise); scale_a / scale_b: float32
    arrays of 1 value (scale_mode 0) or M / N values (scale_mode 1); bias:
    [N] bit patterns (``BIAS_BITS[out_type]``: bf16 for bf16 and e4m3
    outputs, fp16 for fp16, fp32 for fp32) or None; out_type 0 bf16, 1 fp16,
    2 fp32, 3 e4m3fn.

    Returns ``(out_bits, ref64 float64, absum float64)``, each of shape
    [len(rows), len(cols)]; ``out_bits`` has the dtype ``OUT_BITS[out_type]``;
    ``absum`` is S_ij * sum_k |a_ik b_kj|.
    """
    A = np.ascontiguousarray(A, dtype=np.uint8)
    Bt = np.ascontiguousarray(Bt, dtype=np.uint8)
    if A.ndim != 2 or Bt.ndim != 2 or A.shape[1] != Bt.shape[1]:
        raise ValueError("A must be [M,K] and Bt [N,K]")
    M, K = A.shape
    N = Bt.shape[0]
    sa = np.ascontiguousarray(scale_a, dtype=np.float32).reshape(-1)
    sb = np.ascontiguousarray(scale_b, dtype=np.float32).reshape(-1)
    if scale_mode == 0:
        if sa.size != 1 or sb.size != 1:
            raise ValueError("per-tensor scales must hold one value each")
    elif scale_mode == 1:
        if sa.size != M or sb.size != N:
            raise ValueError("row-wise scales must hold M and N values")
    else:
        raise ValueError("scale_mode must be 0 or 1")
    bias_arr = None
    if bias is not None:
        bias_arr = np.ascontiguousarray(bias, dtype=BIAS_BITS[int(out_type)]).reshape(-1)
        if bias_arr.size != N:
            raise ValueError("bias must hold N values")
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    c = None if cols is None else np.ascontiguousarray(cols, dtype=np.int64)
    nr = M if r is None else r.size
    nc = N if c is None else c.size
    out = np.zeros((nr, nc), dtype=OUT_BITS[int(out_type)])
    ref = np.zeros((nr, nc), dtype=np.float64)
    mag = np.zeros((nr, nc), dtype=np.float64)
    c_i64p = ctypes.POINTER(ctypes.c_int64)
    rc = _load().oracle_scaled_mm_typed(
        A.ctypes.data, int(a_type), Bt.ctypes.data, int(b_type), M, N, K,
        sa.ctypes.data, sb.ctypes.data, int(scale_mode),
        None if bias_arr is None else bias_arr.ctypes.data, int(out_type),
        None if r is None else r.ctypes.data_as(c_i64p), nr,
        None if c is None else c.ctypes.data_as(c_i64p), nc,
        out.ctypes.data, ref.ctypes.data, mag.ctypes.data, int(threads))
    if rc != 0:
        raise RuntimeError(f"oracle_scaled_mm failed with code {rc}")
    return out, ref, mag


def encode(values, q_type: int = E4M3) -> np.ndarray:
    """fp32 values -> fp8 codes (round to nearest even); NaN -> 0x7F | sign."""
    lib = _load()
    f = lib.oracle_encode_e4m3 if q_type == E4M3 else lib.oracle_encode_e5m2
    v = np.asarray(values, dtype=np.float32).reshape(-1)
    return np.fromiter((f(float(x)) for x in v), dtype=np.uint8, count=v.size)


def quantize(x_bf16_bits, scale_mode: int, q_type: int = E4M3, threads: int = 0):
    """bf16 bit patterns [R, C] -> (fp8 codes uint8 [R, C], fp32 scales [1] or [R]).

    The quantisation recipe of the gist "matmul_fp8.py" (`get_scale`,
    `benchmark()`): amax over the tensor or each row, scale = amax / qmax,
    codes = encode(clamp(x / scale, -qmax, qmax)), all in fp32.
    """
    x = np.ascontiguousarray(x_bf16_bits, dtype=np.uint16)
    if x.ndim != 2:
        raise ValueError("x must be [R, C]")
    R, C = x.shape
    q = np.zeros((R, C), dtype=np.uint8)
    scale = np.zeros(1 if scale_mode == 0 else R, dtype=np.float32)
    rc = _load().oracle_quantize(x.ctypes.data, R, C, int(scale_mode), int(q_type), q.ctypes.data,
                                 scale.ctypes.data, int(threads))
    if rc != 0:
        raise RuntimeError(f"oracle_quantize failed with code {rc}")
    return q, scale


def tolerance(ref_bits, absum, out_type: int = BF16) -> np.ndarray:
    """Allowed |gpu - ref| per element: ulp_rel |ref| + 2^-20 absum.

    ``ref`` is the rounded oracle value; the first term admits one unit in
    the last place of the output type (2^-7 relative for bf16, 2^-10 for
    fp16; a rounding boundary crossed by fp32 accumulation), the second the
    fp32 accumulation error near cancellation. For the other output types
    the same form with their unit in the last place and, because a relative
    term cannot cover the subnormal range, one subnormal quantum: fp16
    2^-10 |ref| + 2^-24, fp32 2^-23 |ref| + 2^-149, e4m3 2^-3 |ref| + 2^-9.
    """
    ref = out_to_f64(ref_bits, out_type)
    acc = np.asarray(absum) * 2.0 ** -20
    if out_type == BF16:
        return np.abs(ref) * 2.0 ** -7 + acc
    if out_type == F16:
        return np.abs(ref) * 2.0 ** -10 + acc + 2.0 ** -24
    if out_type == F32:
        return np.abs(ref) * 2.0 ** -23 + acc + 2.0 ** -149
    return np.abs(ref) * 2.0 ** -3 + acc + 2.0 ** -9
