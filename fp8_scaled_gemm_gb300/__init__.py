"""GB300 (sm_103a) FP8 scaled matrix multiply.

    out[M, N] = bf16( (A[M, K] . B[K, N]) * (scale_a (x) scale_b) + bias[N] )

A thin ctypes binding over ``libfp8mm.so`` (``include/fp8mm.h``): each
function has the name of the C entry point it calls and only checks and
marshals arguments; every step of the computation runs in the CUDA kernels.
There is no CPU fallback: if the library cannot be loaded, calls raise.

Operation sources: gist "matmul_fp8.py" (FP8 Matmul), ``matmul_fp8_kernel``
(scale epilogue) and ``benchmark()`` (B column-major); PyTorch PR #125204,
Summary (row-wise scales of length M and N, TN layout); PyTorch PR #142045,
Summary (bias).
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

from . import _build

SCALE_TENSOR = 0
SCALE_ROWWISE = 1
VARIANT_AUTO = 0
VARIANT_TILE = 1
VARIANT_SWAP = 2
VARIANT_PAIR = 3
VARIANT_SWAPK = 4
VARIANT_SWAPPAIR = 5

TYPE_E4M3, TYPE_E5M2 = 0, 1
MAJOR_K, MAJOR_MN = 0, 1
OUT_BF16, OUT_F16, OUT_F32, OUT_E4M3 = 0, 1, 2, 3
_FP8 = {torch.float8_e4m3fn: TYPE_E4M3, torch.float8_e5m2: TYPE_E5M2}
_OUT = {torch.bfloat16: OUT_BF16, torch.float16: OUT_F16, torch.float32: OUT_F32,
        torch.float8_e4m3fn: OUT_E4M3}
# the bias dtype each output dtype takes (an e4m3 output takes a bf16 bias)
_BIAS = {torch.bfloat16: torch.bfloat16, torch.float16: torch.float16, torch.float32: torch.float32,
         torch.float8_e4m3fn: torch.bfloat16}


class Options(ctypes.Structure):
    """fp8mm_options of include/fp8mm.h."""
    _fields_ = [("a_type", ctypes.c_int), ("b_type", ctypes.c_int), ("out_type", ctypes.c_int),
                ("variant", ctypes.c_int), ("tile_n", ctypes.c_int), ("split_k", ctypes.c_int),
                ("ldo", ctypes.c_int64)]


STATUS = {
    0: "FP8MM_OK", -1: "FP8MM_ERR_NULL", -2: "FP8MM_ERR_SHAPE", -3: "FP8MM_ERR_ALIGN",
    -4: "FP8MM_ERR_MODE", -5: "FP8MM_ERR_CUDA", -6: "FP8MM_ERR_NODEV", -7: "FP8MM_ERR_TIMEOUT",
}

# Every symbol include/fp8mm.h declares.
EXPORTS = (
    "fp8_scaled_mm", "fp8_scaled_mm_config", "fp8_scaled_mm_ex", "fp8_scaled_mm_host",
    "fp8_scaled_mm_noalloc", "fp8_quantize", "fp8_scaled_mm_bf16", "fp8_scaled_bmm",
    "fp8_scaled_mm_layout",
    "fp8mm_reserve_workspace", "fp8mm_device_status", "fp8mm_status_string",
    "fp8mm_last_cuda_error", "fp8mm_last_error", "fp8mm_describe_choice", "fp8mm_describe_bmm_choice", "fp8mm_debug_inject", "fp8mm_debug_quant", "fp8mm_describe_model_choice",
    "fp8mm_describe_quant_plan",
    "fp8mm_autotune", "fp8mm_autotune_clear", "fp8mm_autotune_count", "fp8mm_autotune_save",
    "fp8mm_autotune_load",
)

_lib = None
_lock = threading.Lock()


class Fp8mmError(RuntimeError):
    def __init__(self, status: int, detail: str = ""):
        self.status = status
        name = STATUS.get(status, str(status))
        super().__init__(f"{name}: {detail}" if detail else name)


def lib_path() -> str:
    return _build.LIB_PATH


def load(build_if_missing: bool = False) -> ctypes.CDLL:
    """Load ``libfp8mm.so`` (built by ``__graft_entry__.build()``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB_PATH
        if not os.path.exists(path):
            if not build_if_missing:
                raise RuntimeError(
                    f"CUDA library {path} is missing; build it with "
                    "`python -c 'import __graft_entry__ as g; g.build()'`")
            _build.build()
        lib = ctypes.CDLL(path)
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        common = [vp, vp, vp, vp, i32, vp, vp, i64, i64, i64, vp]
        lib.fp8_scaled_mm.argtypes = common
        lib.fp8_scaled_mm.restype = i32
        lib.fp8_scaled_mm_config.argtypes = common + [i32, i32, i32]
        lib.fp8_scaled_mm_config.restype = i32
        lib.fp8_scaled_mm_ex.argtypes = common + [ctypes.POINTER(Options)]
        lib.fp8_scaled_mm_ex.restype = i32
        lib.fp8_scaled_mm_host.argtypes = common
        lib.fp8_scaled_mm_host.restype = i32
        lib.fp8_scaled_mm_noalloc.argtypes = common
        lib.fp8_scaled_mm_noalloc.restype = i32
        lib.fp8_scaled_mm_layout.argtypes = [vp, i32, vp, i32, vp, vp, i32, vp, vp, i64, i64, i64, vp,
                                             ctypes.POINTER(Options)]
        lib.fp8_scaled_mm_layout.restype = i32
        lib.fp8_scaled_bmm.argtypes = [vp, vp, vp, vp, i32, vp, vp, i64, i64, i64, i64, vp,
                                       ctypes.POINTER(Options)]
        lib.fp8_scaled_bmm.restype = i32
        lib.fp8_quantize.argtypes = [vp, i64, i64, i32, i32, vp, vp, vp]
        lib.fp8_quantize.restype = i32
        lib.fp8_scaled_mm_bf16.argtypes = [vp, vp, i32, vp, vp, i64, i64, i64, vp, vp, vp, vp, vp,
                                           ctypes.POINTER(Options)]
        lib.fp8_scaled_mm_bf16.restype = i32
        lib.fp8mm_reserve_workspace.argtypes = [i64]
        lib.fp8mm_reserve_workspace.restype = i32
        lib.fp8mm_device_status.argtypes = [vp]
        lib.fp8mm_device_status.restype = i32
        lib.fp8mm_status_string.argtypes = [i32]
        lib.fp8mm_status_string.restype = ctypes.c_char_p
        lib.fp8mm_last_cuda_error.argtypes = []
        lib.fp8mm_last_cuda_error.restype = ctypes.c_char_p
        lib.fp8mm_last_error.argtypes = []
        lib.fp8mm_last_error.restype = ctypes.c_char_p
        lib.fp8mm_debug_inject.argtypes = [i64, i64]
        lib.fp8mm_debug_inject.restype = i32
        lib.fp8mm_debug_quant.argtypes = [i32]
        lib.fp8mm_debug_quant.restype = i32
        lib.fp8mm_describe_model_choice.argtypes = [i64, i64, i64, i64, i32]
        lib.fp8mm_describe_model_choice.restype = ctypes.c_char_p
        lib.fp8mm_describe_quant_plan.argtypes = [i64, i64, i32, i32]
        lib.fp8mm_describe_quant_plan.restype = ctypes.c_char_p
        lib.fp8mm_describe_choice.argtypes = [i64, i64, i64, i32]
        lib.fp8mm_describe_choice.restype = ctypes.c_char_p
        lib.fp8mm_autotune.argtypes = [i64, i64, i64, i64, i32, ctypes.POINTER(Options), vp]
        lib.fp8mm_autotune.restype = i32
        lib.fp8mm_autotune_clear.argtypes = []
        lib.fp8mm_autotune_clear.restype = i32
        lib.fp8mm_autotune_count.argtypes = []
        lib.fp8mm_autotune_count.restype = i32
        lib.fp8mm_autotune_save.argtypes = [ctypes.c_char_p]
        lib.fp8mm_autotune_save.restype = i32
        lib.fp8mm_autotune_load.argtypes = [ctypes.c_char_p]
        lib.fp8mm_autotune_load.restype = i32
        lib.fp8mm_describe_bmm_choice.argtypes = [i64, i64, i64, i64, i32]
        lib.fp8mm_describe_bmm_choice.restype = ctypes.c_char_p
        _lib = lib
        return lib


def _check(rc: int):
    if rc != 0:
        detail = load().fp8mm_last_cuda_error().decode(errors="replace")
        raise Fp8mmError(rc, detail)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(int(stream.cuda_stream))


def _validate(A, B, scale_a, scale_b, scale_mode, bias, out, device_side: bool, typed: bool = False):
    if A.dim() != 2 or B.dim() != 2:
        raise ValueError("A must be [M, K] and B [K, N]")
    M, K = A.shape
    K2, N = B.shape
    if K2 != K:
        raise ValueError(f"inner dimensions differ: A is {tuple(A.shape)}, B is {tuple(B.shape)}")
    fp8 = tuple(_FP8) if typed else (torch.float8_e4m3fn,)
    if A.dtype not in fp8 or B.dtype not in fp8:
        raise ValueError("A and B must be torch.float8_e4m3fn" + (" or float8_e5m2" if typed else ""))
    if A.stride() != (K, 1) and M > 1:
        raise ValueError("A must be row-major contiguous [M, K]")
    if B.stride() != (1, K) and N > 1:
        raise ValueError("B must be column-major [K, N] (B.t() contiguous)")
    if scale_mode not in (SCALE_TENSOR, SCALE_ROWWISE):
        raise ValueError("scale_mode must be 0 (per-tensor) or 1 (row-wise)")
    want_a = 1 if scale_mode == SCALE_TENSOR else M
    want_b = 1 if scale_mode == SCALE_TENSOR else N
    for name, s, n in (("scale_a", scale_a, want_a), ("scale_b", scale_b, want_b)):
        if s.dtype != torch.float32 or s.numel() != n or not s.is_contiguous():
            raise ValueError(f"{name} must be a contiguous float32 tensor of {n} values")
    outs = tuple(_OUT) if typed else (torch.bfloat16,)
    # typed calls also take a row-strided out (row stride >= N, columns contiguous)
    strided_ok = typed and out.dim() == 2 and (out.stride(1) == 1 or N == 1) and out.stride(0) >= N
    if out.dtype not in outs or tuple(out.shape) != (M, N) or not (out.is_contiguous() or strided_ok):
        raise ValueError("out must be a [M, N] tensor of " +
                         ("bfloat16, float16, float32 or float8_e4m3fn with contiguous rows" if typed
                          else "bfloat16, contiguous"))
    if bias is not None and (bias.dtype != _BIAS[out.dtype] or bias.numel() != N or
                             not bias.is_contiguous()):
        raise ValueError("bias must be a contiguous tensor of N values of out's dtype "
                         "(bfloat16 for a float8_e4m3fn output)")
    tensors = [A, B, scale_a, scale_b, out] + ([bias] if bias is not None else [])
    for t in tensors:
        if device_side and not t.is_cuda:
            raise ValueError("fp8_scaled_mm takes CUDA tensors (use fp8_scaled_mm_host for host memory)")
        if not device_side and t.is_cuda:
            raise ValueError("fp8_scaled_mm_host takes host (CPU) tensors")
    return M, N, K


def fp8_scaled_mm(A, B, scale_a, scale_b, scale_mode: int, bias=None, out=None, stream=None):
    """out = bf16(A.B * scale + bias) on the GPU. B is [K, N] column-major."""
    if out is None:
        out = torch.empty((A.shape[0], B.shape[1]), dtype=torch.bfloat16, device=A.device)
    M, N, K = _validate(A, B, scale_a, scale_b, scale_mode, bias, out, True)
    _check(load().fp8_scaled_mm(_ptr(A), _ptr(B), _ptr(scale_a), _ptr(scale_b), scale_mode,
                                _ptr(bias), _ptr(out), M, N, K, _stream_handle(stream)))
    return out


def fp8_scaled_mm_config(A, B, scale_a, scale_b, scale_mode: int, bias=None, out=None,
                         stream=None, variant: int = VARIANT_AUTO, tile_n: int = 0,
                         split_k: int = 0):
    """fp8_scaled_mm with an explicit kernel choice (see include/fp8mm.h)."""
    if out is None:
        out = torch.empty((A.shape[0], B.shape[1]), dtype=torch.bfloat16, device=A.device)
    M, N, K = _validate(A, B, scale_a, scale_b, scale_mode, bias, out, True)
    _check(load().fp8_scaled_mm_config(_ptr(A), _ptr(B), _ptr(scale_a), _ptr(scale_b), scale_mode,
                                       _ptr(bias), _ptr(out), M, N, K, _stream_handle(stream),
                                       int(variant), int(tile_n), int(split_k)))
    return out


def fp8_scaled_mm_ex(A, B, scale_a, scale_b, scale_mode: int, bias=None, out=None, stream=None,
                     out_dtype=torch.bfloat16, variant: int = VARIANT_AUTO, tile_n: int = 0,
                     split_k: int = 0):
    """The operation with e4m3fn / e5m2 operands and a bf16 / fp16 / fp32 /
    e4m3fn output (types taken from the tensors; bias has out's dtype, bf16
    for an e4m3fn output, which saturates at +-448). ``out`` may be a view
    with a row stride of at least N (e.g. columns of a wider matrix)."""
    if out is None:
        out = torch.empty((A.shape[0], B.shape[1]), dtype=out_dtype, device=A.device)
    M, N, K = _validate(A, B, scale_a, scale_b, scale_mode, bias, out, True, typed=True)
    ldo = 0 if out.is_contiguous() else int(out.stride(0))
    opt = Options(_FP8[A.dtype], _FP8[B.dtype], _OUT[out.dtype], int(variant), int(tile_n), int(split_k), ldo)
    _check(load().fp8_scaled_mm_ex(_ptr(A), _ptr(B), _ptr(scale_a), _ptr(scale_b), scale_mode,
                                   _ptr(bias), _ptr(out), M, N, K, _stream_handle(stream),
                                   ctypes.byref(opt)))
    return out


def _major(t, k_stride_dim: int) -> int:
    """MAJOR_K if the operand's K dimension (dim k_stride_dim) is contiguous,
    MAJOR_MN if the other one is; raises otherwise."""
    other = 1 - k_stride_dim
    if t.stride(k_stride_dim) == 1 and t.stride(other) == t.shape[k_stride_dim]:
        return MAJOR_K
    if t.stride(other) == 1 and t.stride(k_stride_dim) == t.shape[other]:
        return MAJOR_MN
    raise ValueError("operands must be contiguous in one of their two dimensions")


def fp8_scaled_mm_layout(A, B, scale_a, scale_b, scale_mode: int, bias=None, out=None, stream=None,
                         out_dtype=torch.bfloat16, variant: int = VARIANT_AUTO, tile_n: int = 0,
                         split_k: int = 0):
    """The operation with A [M, K] and B [K, N] in any of the four layouts
    (each operand row- or column-major, read from its strides). An operand
    whose K dimension is not contiguous is transposed on the GPU first."""
    if A.dim() != 2 or B.dim() != 2 or A.shape[1] != B.shape[0]:
        raise ValueError("A must be [M, K] and B [K, N]")
    M, K = A.shape
    N = B.shape[1]
    a_major = _major(A, 1)
    b_major = _major(B, 0)
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=A.device)
    if A.dtype not in _FP8 or B.dtype not in _FP8:
        raise ValueError("A and B must be torch.float8_e4m3fn or float8_e5m2")
    if scale_mode not in (SCALE_TENSOR, SCALE_ROWWISE):
        raise ValueError("scale_mode must be 0 (per-tensor) or 1 (row-wise)")
    for name, s, n in (("scale_a", scale_a, 1 if scale_mode == SCALE_TENSOR else M),
                       ("scale_b", scale_b, 1 if scale_mode == SCALE_TENSOR else N)):
        if s.dtype != torch.float32 or s.numel() != n or not s.is_contiguous():
            raise ValueError(f"{name} must be a contiguous float32 tensor of {n} values")
    if out.dtype not in _OUT or tuple(out.shape) != (M, N) or not out.is_contiguous():
        raise ValueError("out must be a contiguous [M, N] bfloat16, float16, float32 or float8_e4m3fn tensor")
    if bias is not None and (bias.dtype != _BIAS.get(out.dtype) or bias.numel() != N or not bias.is_contiguous()):
        raise ValueError("bias must be a contiguous tensor of N values with out's dtype")
    for t in [A, B, scale_a, scale_b, out] + ([bias] if bias is not None else []):
        if not t.is_cuda:
            raise ValueError("fp8_scaled_mm_layout takes CUDA tensors")
    opt = Options(_FP8[A.dtype], _FP8[B.dtype], _OUT[out.dtype], int(variant), int(tile_n), int(split_k))
    _check(load().fp8_scaled_mm_layout(_ptr(A), a_major, _ptr(B), b_major, _ptr(scale_a), _ptr(scale_b),
                                       scale_mode, _ptr(bias), _ptr(out), M, N, K, _stream_handle(stream),
                                       ctypes.byref(opt)))
    return out


def fp8_scaled_bmm(A, B, scale_a, scale_b, scale_mode: int, bias=None, out=None, stream=None,
                   out_dtype=torch.bfloat16, variant: int = VARIANT_AUTO, tile_n: int = 0, split_k: int = 0):
    """Batched scaled matmul: out[b] = A[b] . B[b] * scale + bias for every b.

    A is [batch, M, K] contiguous; B is [batch, K, N] with every item
    column-major (``B.transpose(1, 2)`` contiguous); scale_a is [batch] or
    [batch, M], scale_b [batch] or [batch, N]; bias [N] is shared; out is
    [batch, M, N]. Element types as for fp8_scaled_mm_ex.
    """
    if A.dim() != 3 or B.dim() != 3 or A.shape[0] != B.shape[0] or A.shape[2] != B.shape[1]:
        raise ValueError("A must be [batch, M, K] and B [batch, K, N]")
    nb, M, K = A.shape
    N = B.shape[2]
    if out is None:
        out = torch.empty((nb, M, N), dtype=out_dtype, device=A.device)
    if A.dtype not in _FP8 or B.dtype not in _FP8:
        raise ValueError("A and B must be torch.float8_e4m3fn or float8_e5m2")
    if not A.is_contiguous():
        raise ValueError("A must be contiguous [batch, M, K]")
    if not B.transpose(1, 2).is_contiguous():
        raise ValueError("every item of B must be column-major (B.transpose(1, 2) contiguous)")
    if scale_mode not in (SCALE_TENSOR, SCALE_ROWWISE):
        raise ValueError("scale_mode must be 0 (per-tensor) or 1 (row-wise)")
    for name, s, n in (("scale_a", scale_a, nb * (1 if scale_mode == SCALE_TENSOR else M)),
                       ("scale_b", scale_b, nb * (1 if scale_mode == SCALE_TENSOR else N))):
        if s.dtype != torch.float32 or s.numel() != n or not s.is_contiguous():
            raise ValueError(f"{name} must be a contiguous float32 tensor of {n} values")
    if out.dtype not in _OUT or tuple(out.shape) != (nb, M, N) or not out.is_contiguous():
        raise ValueError("out must be a contiguous [batch, M, N] bfloat16, float16, float32 or float8_e4m3fn tensor")
    if bias is not None and (bias.dtype != _BIAS.get(out.dtype) or bias.numel() != N or not bias.is_contiguous()):
        raise ValueError("bias must be a contiguous tensor of N values with out's dtype")
    for t in [A, B, scale_a, scale_b, out] + ([bias] if bias is not None else []):
        if not t.is_cuda:
            raise ValueError("fp8_scaled_bmm takes CUDA tensors")
    opt = Options(_FP8[A.dtype], _FP8[B.dtype], _OUT[out.dtype], int(variant), int(tile_n), int(split_k))
    _check(load().fp8_scaled_bmm(_ptr(A), _ptr(B), _ptr(scale_a), _ptr(scale_b), scale_mode, _ptr(bias),
                                 _ptr(out), nb, M, N, K, _stream_handle(stream), ctypes.byref(opt)))
    return out


def fp8_scaled_mm_host(A, B, scale_a, scale_b, scale_mode: int, bias=None, out=None, stream=None):
    """Same operation on host (CPU) tensors: copies in, computes, copies out."""
    if out is None:
        out = torch.empty((A.shape[0], B.shape[1]), dtype=torch.bfloat16)
    M, N, K = _validate(A, B, scale_a, scale_b, scale_mode, bias, out, False)
    _check(load().fp8_scaled_mm_host(_ptr(A), _ptr(B), _ptr(scale_a), _ptr(scale_b), scale_mode,
                                     _ptr(bias), _ptr(out), M, N, K, _stream_handle(stream)))
    return out


def fp8_scaled_mm_noalloc(A, B, scale_a, scale_b, scale_mode: int, bias=None, out=None, stream=None):
    """fp8_scaled_mm for callers that cannot allocate device memory mid-run.

    The library keeps its split-K scratch in a fixed array inside its device
    image instead of allocating a workspace; problems that would need more
    than that array holds raise Fp8mmError (FP8MM_ERR_SHAPE). ``out`` must be
    given (allocating it here would defeat the purpose).
    """
    if out is None:
        raise ValueError("fp8_scaled_mm_noalloc needs a preallocated out tensor")
    M, N, K = _validate(A, B, scale_a, scale_b, scale_mode, bias, out, True)
    _check(load().fp8_scaled_mm_noalloc(_ptr(A), _ptr(B), _ptr(scale_a), _ptr(scale_b), scale_mode,
                                        _ptr(bias), _ptr(out), M, N, K, _stream_handle(stream)))
    return out


def _validate_bf16_rows(name, x, device_side=True):
    if x.dtype != torch.bfloat16 or x.dim() != 2 or not x.is_contiguous():
        raise ValueError(f"{name} must be a contiguous 2-D bfloat16 tensor")
    if x.shape[1] % 8 != 0:
        raise ValueError(f"{name}'s row length must be a multiple of 8")
    if device_side and not x.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")


def fp8_quantize(x, scale_mode: int, dtype=torch.float8_e4m3fn, out=None, scale=None, stream=None):
    """bf16 x [R, C] -> (fp8 codes [R, C], fp32 scales [1] or [R]) on the GPU.

    amax over the tensor (scale_mode 0) or each row (1), scale = amax / qmax,
    codes = fp8(clamp(x / scale, -qmax, qmax)): the recipe of the gist
    "matmul_fp8.py" (``get_scale``, ``benchmark()``). For B pass ``B.t()``
    of a column-major B, i.e. Bt [N, K].
    """
    _validate_bf16_rows("x", x)
    if dtype not in _FP8:
        raise ValueError("dtype must be torch.float8_e4m3fn or torch.float8_e5m2")
    if scale_mode not in (SCALE_TENSOR, SCALE_ROWWISE):
        raise ValueError("scale_mode must be 0 (per-tensor) or 1 (row-wise)")
    R, C = x.shape
    if out is None:
        out = torch.empty((R, C), dtype=dtype, device=x.device)
    if scale is None:
        scale = torch.empty(1 if scale_mode == SCALE_TENSOR else R, dtype=torch.float32, device=x.device)
    if out.dtype != dtype or tuple(out.shape) != (R, C) or not out.is_contiguous() or not out.is_cuda:
        raise ValueError("out must be a contiguous CUDA [R, C] tensor of the requested fp8 dtype")
    n_scale = 1 if scale_mode == SCALE_TENSOR else R
    if scale.dtype != torch.float32 or scale.numel() != n_scale or not scale.is_contiguous() or not scale.is_cuda:
        raise ValueError(f"scale must be a contiguous CUDA float32 tensor of {n_scale} values")
    _check(load().fp8_quantize(_ptr(x), R, C, int(scale_mode), _FP8[dtype], _ptr(out), _ptr(scale),
                               _stream_handle(stream)))
    return out, scale


def fp8_scaled_mm_bf16(A, B, scale_mode: int, bias=None, out=None, stream=None,
                       out_dtype=torch.bfloat16, a_dtype=torch.float8_e4m3fn, b_dtype=torch.float8_e4m3fn,
                       variant: int = VARIANT_AUTO, tile_n: int = 0, split_k: int = 0,
                       return_quantized: bool = False):
    """The whole path from bf16 operands: quantise A [M, K] and B [K, N]
    (column-major) with ``scale_mode``, then the scaled matmul. Returns out,
    or (out, A_q, B_q, scale_a, scale_b) with ``return_quantized``."""
    if A.dim() != 2 or B.dim() != 2 or A.shape[1] != B.shape[0]:
        raise ValueError("A must be [M, K] and B [K, N]")
    Bt = B.t()
    _validate_bf16_rows("A", A)
    _validate_bf16_rows("B.t()", Bt)
    M, K = A.shape
    N = B.shape[1]
    dev = A.device
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=dev)
    a_q = torch.empty((M, K), dtype=a_dtype, device=dev)
    bt_q = torch.empty((N, K), dtype=b_dtype, device=dev)
    ns_a, ns_b = (1, 1) if scale_mode == SCALE_TENSOR else (M, N)
    scale_a = torch.empty(ns_a, dtype=torch.float32, device=dev)
    scale_b = torch.empty(ns_b, dtype=torch.float32, device=dev)
    _validate(a_q, bt_q.t(), scale_a, scale_b, scale_mode, bias, out, True, typed=True)
    ldo = 0 if out.is_contiguous() else int(out.stride(0))
    opt = Options(_FP8[a_dtype], _FP8[b_dtype], _OUT[out.dtype], int(variant), int(tile_n), int(split_k), ldo)
    _check(load().fp8_scaled_mm_bf16(_ptr(A), _ptr(Bt), int(scale_mode), _ptr(bias), _ptr(out), M, N, K,
                                     _ptr(a_q), _ptr(bt_q), _ptr(scale_a), _ptr(scale_b),
                                     _stream_handle(stream), ctypes.byref(opt)))
    if return_quantized:
        return out, a_q, bt_q.t(), scale_a, scale_b
    return out


def fp8mm_reserve_workspace(nbytes: int) -> None:
    _check(load().fp8mm_reserve_workspace(int(nbytes)))


def fp8mm_device_status(stream=None) -> int:
    """Synchronise and return the in-kernel status (0 = ok, -7 = a wait ran out)."""
    return int(load().fp8mm_device_status(_stream_handle(stream)))


def fp8mm_status_string(status: int) -> str:
    return load().fp8mm_status_string(int(status)).decode()


def fp8mm_last_cuda_error() -> str:
    """Detail of the last failure on this host thread ("" if none)."""
    return load().fp8mm_last_cuda_error().decode(errors="replace")


def fp8mm_last_error() -> str:
    """Alias of fp8mm_last_cuda_error."""
    return load().fp8mm_last_error().decode(errors="replace")


def fp8mm_debug_quant(mode: int = 0) -> None:
    """Test hook for per-tensor quantisation (see include/fp8mm.h): 1 forces
    the two-launch form, 2 makes the one-launch kernel's grid-wide wait run
    out; fp8mm_debug_quant() restores normal operation."""
    _check(load().fp8mm_debug_quant(int(mode)))


def fp8mm_debug_inject(stop_after_kblocks: int = -1, wait_limit_cycles: int = 0) -> None:
    """Test hook: make CTA 0's producer stop early so a bounded wait runs out
    (see include/fp8mm.h). fp8mm_debug_inject() restores normal operation."""
    _check(load().fp8mm_debug_inject(int(stop_after_kblocks), int(wait_limit_cycles)))


def fp8mm_describe_choice(M: int, N: int, K: int, scale_mode: int = SCALE_TENSOR) -> str:
    return load().fp8mm_describe_choice(int(M), int(N), int(K), int(scale_mode)).decode()


def fp8mm_describe_model_choice(M: int, N: int, K: int, sms: int, batch: int = 1) -> str:
    """The time model's automatic choice for a device with `sms` SMs (no
    device needed, tuned entries not consulted)."""
    return load().fp8mm_describe_model_choice(int(batch), int(M), int(N), int(K), int(sms)).decode()


def fp8mm_describe_quant_plan(R: int, C: int, scale_mode: int, sms: int) -> str:
    """The launch plan fp8_quantize takes for bf16 [R, C] on a device with
    `sms` SMs (no device needed)."""
    return load().fp8mm_describe_quant_plan(int(R), int(C), int(scale_mode), int(sms)).decode()


def fp8mm_describe_bmm_choice(batch: int, M: int, N: int, K: int, scale_mode: int = SCALE_TENSOR) -> str:
    return load().fp8mm_describe_bmm_choice(int(batch), int(M), int(N), int(K), int(scale_mode)).decode()


def fp8mm_autotune(M: int, N: int, K: int, scale_mode: int = SCALE_TENSOR, batch: int = 1,
                   a_dtype=torch.float8_e4m3fn, b_dtype=torch.float8_e4m3fn, out_dtype=torch.bfloat16,
                   stream=None) -> str:
    """Time the compiled kernel configurations for this problem and remember
    the fastest for automatic choice; returns the chosen configuration."""
    opt = Options(_FP8[a_dtype], _FP8[b_dtype], _OUT[out_dtype], VARIANT_AUTO, 0, 0)
    _check(load().fp8mm_autotune(int(batch), int(M), int(N), int(K), int(scale_mode), ctypes.byref(opt),
                                 _stream_handle(stream)))
    return fp8mm_describe_bmm_choice(batch, M, N, K, scale_mode)


def fp8mm_autotune_clear() -> None:
    _check(load().fp8mm_autotune_clear())


def fp8mm_autotune_count() -> int:
    return int(load().fp8mm_autotune_count())


def fp8mm_autotune_save(path: str) -> int:
    rc = load().fp8mm_autotune_save(os.fsencode(path))
    if rc < 0:
        _check(rc)
    return rc


def fp8mm_autotune_load(path: str) -> int:
    rc = load().fp8mm_autotune_load(os.fsencode(path))
    if rc < 0:
        _check(rc)
    return rc
