"""Host-only checks of the C ABI (no GPU): the library builds and loads, it
exports every function include/fp8mm.h declares, and argument errors come
back as status codes before any CUDA call is made."""
from __future__ import annotations

import ctypes
import os
import re

import pytest
import torch

import fp8_scaled_gemm_gb300 as fm
from fp8_scaled_gemm_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8mm.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return fm.load()


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_binding_exports():
    assert header_functions() == sorted(fm.EXPORTS)


def test_library_exports_every_header_function(lib):
    for name in header_functions():
        assert hasattr(lib, name), name
        assert isinstance(getattr(lib, name), ctypes._CFuncPtr)


# The boundary the scope table fixes: these names, these codes.
BOUNDARY_CALLS = ("fp8_scaled_mm", "fp8mm_status_string", "fp8mm_last_cuda_error",
                  "fp8mm_reserve_workspace")
BOUNDARY_ENUMS = {
    "FP8MM_SCALE_TENSOR": 0, "FP8MM_SCALE_ROWWISE": 1,
    "FP8MM_OK": 0, "FP8MM_ERR_NULL": -1, "FP8MM_ERR_SHAPE": -2, "FP8MM_ERR_ALIGN": -3,
    "FP8MM_ERR_MODE": -4, "FP8MM_ERR_CUDA": -5, "FP8MM_ERR_NODEV": -6, "FP8MM_ERR_TIMEOUT": -7,
}


def test_boundary_names_are_exported_and_callable(lib):
    for name in BOUNDARY_CALLS:
        assert name in header_functions(), name
        assert isinstance(getattr(lib, name), ctypes._CFuncPtr), name
    text = open(HEADER).read()
    for name, value in BOUNDARY_ENUMS.items():
        m = re.search(rf"\b{name}\s*=\s*(-?\d+)", text)
        assert m and int(m.group(1)) == value, name
    # each call answers without a GPU on these arguments
    assert fm.fp8mm_status_string(-5) == "CUDA call failed"
    assert isinstance(fm.fp8mm_last_cuda_error(), str)
    assert fm.fp8mm_last_cuda_error() == fm.fp8mm_last_error()
    assert lib.fp8mm_reserve_workspace(-1) == -2
    assert call(lib, mode=7) == -4


def test_status_strings(lib):
    for code, name in fm.STATUS.items():
        s = fm.fp8mm_status_string(code)
        assert isinstance(s, str) and s
    assert fm.fp8mm_status_string(0) == "ok"
    assert fm.fp8mm_status_string(12345) == "unknown status"


# Fake, never-dereferenced device addresses: argument checks must reject the
# call before it touches CUDA.
ALIGNED = 0x7F0000000000
P = ctypes.c_void_p


def call(lib, A=ALIGNED, B=ALIGNED, sa=ALIGNED, sb=ALIGNED, mode=0, bias=None, out=ALIGNED,
         M=64, N=64, K=64):
    return lib.fp8_scaled_mm(P(A) if A else None, P(B) if B else None, P(sa) if sa else None,
                             P(sb) if sb else None, mode, P(bias) if bias else None,
                             P(out) if out else None, M, N, K, None)


@pytest.mark.parametrize("kw,code", [
    (dict(A=0), -1), (dict(B=0), -1), (dict(sa=0), -1), (dict(sb=0), -1), (dict(out=0), -1),
    (dict(mode=2), -4), (dict(mode=-1), -4),
    (dict(K=0), -2), (dict(K=8), -2), (dict(K=24), -2), (dict(K=-16), -2), (dict(M=-1), -2),
    (dict(N=-5), -2), (dict(M=2 ** 31), -2), (dict(K=2 ** 24 + 16), -2),
    (dict(A=ALIGNED + 8), -3), (dict(B=ALIGNED + 1), -3), (dict(sa=ALIGNED + 2), -3),
    (dict(out=ALIGNED + 2), -3), (dict(bias=ALIGNED + 1), -3),
])
def test_argument_errors_before_any_cuda_call(lib, kw, code):
    assert call(lib, **kw) == code


def test_empty_problem_is_a_noop(lib):
    assert call(lib, M=0) == 0
    assert call(lib, N=0) == 0


def test_config_rejects_unsupported_choices(lib):
    def cfg(variant, tile_n, split):
        return lib.fp8_scaled_mm_config(P(ALIGNED), P(ALIGNED), P(ALIGNED), P(ALIGNED), 0, None,
                                        P(ALIGNED), 64, 64, 64, None, variant, tile_n, split)
    assert cfg(6, 0, 0) == -4
    assert cfg(5, 256, 0) == -4       # SWAPPAIR takes 16..128
    assert cfg(5, 64, 2) == -4        # SWAPPAIR has no split-K
    assert cfg(4, 16, 3) == -4        # SWAPK cluster size is 2, 4 or 8
    assert cfg(3, 64, 0) == -4        # PAIR takes 128 or 256
    assert cfg(3, 256, 17) == -4      # split-K of at most 16 slices
    assert cfg(1, 64, 0) == -4        # TILE takes 128 or 256
    assert cfg(2, 256, 0) == -4       # SWAP takes 16..128
    assert cfg(1, 128, 17) == -4
    assert cfg(1, 128, -1) == -4


def test_ex_rejects_unknown_types(lib):
    def ex(at, bt, ot):
        opt = fm.Options(at, bt, ot, 0, 0, 0)
        return lib.fp8_scaled_mm_ex(P(ALIGNED), P(ALIGNED), P(ALIGNED), P(ALIGNED), 0, None, P(ALIGNED),
                                    64, 64, 64, None, ctypes.byref(opt))
    assert ex(2, 0, 0) == -4
    assert ex(0, -1, 0) == -4
    assert ex(0, 0, 4) == -4          # output types are 0..3 (bf16, fp16, fp32, e4m3fn)
    assert ex(0, 0, -1) == -4

    def ex_bias(ot, bias_addr):
        opt = fm.Options(0, 0, ot, 0, 0, 0)
        return lib.fp8_scaled_mm_ex(P(ALIGNED), P(ALIGNED), P(ALIGNED), P(ALIGNED), 0, P(bias_addr),
                                    P(ALIGNED), 64, 64, 64, None, ctypes.byref(opt))
    assert ex_bias(2, ALIGNED + 2) == -3   # an fp32 bias must be 4-byte aligned
    assert lib.fp8_scaled_mm_ex(P(ALIGNED), P(ALIGNED), P(ALIGNED), P(ALIGNED), 0, None, P(ALIGNED),
                                64, 64, 64, None, None) == -1


def test_debug_inject_validates_arguments(lib):
    assert lib.fp8mm_debug_inject(-2, 0) == -2
    assert lib.fp8mm_debug_inject(5, -1) == -2
    assert lib.fp8mm_debug_inject(2 ** 31, 0) == -2
    assert lib.fp8mm_debug_inject(3, 1 << 22) == 0
    assert lib.fp8mm_debug_inject(-1, 0) == 0      # back to normal


def test_debug_quant_validates_its_mode(lib):
    assert lib.fp8mm_debug_quant(3) == -4
    assert lib.fp8mm_debug_quant(-1) == -4
    for mode in (1, 2, 0):                         # ends in normal operation
        assert lib.fp8mm_debug_quant(mode) == 0


def test_python_layer_validates_layouts():
    M, N, K = 4, 8, 32
    A = torch.zeros(M, K, dtype=torch.float8_e4m3fn)
    Bt = torch.zeros(N, K, dtype=torch.float8_e4m3fn)
    sa = torch.ones(1)
    sb = torch.ones(1)
    out = torch.empty(M, N, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="column-major"):
        fm._validate(A, Bt.t().contiguous(), sa, sb, 0, None, out, False)
    with pytest.raises(ValueError, match="float8"):
        fm._validate(A.float(), Bt.t(), sa, sb, 0, None, out, False)
    with pytest.raises(ValueError, match="scale_a"):
        fm._validate(A, Bt.t(), torch.ones(M), sb, 0, None, out, False)
    with pytest.raises(ValueError, match="scale_b"):
        fm._validate(A, Bt.t(), torch.ones(M), torch.ones(1), 1, None, out, False)
    with pytest.raises(ValueError, match="bias"):
        fm._validate(A, Bt.t(), sa, sb, 0, torch.zeros(N), out, False)
    with pytest.raises(ValueError, match="float8"):      # e5m2 only through the typed entry
        fm._validate(A.view(torch.float8_e5m2), Bt.t(), sa, sb, 0, None, out, False)
    assert fm._validate(A.view(torch.float8_e5m2), Bt.t(), sa, sb, 0, None, out.half(), False,
                        typed=True) == (M, N, K)
    with pytest.raises(ValueError, match="CUDA"):
        fm._validate(A, Bt.t(), sa, sb, 0, None, out, True)
    assert fm._validate(A, Bt.t(), sa, sb, 0, None, out, False) == (M, N, K)


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(fm, "_lib", None)
    monkeypatch.setattr(_build, "LIB_PATH", str(tmp_path / "absent.so"))
    with pytest.raises(RuntimeError, match="missing"):
        fm.load()


def qcall(lib, x=ALIGNED, R=64, C=64, mode=0, q_type=0, q=ALIGNED, scale=ALIGNED):
    return lib.fp8_quantize(P(x) if x else None, R, C, mode, q_type, P(q) if q else None,
                            P(scale) if scale else None, None)


@pytest.mark.parametrize("kw,code", [
    (dict(C=12), -2), (dict(C=-8), -2), (dict(R=-1), -2), (dict(R=2 ** 40, C=64), -2),
    (dict(mode=2), -4), (dict(q_type=2), -4), (dict(q_type=-1), -4),
    (dict(x=0), -1), (dict(q=0), -1), (dict(scale=0), -1),
    (dict(x=ALIGNED + 8), -3), (dict(q=ALIGNED + 4), -3), (dict(scale=ALIGNED + 2), -3),
    (dict(R=0, x=0, q=0, scale=0), 0), (dict(C=0, x=0, q=0, scale=0), 0),
])
def test_quantize_argument_errors_before_any_cuda_call(lib, kw, code):
    assert qcall(lib, **kw) == code


def test_bf16_path_argument_errors(lib):
    def bf(A=ALIGNED, B=ALIGNED, M=64, N=64, K=64, aq=ALIGNED, bq=ALIGNED, opt=None, mode=0):
        return lib.fp8_scaled_mm_bf16(P(A) if A else None, P(B) if B else None, mode, None, P(ALIGNED),
                                      M, N, K, P(aq) if aq else None, P(bq) if bq else None,
                                      P(ALIGNED), P(ALIGNED), None,
                                      ctypes.byref(opt) if opt is not None else None)
    assert bf(aq=0) == -1
    assert bf(A=0) == -1
    assert bf(K=24) == -2
    assert bf(mode=3) == -4
    assert bf(opt=fm.Options(3, 0, 0, 0, 0, 0)) == -4
    assert bf(A=ALIGNED + 8) == -3
    assert bf(M=0, A=0, B=0, aq=0, bq=0) == 0


def test_python_quantize_validation():
    x = torch.zeros(4, 16, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        fm.fp8_quantize(x, 0)
    with pytest.raises(ValueError, match="multiple of 8"):
        fm.fp8_quantize(torch.zeros(4, 12, dtype=torch.bfloat16), 0)
    with pytest.raises(ValueError, match="bfloat16"):
        fm.fp8_quantize(x.float(), 0)


def test_bmm_argument_errors(lib):
    def bmm(batch=2, M=64, N=64, K=64, opt=None, A=ALIGNED):
        return lib.fp8_scaled_bmm(P(A) if A else None, P(ALIGNED), P(ALIGNED), P(ALIGNED), 0, None, P(ALIGNED),
                                  batch, M, N, K, None, ctypes.byref(opt) if opt is not None else None)
    assert bmm(batch=-1) == -2
    assert bmm(batch=0, A=0) == 0                  # empty batch: no-op before the pointer checks
    assert bmm(batch=2 ** 30, M=4096, N=4096) == -2  # work units would overflow
    assert bmm(K=24) == -2
    assert bmm(A=0) == -1
    assert bmm(opt=fm.Options(0, 5, 0, 0, 0, 0)) == -4
    assert bmm(opt=fm.Options(0, 0, 0, 9, 0, 0)) == -4


def test_layout_argument_errors(lib):
    def lay(am, bm, K=64):
        return lib.fp8_scaled_mm_layout(P(ALIGNED), am, P(ALIGNED), bm, P(ALIGNED), P(ALIGNED), 0, None,
                                        P(ALIGNED), 64, 64, K, None, None)
    assert lay(2, 0) == -4
    assert lay(0, -1) == -4
    assert lay(1, 1, K=24) == -2


def test_python_layout_detection():
    A = torch.zeros(6, 32, dtype=torch.float8_e4m3fn)
    assert fm._major(A, 1) == fm.MAJOR_K
    assert fm._major(A.t().contiguous().t(), 1) == fm.MAJOR_MN
    B = torch.zeros(32, 8, dtype=torch.float8_e4m3fn)       # row-major [K, N]
    assert fm._major(B, 0) == fm.MAJOR_MN
    assert fm._major(B.t().contiguous().t(), 0) == fm.MAJOR_K
    with pytest.raises(ValueError):
        fm._major(torch.zeros(6, 64, dtype=torch.float8_e4m3fn)[:, ::2], 1)


def test_autotune_table_save_and_load_without_a_gpu(lib, tmp_path):
    assert lib.fp8mm_autotune_clear() == 0
    assert lib.fp8mm_autotune_count() == 0
    good = tmp_path / "tuned.txt"
    good.write_text("# comment\n10 3 152 1 512 3072 12288 1 0 0 0 3 256 3 27.5\n"
                    "10 3 152 4 16 4096 4096 0 1 0 1 4 16 4 7.1\n")
    assert lib.fp8mm_autotune_load(str(good).encode()) == 2
    assert lib.fp8mm_autotune_count() == 2
    out = tmp_path / "saved.txt"
    assert lib.fp8mm_autotune_save(str(out).encode()) == 2
    lines = [l for l in out.read_text().splitlines() if not l.startswith("#")]
    assert sorted(l.split()[:14] for l in lines) == sorted(
        l.split()[:14] for l in good.read_text().splitlines() if not l.startswith("#"))
    assert lib.fp8mm_autotune_clear() == 0 and lib.fp8mm_autotune_count() == 0
    assert lib.fp8mm_autotune_load(str(out).encode()) == 2
    lib.fp8mm_autotune_clear()


@pytest.mark.parametrize("line", [
    "10 3 152 1 512 3072 12288 1 0 0 0 3 256 3",          # missing the time
    "10 3 152 1 512 3072 12300 1 0 0 0 3 256 1 1.0",      # K not a multiple of 16
    "10 3 152 1 512 3072 12288 1 0 0 0 4 16 3 1.0",       # cluster size 3
    "10 3 152 1 512 3072 12288 1 0 0 0 1 64 1 1.0",       # TILE takes 128 or 256
    "10 3 152 1 512 3072 12288 2 0 0 0 3 256 1 1.0",      # scale mode 2
])
def test_autotune_load_rejects_malformed_lines(lib, tmp_path, line):
    f = tmp_path / "bad.txt"
    f.write_text(line + "\n")
    assert lib.fp8mm_autotune_load(str(f).encode()) == -2
    assert lib.fp8mm_autotune_load(str(tmp_path / "absent.txt").encode()) == -1
    lib.fp8mm_autotune_clear()


def test_autotune_argument_errors(lib):
    assert lib.fp8mm_autotune(1, 64, 64, 24, 0, None, None) == -2
    assert lib.fp8mm_autotune(0, 64, 64, 64, 0, None, None) == -2
    assert lib.fp8mm_autotune(1, 64, 64, 64, 3, None, None) == -4
    assert lib.fp8mm_autotune(1, 64, 64, 64, 0, ctypes.byref(fm.Options(0, 0, 7, 0, 0, 0)), None) == -4
