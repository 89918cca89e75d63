"""FP8MM_LOG=1: one stderr line per new problem with the kernel chosen for it."""
from __future__ import annotations

import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r"""
import torch
import fp8_scaled_gemm_gb300 as fm
from fp8_scaled_gemm_gb300.inputs import make_inputs
for (M, N, K) in ((64, 512, 256), (64, 512, 256), (300, 520, 400)):
    inp = make_inputs(M, N, K, 1, 1)
    fm.fp8_scaled_mm(inp.a_q.cuda(), inp.bt_q.cuda().t(), inp.scale_a.cuda(), inp.scale_b.cuda(), 1)
torch.cuda.synchronize()
print(fm.fp8mm_describe_choice(300, 520, 400, 1))
"""


def test_log_prints_one_line_per_new_problem():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    env = dict(os.environ, FP8MM_LOG="1", PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, "-c", SCRIPT], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stderr.splitlines() if ln.startswith("fp8mm: ")]
    assert len(lines) == 2, r.stderr
    assert "64x512x256 row-wise e4m3 x e4m3 -> bf16" in lines[0] and lines[0].endswith("(model)")
    assert r.stdout.strip().splitlines()[-1] in lines[1]
    # without the variable: silent
    env.pop("FP8MM_LOG")
    r = subprocess.run([sys.executable, "-c", SCRIPT], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0 and "fp8mm: " not in r.stderr
