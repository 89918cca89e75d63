"""Host-side logic of bench.py on the CPU: the byte counts behind the
roofline figures, the traffic lookup, the clock summary and the defaults.

The byte counts are checked against the scope table's figures, which were
worked out from the pages' operation (fp8 operands, 16-bit output and bias,
fp32 scales) independently of bench.py.
"""
from __future__ import annotations

import pytest

import bench


@pytest.mark.parametrize("M,N,K,mode,bias,mb", [
    (256, 256, 256, 0, False, 0.262),
    (8192, 8192, 8192, 0, False, 268.4),
    (8192, 8192, 8192, 1, False, 268.5),
    (16, 4096, 4096, 1, False, 16.99),
    (128, 14336, 4096, 1, False, 62.97),
    (3000, 5000, 4112, 1, True, 62.94),
    (16384, 8192, 1024, 1, True, 293.7),
    (1, 8192, 8192, 1, True, 67.18),
    (8191, 8193, 32, 1, True, 134.8),
])
def test_algorithmic_bytes_match_the_scope_table(M, N, K, mode, bias, mb):
    # the table prints four significant figures: half a unit of the last one
    assert bench.algorithmic_bytes(M, N, K, mode, bias) / 1e6 == pytest.approx(mb, rel=4e-4, abs=0.006)


def test_algorithmic_bytes_of_a_batch_scale_with_the_items():
    one = bench.algorithmic_bytes(512, 1024, 2048, 1, False)
    assert bench.algorithmic_bytes(512, 1024, 2048, 1, False, batch=4) == 4 * one
    # the bias is shared by the items of a batch
    with_bias = bench.algorithmic_bytes(512, 1024, 2048, 1, True, batch=4)
    assert with_bias == 4 * one + 2 * 1024


def test_quantiser_bytes():
    # 2 bytes in and 1 out per element, plus the fp32 scales
    assert bench.quant_bytes(8192, 8192, 1) == 3 * 8192 * 8192 + 4 * 8192
    assert bench.quant_bytes(8192, 8192, 0) == 3 * 8192 * 8192 + 4


def test_traffic_lookup_needs_the_exact_launch():
    assert bench.measured_traffic("tensor", "pair tile_n=256 split=1 no-such-launch") is None
    assert bench.measured_traffic("no-such-key", "") is None


def test_kernel_source_hash_is_stable_and_short():
    h = bench.kernel_src_sha()
    assert h == bench.kernel_src_sha()
    assert len(h) == 16 and all(c in "0123456789abcdef" for c in h)


def test_clock_summary_median_and_reasons():
    s = bench.ClockSampler(0)
    # (time, sm_mhz, max_mhz, reasons mask): sw_power_cap (0x4) while timed, idle (0x1) outside
    s.samples = [(0.5, 2070.0, 2070.0, 0x1), (1.0, 1600.0, 2070.0, 0x4), (1.1, 1580.0, 2070.0, 0x4),
                 (1.2, 1620.0, 2070.0, 0x4), (2.5, 2070.0, 2070.0, 0x1)]
    c = s.summary(0.9, 1.3)
    assert c["sm_mhz"] == 1600.0 and c["sm_max_mhz"] == 2070.0
    assert c["reasons"] == ["sw_power_cap"] and c["samples"] == 3 and c["window"] == "timed"


def test_clock_summary_of_a_window_shorter_than_the_sampling_period():
    s = bench.ClockSampler(0)
    s.samples = [(1.0, 1900.0, 2070.0, 0x0), (1.1, 1890.0, 2070.0, 0x40), (5.0, 900.0, 2070.0, 0x0)]
    c = s.summary(1.04, 1.05)
    assert c["window"] == "nearest"
    assert "hw_thermal_slowdown" in c["reasons"]   # a throttle reason seen next to the window is kept
    assert bench.ClockSampler(0).summary(0.0, 1.0)["window"] == "unavailable"


def test_default_arguments_keep_the_contract():
    a = bench.parse_args([])
    assert a.gpus == 1 and a.impl == "ours" and a.workload == "tensor"
    assert a.warmup >= 3 and a.steps >= 1
    assert not a.sweep and not a.quant and not a.plain_launches


def test_algorithmic_bytes_of_the_other_output_types():
    # fp32 output: 4 bytes per element and an fp32 bias; e4m3: 1 byte and a bf16 bias
    M, N, K = 512, 1024, 2048
    base = M * K + N * K + 4 * (M + N)
    assert bench.algorithmic_bytes(M, N, K, 1, True, out="fp32") == base + 4 * M * N + 4 * N
    assert bench.algorithmic_bytes(M, N, K, 1, True, out="e4m3") == base + M * N + 2 * N
    assert bench.algorithmic_bytes(M, N, K, 1, True, out="fp16") == bench.algorithmic_bytes(M, N, K, 1, True)


def test_nvml_sampler_without_nvml_reports_unavailable(monkeypatch):
    import ctypes

    def no_lib(*a, **k):
        raise OSError("no libnvidia-ml here")
    monkeypatch.setattr(ctypes, "CDLL", no_lib)
    s = bench.NvmlSampler(0)
    assert s.ok is False
    # its summary is the same as the nvidia-smi sampler's
    s.samples = [(1.000, 1800.0, 2070.0, 0x4), (1.001, 1810.0, 2070.0, 0x4), (1.002, 1790.0, 2070.0, 0x0)]
    c = s.summary(0.9995, 1.0025)
    assert c["window"] == "timed" and c["samples"] == 3 and c["sm_mhz"] == 1800.0
    assert c["reasons"] == ["sw_power_cap"]


def test_skinny_shapes_are_the_memory_bound_benchmark_shapes():
    pk_hbm = 6747.0
    for (m, n, k, mode, bias) in bench.SKINNY_SHAPES:
        assert m <= 128
        flops = 2 * m * n * k
        nbytes = bench.algorithmic_bytes(m, n, k, mode, bias)
        # below the ridge point of the measured peaks (fp8 ~ 3846 TFLOP/s / 6747 GB/s)
        assert flops / nbytes < 3846e12 / (pk_hbm * 1e9)
    assert bench.parse_args([]).no_skinny is False


def test_kernel_source_hash_ignores_comments_and_white_space():
    code = "int f(int x)\n{\n    return x + 1;   // one more\n}\n"
    commented = "/* a block\n   comment */\nint f(int x)\n{\n\n        return x + 1;\n}\n"
    assert bench.source_code_only(code) == bench.source_code_only(commented)
    assert bench.source_code_only(code) != bench.source_code_only(code.replace("+ 1", "+ 2"))
