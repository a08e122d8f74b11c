"""Host-side arithmetic of bench.py, on the CPU: the roofline bound and fraction, the whole-job
throughput, and the source key of the stored DRAM counters (comments and blank lines do not
change it, code does)."""
import importlib.util
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_host_under_test", os.path.join(ROOT, "bench.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    return b


PEAKS = dict(hbm_gbs=5000.0, bf16_tflops=2000.0, bf16_tflops_sustained=1800.0)


def test_roofline_picks_the_longer_of_tensor_and_hbm_time(bench):
    # 4e12 flops at 2000 TFLOP/s = 2 ms; 1e9 bytes at 5000 GB/s = 0.2 ms: tensor-bound
    r = bench.roofline_of(4e12, 1e9, 4.0, PEAKS, "bf16")
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["achieved"] == pytest.approx(1000.0) and r["frac"] == pytest.approx(0.5)
    # e4m3 operands: the nominal 2x peak halves the tensor time, so the same kernel reads 0.25
    r8 = bench.roofline_of(4e12, 1e9, 4.0, PEAKS, "e4m3")
    assert r8["peak"] == pytest.approx(4000.0) and r8["frac"] == pytest.approx(0.25)
    # 1e10 bytes = 2 ms at the copy bandwidth, 1e11 flops = 0.05 ms: HBM-bound
    h = bench.roofline_of(1e11, 1e10, 2.5, PEAKS, "bf16")
    assert h["bound"] == "hbm" and h["unit"] == "GB/s"
    assert h["achieved"] == pytest.approx(4000.0) and h["frac"] == pytest.approx(0.8)


def test_whole_job_throughput_counts_every_rank_at_the_slowest_rank_time(bench):
    assert bench.aggregate_tokens_per_s(4096, 1, 1.0) == pytest.approx(4.096e6)
    assert bench.aggregate_tokens_per_s(4096, 8, 2.0) == pytest.approx(8 * 4096 / 2e-3)


def test_counter_key_ignores_comments_but_not_code(bench):
    src = "int f(int a) {\n  return a + 1;  // one\n}\n"
    commented = "/* header\n   text */\nint f(int a) {\n\n  return a + 1;   // one more\n}\n"
    changed = "int f(int a) {\n  return a + 2;\n}\n"
    assert bench._code_only(src) == bench._code_only(commented)
    assert bench._code_only(src) != bench._code_only(changed)
    assert len(bench.src_hash()) == 16
