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


def test_stored_counters_are_found_by_workload_and_kernel_and_dropped_when_the_code_changed(bench, tmp_path,
                                                                                            monkeypatch):
    import json
    path = tmp_path / "traffic.json"
    h = bench.src_hash()
    path.write_text(json.dumps({"sweep_zipf1": {"gemm_wgrad_gu": {"dram_bytes_per_launch": 7.6e9, "src_hash": h,
                                                                   "note": "one pass"}},
                                "bf16_e64": {"gemm_wgrad_gu": {"dram_bytes_per_launch": 1.2e9,
                                                               "src_hash": "0000000000000000"}}}))
    monkeypatch.setattr(bench, "PROFILE_TRAFFIC", str(path))
    assert bench.traffic_for("gemm_wgrad_gu", "sweep_zipf1") == (7.6e9, "one pass")
    assert bench.traffic_for("gemm_wgrad_d", "sweep_zipf1") == (None, "kernel not captured")
    assert bench.traffic_for("gemm_wgrad_gu", "dsv3_e256") == (None, "kernel not captured")
    assert bench.traffic_for("gemm_wgrad_gu", "bf16_e64")[0] is None
    monkeypatch.setattr(bench, "PROFILE_TRAFFIC", str(tmp_path / "absent.json"))
    assert bench.traffic_for("gemm_wgrad_gu", "sweep_zipf1")[0] is None


def test_the_timed_step_keeps_its_workload_name_for_the_counter_lookup():
    """The per-kernel loop of the timed step once reused the variable holding the workload's name,
    so the stored counters were looked up under a kernel's name and never found: nothing in the
    function may rebind it."""
    import ast
    tree = ast.parse(open(os.path.join(ROOT, "bench.py")).read())
    fn = next(n for n in ast.walk(tree) if isinstance(n, ast.FunctionDef) and n.name == "ours")
    assert "name" in [a.arg for a in fn.args.args]
    rebound = [n.lineno for n in ast.walk(fn) if isinstance(n, ast.Name) and n.id == "name"
               and isinstance(n.ctx, ast.Store)]
    assert rebound == []
