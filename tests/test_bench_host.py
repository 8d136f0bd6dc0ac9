"""Host logic of bench.py on CPU: algorithmic byte counts, the traffic record
tied to the GEMM source hash, argument defaults, the clock-record parser, the
peak fallback and the reference arm's JSON line (the CPU oracle arm runs
here as it does on the GPU machine)."""
import io
import json
import os
import sys
import tempfile
from contextlib import redirect_stdout

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from nvfp4_quantized_linear_gb300 import synthetic as syn  # noqa: E402


def test_algorithmic_bytes():
    gate_up = [p for p in syn.llama([8192]) if p.name == "gate_up"][0]
    # packed A + A scales + packed B + B scales + bf16 output
    assert bench.gemm_bytes(gate_up) == 8192 * 2048 + 8192 * 256 + 28672 * 2048 + 28672 * 256 + 2 * 8192 * 28672
    assert bench.gemm_bytes(gate_up) == 554_696_704
    # K = 4104 pads to 4128: 258 scale columns, padded to 260; rows pad to 128
    assert bench.quant_bytes(1, 4104) == 2 * 4104 + 4128 // 2 + 128 * 260
    assert bench.quant_bytes(8192, 4096) == int(8192 * 4096 * 2.5625)


def test_recorded_traffic_follows_the_gemm_source_hash(monkeypatch, tmp_path):
    f = tmp_path / "traffic.txt"
    f.write_text(f"# comment: with a colon\ngemm_source_hash: {bench.gemm_source_hash()}\n"
                 "dram_bytes_per_launch: 123456\n")
    monkeypatch.setattr(bench, "PROFILE_TRAFFIC", str(f))
    assert bench.recorded_traffic() == 123456.0
    f.write_text("gemm_source_hash: 0000000000000000\ndram_bytes_per_launch: 123456\n")
    assert bench.recorded_traffic() is None                     # taken on another GEMM source
    monkeypatch.setattr(bench, "PROFILE_TRAFFIC", str(tmp_path / "missing.txt"))
    assert bench.recorded_traffic() is None


def test_committed_traffic_record_is_readable():
    """The committed ncu traffic summary names the GEMM source it was taken on
    and the bytes per launch (bench.py reports it only while that source is
    current)."""
    rec = bench.read_traffic_record()
    assert rec is not None, f"{bench.PROFILE_TRAFFIC} missing or unreadable"
    assert len(rec[0]) == 16 and rec[1] > 0


def test_argument_defaults_and_warmup_floor():
    a = bench.parse_args([])
    assert (a.gpus, a.steps, a.warmup, a.impl, a.workload, a.m, a.suite, a.case) == \
        (1, 100, 5, "ours", "qwen", 16384, False, None)
    assert bench.parse_args(["--workload", "llama"]).m == 8192
    assert bench.parse_args(["--warmup", "1"]).warmup == 3                  # at least 3 warm-up steps
    c = bench.parse_args(["--case", "quant", "--m", "64", "--k", "512", "--bs", "16"])
    assert (c.case, c.m, c.k, c.bs) == ("quant", 64, 512, 16)


def test_clock_record_parser():
    s = bench.ClockSampler(0)
    s.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
    s.file.write("0, 300, 2070, 120.5, 0x0, Not Active, Not Active, Not Active, Not Active\n"
                 "0, 2070, 2070, 850.0, 0x4, Not Active, Not Active, Not Active, Active\n"
                 "0, 2055, 2070, 900.1, 0x4, Not Active, Not Active, Not Active, Active\n"
                 "garbage line\n")
    s.file.flush()
    out = s.summary()
    assert out["sm_max_mhz"] == 2070.0
    assert out["sm_mhz"] == pytest.approx(2062.5)                           # median of the loaded samples
    assert out["reasons"] == ["sw_power_cap"]
    assert out["power_w_max"] == 900.1 and out["samples"] == 3


def test_peak_fallback(monkeypatch, tmp_path):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    peaks, src = bench.load_peaks()
    assert peaks == bench.FALLBACK_PEAKS and "fallback" in src
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps(
        {"hbm_gbs": 6794.5, "bf16_tflops": 1903.5, "bf16_tflops_sustained": 1700.2, "other": 1}))
    peaks, src = bench.load_peaks()
    assert peaks["bf16_tflops_sustained"] == 1700.2 and "measured" in src


def test_reference_arm_json_line():
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3"])
    line = buf.getvalue().strip().splitlines()
    assert len(line) == 1
    d = json.loads(line[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["steps"] == 1 and d["warmup"] == 3
    assert d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == bench.host_cores()
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["metric"] == bench.METRIC


def test_cpu_list_parser():
    """sysfs CPU lists (the GPU's local_cpulist) as sets of CPU numbers."""
    assert bench._cpu_list("0-3,8,10-11\n") == {0, 1, 2, 3, 8, 10, 11}
    assert bench._cpu_list("5") == {5}
    assert bench._cpu_list("") == set()
