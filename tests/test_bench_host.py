"""Host logic of bench.py that needs no GPU: the clock record of the timed
region, the kernel-source hash that keeps committed ncu traffic figures tied
to the code they were taken on, and the peaks the roofline divides by."""
import json
import os
import shutil
import sys

import pytest

ROOT = os.path.abspath(os.path.join(os.path.dirname(__file__), ".."))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

ROW = "0, {sm}, 2070, {pw}, 0x0, {hw}, Not Active, Not Active, {cap}, {lim}"


def _sampler(lines):
    c = bench.ClockSampler(0)
    c.out = "\n".join(lines) + "\n"
    return c.summary()


def test_clock_record_under_load():
    s = _sampler([ROW.format(sm=2070, pw=180.0, hw="Not Active", cap="Not Active", lim="1400.00"),
                  ROW.format(sm=1980, pw=1310.5, hw="Not Active", cap="Active", lim="1400.00"),
                  ROW.format(sm=1950, pw=1320.0, hw="Not Active", cap="Active", lim="1400.00")])
    assert s["samples"] == 3 and s["samples_under_load"] == 2  # 180 W is idle
    assert s["sm_mhz"] == 1965.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]
    assert s["power_w_max"] == 1320.0 and s["power_limit_w"] == 1400.0


def test_clock_record_flags_hardware_slowdown():
    s = _sampler([ROW.format(sm=1200, pw=900.0, hw="Active", cap="Not Active", lim="1400.00")])
    assert s["reasons"] == ["hw_slowdown"]


def test_clock_record_tolerates_missing_power_limit():
    s = _sampler([ROW.format(sm=2070, pw=900.0, hw="Not Active", cap="Not Active", lim="[N/A]")])
    assert s["samples"] == 1 and s["power_limit_w"] is None
    s = _sampler(["0, 2070, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Not Active"])
    assert s["samples"] == 1 and s["power_limit_w"] is None


def test_clock_record_without_samples():
    s = _sampler(["garbage", ""])
    assert s["samples"] == 0 and s["reasons"] == ["no samples"]


def _copy_tree(tmp_path):
    for sub in ("normalization_gemm_tcgen05_gb300/csrc", "profiles"):
        shutil.copytree(os.path.join(ROOT, sub), os.path.join(tmp_path, sub))
    return str(tmp_path)


def test_kernel_hash_ignores_comments_but_not_code(tmp_path, monkeypatch):
    root = _copy_tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", root)
    h0 = bench.kernel_source_hash()
    assert h0 == bench.kernel_source_hash()
    path = os.path.join(root, "normalization_gemm_tcgen05_gb300", "csrc", bench.KERNEL_SOURCES[0])
    with open(path, "a") as f:
        f.write("\n   // a comment line\n\n")
    assert bench.kernel_source_hash() == h0
    with open(path, "a") as f:
        f.write("namespace fnorm { constexpr int kProbe = 1; }\n")
    assert bench.kernel_source_hash() != h0


def test_traffic_is_null_once_the_kernels_change(tmp_path, monkeypatch):
    root = _copy_tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", root)
    with open(os.path.join(root, "profiles", "ncu_traffic.json")) as f:
        table = json.load(f)
    name = "cfg2_n128"
    if table[name]["kernel_source_hash"] != bench.kernel_source_hash():
        pytest.skip("committed traffic figures were taken on other kernel sources")
    assert bench.load_traffic(name) == table[name]["bytes_per_launch"]
    assert bench.load_traffic("no such workload") is None
    path = os.path.join(root, "normalization_gemm_tcgen05_gb300", "csrc", bench.KERNEL_SOURCES[0])
    with open(path, "a") as f:
        f.write("namespace fnorm { constexpr int kProbe = 2; }\n")
    assert bench.load_traffic(name) is None


def test_peaks_prefer_the_measured_file(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.load_peaks()["source"] == "fallback"
    with open(os.path.join(tmp_path, "MEASURED_PEAKS.json"), "w") as f:
        json.dump({"hbm_gbs": 1.0, "bf16_tflops": 2.0}, f)
    p = bench.load_peaks()
    assert p == {"hbm_gbs": 1.0, "bf16_tflops": 2.0, "bf16_tflops_sustained": 2.0, "source": "measured"}
