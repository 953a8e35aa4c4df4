"""Host-side logic of bench.py (no GPU): the clock record, the link between
the committed DRAM-traffic record and the kernel source it was taken on, and
the CPU baseline's report."""
import json
import os
import shutil

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_clock_summary_reports_median_and_active_reasons():
    lines = ["0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
             "0, 1995, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active",
             "0, 2040, 2070, 1200.0, 0x0, Not Active, Not Active, Not Active, Not Active",
             "garbage line", "0, [N/A], 2070, 0, 0x0, Not Active, Not Active, Not Active, x"]
    rec = bench.ClockSampler.summarise(lines)
    assert rec["sm_mhz"] == 2040 and rec["sm_max_mhz"] == 2070 and rec["samples"] == 3
    assert rec["reasons"] == ["sw_power_cap"]
    hot = bench.ClockSampler.summarise(
        ["0, 1500, 2070, 1400, 0x40, Active, Not Active, Active, Not Active"])
    assert hot["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]


def test_traffic_record_follows_the_kernel_source(tmp_path, monkeypatch):
    """The record counts only for the source it was captured on: a copy of the
    tree with the same sources reads it, an edited kernel reads nothing."""
    csrc = os.path.join("latent_causal_attention_gb300", "csrc")
    os.makedirs(tmp_path / csrc)
    os.makedirs(tmp_path / "profiles")
    for name in ("flash_tc.cu", "ptx.cuh"):
        shutil.copy(os.path.join(ROOT, csrc, name), tmp_path / csrc / name)
    rec = json.load(open(os.path.join(ROOT, "profiles", "flash_prefill_traffic.json")))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    import hashlib
    h = hashlib.sha256()
    for name in ("flash_tc.cu", "ptx.cuh"):
        h.update(open(tmp_path / csrc / name, "rb").read())
    rec["source_sha256_16"] = h.hexdigest()[:16]
    (tmp_path / "profiles" / "flash_prefill_traffic.json").write_text(json.dumps(rec))
    assert bench.flash_traffic() == rec["traffic_bytes_per_launch"]
    with open(tmp_path / csrc / "flash_tc.cu", "a") as f:
        f.write("\n// edited\n")
    assert bench.flash_traffic() is None


def test_cpu_baseline_report():
    value, detail = bench.time_oracle(budget_s=0.3, seed_rows=5, literal=True)
    assert value > 0
    assert detail["kind"] == "oracle" and detail["cores"] >= 1 and "rows" in detail["sample"]
    assert detail["literal_form"]["value"] > 0
    _, plain = bench.time_oracle(budget_s=0.3, seed_rows=6, literal=False)
    assert plain["literal_form"] is None


def test_peaks_come_from_the_measured_record_else_the_fallback(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    peaks, kind = bench.load_peaks()                       # no record
    assert kind == "fallback" and peaks["hbm_gbs"] == 6800.0 and peaks["bf16_tflops"] == 1900.0
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6788.3}))
    assert bench.load_peaks()[1] == "fallback"             # incomplete record
    (tmp_path / "MEASURED_PEAKS.json").write_text("not json")
    assert bench.load_peaks()[1] == "fallback"
    (tmp_path / "MEASURED_PEAKS.json").write_text(
        json.dumps({"hbm_gbs": 6788.3, "bf16_tflops": 1909.8, "bf16_tflops_sustained": 1707.2}))
    peaks, kind = bench.load_peaks()
    assert kind == "measured" and peaks["bf16_tflops"] == 1909.8


def test_peaks_record_of_another_gpu_is_not_used(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (tmp_path / "MEASURED_PEAKS.json").write_text(
        json.dumps({"hbm_gbs": 6758.2, "bf16_tflops": 1887.9, "gpu_name": "NVIDIA GB300"}))
    assert bench.load_peaks("NVIDIA GB300")[1] == "measured"
    peaks, kind = bench.load_peaks("NVIDIA B200")
    assert kind.startswith("fallback") and peaks["bf16_tflops"] == 1900.0
    assert bench.load_peaks()[1] == "measured"            # no device to compare with


def test_spec_denominators_are_the_published_figures():
    assert bench.SPEC_PEAKS["hbm_gbs"] == 8000.0
    assert bench.SPEC_PEAKS["bf16_tflops"] == 2250.0 and "sparsity" in bench.SPEC_PEAKS["source"]


def test_oracle_table_covers_every_workload_and_form():
    t = bench.oracle_table(budget_s=0.05)
    assert t["cores"] >= 1 and t["kind"] == "oracle"
    assert set(t["workloads"]) == {"tiny_f32", "proj_f32", "mid_bf16", "prefill_bf16",
                                   "decode_bf16"}
    for name, rec in t["workloads"].items():
        for form in ("literal", "absorbed", "explicit"):
            assert rec[form]["seconds_full"] > 0 and rec[form]["mode"] in ("full", "sampled")
    assert t["workloads"]["tiny_f32"]["literal"]["mode"] == "full"
    assert set(t["single_core"]) == {"tiny_f32", "proj_f32", "mid_bf16"}
