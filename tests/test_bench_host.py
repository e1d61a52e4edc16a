"""Host-side pieces of bench.py that shape its JSON line, checked on CPU: the clock summary
read from nvidia-smi samples, and the recorded ncu traffic, which counts only while the kernel
sources it was taken from are unchanged."""
import json
import os

import bench


def _sampler_with(lines):
    s = bench.ClockSampler(0)
    s.proc = object()   # a sampler that ran: summary() reads its file
    with open(s.path, "w") as f:
        f.write("\n".join(lines) + "\n")
    return s


def test_clock_summary_median_of_busy_samples_and_reasons():
    idle = "0, 345, 2070, 120.0, 0x1, Not Active, Not Active, Not Active, Not Active"
    busy = "0, {mhz}, 2070, 1100.0, 0x0, Not Active, Not Active, Not Active, {cap}"
    lines = [idle, busy.format(mhz=2070, cap="Not Active"), busy.format(mhz=2055, cap="Active"),
             busy.format(mhz=2070, cap="Not Active"), "garbage line", idle]
    s = _sampler_with(lines)
    out = s.summary()
    assert out["sm_mhz"] == 2070.0            # idle samples (< half the peak) are left out
    assert out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["sw_power_cap"]
    assert out["samples"] == 5
    assert not os.path.exists(s.path)         # the sample file is removed after reading


def test_clock_summary_reports_throttle_reasons():
    row = "0, 1500, 2070, 1390.0, 0x8, Not Active, Active, Not Active, Active"
    out = _sampler_with([row, row]).summary()
    assert out["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]
    assert out["sm_mhz"] == 1500.0


def test_clock_summary_without_sampler():
    s = bench.ClockSampler(0)
    assert s.summary()["reasons"] == ["nvidia-smi unavailable"]


def test_recorded_traffic_only_while_sources_unchanged(tmp_path, monkeypatch):
    src = tmp_path / "k.cu"
    src.write_text("__global__ void k() {}\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    rec = {"kernels": {"dequant/q6": {"bytes_per_launch": 1234, "sources": ["k.cu"],
                                      "source_sha256": bench.kernel_source_hash(["k.cu"])}}}
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "dram_traffic.json").write_text(json.dumps(rec))
    assert bench.recorded_traffic("dequant", 6) == 1234
    assert bench.recorded_traffic("dequant", 8) is None        # no record for this width
    src.write_text("__global__ void k() { /* changed */ }\n")
    assert bench.recorded_traffic("dequant", 6) is None        # stale: the kernel changed
    src.unlink()
    assert bench.recorded_traffic("dequant", 6) is None        # a listed source is missing


def test_committed_traffic_records_name_existing_sources():
    with open(os.path.join(bench.ROOT, "profiles", "dram_traffic.json")) as f:
        rec = json.load(f)
    for name, e in rec["kernels"].items():
        assert e["bytes_per_launch"] > 0, name
        for rel in e["sources"]:
            assert os.path.exists(os.path.join(bench.ROOT, rel)), (name, rel)
