"""Host logic of bench.py on the CPU: the FLOP count of the metric, the clock
summary that decides whether a timed run is kept, and the gate that reports
profiled DRAM traffic only for the kernel sources it was captured on."""
import json
import os

import bench


def test_flops_follow_the_metric_convention():
    w = {"B": 2, "H": 16, "N": 8192, "d": 128, "causal": False}
    assert bench.flops(w) == 4.0 * 2 * 16 * 8192 ** 2 * 128
    assert bench.flops(dict(w, causal=True)) == bench.flops(w) / 2   # halved, not N(N+1)/2


def _sampler(lines=(), tuples=()):
    """A sampler with no polling thread: nvidia-smi CSV lines (time, line) and
    NVML-style samples (time, sm, max, power, reasons)."""
    s = object.__new__(bench.ClockSampler)
    s.samples = list(tuples)
    s.proc = None
    s.source = "test"
    for ts, line in lines:
        s.add_smi_line(ts, line)
    return s


def test_clock_summary_median_window_and_reasons():
    row = lambda sm, *r: ", ".join([str(sm), "2070", "900.0", *r])
    idle = ["Not Active"] * 4
    lines = [(0.5, row(600, *idle)),                                    # before the window
             (1.0, row(1950, *idle)), (1.1, row(1965, *idle)),
             (1.2, row(1980, "Not Active", "Not Active", "Not Active", "Active")),
             (5.0, row(2070, "Active", "Not Active", "Not Active", "Not Active"))]  # after
    got = _sampler(lines).summary(1.0, 2.0)
    assert got["sm_mhz"] == 1965.0 and got["sm_max_mhz"] == 2070.0 and got["sm_min_mhz"] == 1950.0
    assert got["reasons"] == ["sw_power_cap"] and got["samples"] == 3 and got["power_w_max"] == 900.0
    hot = _sampler([(1.0, row(1900, "Active", "Not Active", "Active", "Not Active"))]).summary(0.0, 2.0)
    assert hot["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]


def test_clock_summary_from_nvml_samples():
    t = [(1.0, 2070.0, 2070.0, 800.0, set()), (1.002, 2055.0, 2070.0, 1300.0, {"sw_power_cap"}),
         (1.004, 2040.0, 2070.0, None, set()), (3.0, 900.0, 2070.0, 100.0, {"hw_slowdown"})]
    got = _sampler(tuples=t).summary(0.9, 1.01)
    assert got["samples"] == 3 and got["sm_mhz"] == 2055.0 and got["power_w_max"] == 1300.0
    assert got["reasons"] == ["sw_power_cap"]


def test_nvml_reason_bits():
    assert bench.REASON_BITS["sw_power_cap"] == 0x4 and bench.REASON_BITS["hw_slowdown"] == 0x8
    assert bench.REASON_BITS["sw_thermal_slowdown"] == 0x20 and bench.REASON_BITS["hw_thermal_slowdown"] == 0x40


def test_clock_summary_without_samples_and_with_garbage():
    assert _sampler().summary(0.0, 1.0)["samples"] == 0
    bad = [(0.5, "[N/A], 2070, x, Not Active, Not Active, Not Active, Not Active"),
           (0.6, "1900")]                                               # short line
    got = _sampler(bad).summary(0.0, 1.0)
    assert got["samples"] == 0 and got["sm_mhz"] is None and got["reasons"] == []


def test_profile_traffic_only_for_the_sources_it_was_taken_on(tmp_path, monkeypatch):
    with open(bench.PROFILE_JSON) as f:
        prof = json.load(f)
    current = tmp_path / "current.json"
    current.write_text(json.dumps(dict(prof, kernel_source_sha256=bench.kernel_source_sha256())))
    monkeypatch.setattr(bench, "PROFILE_JSON", str(current))
    assert bench.traffic_from_profile() == prof["dram_bytes_per_launch_full_workload"]
    stale = tmp_path / "stale.json"
    stale.write_text(json.dumps(dict(prof, kernel_source_sha256="0" * 64)))
    monkeypatch.setattr(bench, "PROFILE_JSON", str(stale))
    assert bench.traffic_from_profile() is None
    monkeypatch.setattr(bench, "PROFILE_JSON", os.path.join(str(tmp_path), "missing.json"))
    assert bench.traffic_from_profile() is None
