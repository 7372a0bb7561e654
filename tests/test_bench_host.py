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


def _sampler(samples):
    s = object.__new__(bench.ClockSampler)   # no nvidia-smi process
    s.samples = samples
    s.proc = None
    return s


def test_clock_summary_median_window_and_reasons():
    row = lambda sm, *r: [str(sm), "2070", "900.0", *r]
    idle = ["Not Active"] * 4
    samples = [(0.5, row(600, *idle)),                                  # before the window
               (1.0, row(1950, *idle)), (1.1, row(1965, *idle)),
               (1.2, row(1980, "Not Active", "Not Active", "Not Active", "Active")),
               (5.0, row(2070, "Active", "Not Active", "Not Active", "Not Active"))]  # after
    got = _sampler(samples).summary(1.0, 2.0)
    assert got == {"sm_mhz": 1965.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    hot = _sampler([(1.0, row(1900, "Active", "Not Active", "Active", "Not Active"))]).summary(0.0, 2.0)
    assert hot["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]


def test_clock_summary_without_samples_and_with_garbage():
    assert _sampler([]).summary(0.0, 1.0)["samples"] == 0
    bad = [(0.5, ["[N/A]", "2070", "x", "Not Active", "Not Active", "Not Active", "Not Active"]),
           (0.6, ["1900"])]                                             # short line
    assert _sampler(bad).summary(0.0, 1.0) == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                                               "samples": 0}


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
