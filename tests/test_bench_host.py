"""Host-side pieces of bench.py on CPU: the clock-sample summary that flags
throttling, the profile lookups that feed `roofline.traffic` (valid only
while the kernel sources hash as they did when the counters were taken), and
the reference arm's per-step sample budget."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _summary(lines):
    c = bench.ClockSampler(0)
    c.out = "\n".join(lines)
    return c.summary()


def test_clock_summary_steady():
    s = _summary(["2070, 2070, 900.5, Not Active, Not Active, Not Active, Not Active"] * 4
                 + ["2055, 2070, 910.0, Not Active, Not Active, Not Active, Not Active"])
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == [] and s["samples"] == 5


def test_clock_summary_names_each_reason():
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for k, name in enumerate(names):
        flags = ["Not Active"] * 4
        flags[k] = "Active"
        s = _summary(["1500, 2070, 1400.0, " + ", ".join(flags),
                      "2070, 2070, 900.0, Not Active, Not Active, Not Active, Not Active"])
        assert s["reasons"] == [name]
        assert s["sm_mhz"] == (1500.0 + 2070.0) / 2


def test_clock_summary_skips_malformed_lines_and_reports_no_samples():
    s = _summary(["", "[N/A], [N/A], [N/A], x, y", "not, a, number, Active, Active, Active, Active"])
    assert s["sm_mhz"] is None and s["reasons"] == ["no samples"]


def test_profile_traffic_follows_the_kernel_sources(monkeypatch):
    gu = bench.profile_fields(os.path.join(ROOT, bench.GATEUP_PROFILE_NAME))
    ch = bench.profile_fields(os.path.join(ROOT, bench.CHAIN_PROFILE_NAME))
    if gu.get("source_sha256_16") == bench.kernel_sources_hash(bench.GEMV_SOURCES):
        assert bench.gateup_traffic() == int(gu["traffic_bytes_per_launch"])
    else:
        assert bench.gateup_traffic() is None
    if ch.get("source_sha256_16") == bench.kernel_sources_hash(bench.CHAIN_SOURCES):
        assert bench.chain_traffic(32) == 32 * int(ch["traffic_bytes_per_layer"])
    # any change to the hashed sources makes both lookups null
    monkeypatch.setattr(bench, "kernel_sources_hash", lambda files: "0" * 16)
    assert bench.gateup_traffic() is None
    assert bench.chain_traffic(32) is None


def test_job_throughput_counts_every_rank():
    # 2 ranks x 4.41 GB x 10 steps in 11.66 ms (the slowest rank)
    v = bench.job_throughput(2, 4_410_310_656, 10, 11.66)
    assert abs(v - 2 * 4_410_310_656 * 10 / 11.66e-3 / 1e9) < 1e-6


def test_reference_step_budget_bounds_the_whole_run(monkeypatch):
    monkeypatch.delenv("QX_REF_STEP_S", raising=False)
    monkeypatch.delenv("QX_REF_TOTAL_S", raising=False)
    assert bench.reference_step_budget(1) == 2.0 and bench.reference_step_budget(45) == 2.0
    for steps in (46, 100, 500, 10000):
        b = bench.reference_step_budget(steps)
        assert b < 2.0 and abs(b * steps - 90.0) < 1e-9
    assert bench.reference_step_budget(0) == 2.0
