"""The bench's host-side arithmetic and bookkeeping, without a GPU: the clock
record (throttle reasons must surface, samples outside the timed region must
not count), whole-job throughput, and the lookup of recorded DRAM traffic
(null once the kernel sources change)."""
import bench

CLEAN = "2070, 2070, 160.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active"


def sample(sm=2070, reasons=()):
    cols = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    flags = ["Active" if c in reasons else "Not Active" for c in cols]
    return f"{sm}, 2070, 300.0, 0x1, " + ", ".join(flags)


def test_clean_run():
    s = bench.summarize_clocks([(10.0, CLEAN), (10.05, CLEAN)], (9.99, 10.06))
    assert s["reasons"] == [] and s["sm_mhz"] == 2070 and s["samples_in_timed_region"] == 2


def test_throttle_reasons_surface():
    lines = [(10.0, sample(reasons=("hw_slowdown",))), (10.05, sample(reasons=("sw_power_cap",)))]
    s = bench.summarize_clocks(lines, (9.99, 10.06))
    assert s["reasons"] == ["hw_slowdown", "sw_power_cap"]


def test_only_the_timed_region_counts():
    lines = [(5.0, sample(sm=900, reasons=("hw_thermal_slowdown",))),  # long before
             (10.0, sample(sm=2070)), (10.02, sample(sm=2050)),
             (20.0, sample(sm=1000, reasons=("sw_thermal_slowdown",)))]  # long after
    s = bench.summarize_clocks(lines, (9.99, 10.03))
    assert s["reasons"] == [] and s["sm_mhz"] == 2060 and s["samples_in_timed_region"] == 2


def test_sample_printed_just_after_the_region_counts():
    s = bench.summarize_clocks([(10.08, sample(reasons=("hw_slowdown",)))], (9.9, 10.0))
    assert s["reasons"] == ["hw_slowdown"] and s["samples_in_timed_region"] == 1


def test_short_region_takes_the_nearest_samples():
    lines = [(t, sample(sm=2000 + i)) for i, t in enumerate([1.0, 2.0, 3.0, 4.0, 5.0, 6.0, 7.0])]
    s = bench.summarize_clocks(lines, (4.4, 4.41))
    assert s["samples"] == 4 and s["samples_in_timed_region"] == 0
    assert s["sm_mhz"] == 2003.5  # samples at 3, 4, 5, 6 s


def test_malformed_lines_are_skipped():
    assert bench.summarize_clocks([(1.0, "[N/A]"), (1.0, "garbage, x")], (0.0, 2.0)) is None
    s = bench.summarize_clocks([(1.0, "N/A, 2070, 1, 2, a, b, c, d"), (1.1, CLEAN)], (0.0, 2.0))
    assert s["samples"] == 1


def test_job_throughput():
    # 2 ranks x 10 steps x 1e12 FLOP in 4 ms (slowest rank): 5000 TFLOP/s
    assert abs(bench.job_throughput(2, 10, 10**12, 4.0) - 5000.0) < 1e-9


def test_recorded_traffic_follows_the_source_hash(monkeypatch):
    got = bench.recorded_traffic("dense_b1_n4096_h32_d128")
    assert got is None or got > 0
    assert bench.recorded_traffic("no_such_workload") is None
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0" * 16)
    assert bench.recorded_traffic("dense_b1_n4096_h32_d128") is None
