"""CPU checks of bench.py's host logic: the clock record, the replica rate and the traffic
figure's source-hash gate."""
import bench


def test_clock_summary_parses_samples_and_reasons():
    c = bench.Clocks(0)
    c.lines = [
        "0, 2070, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 2010, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 2070, 2070, 1000.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "garbled line",
    ]
    s = c.summary()
    assert s["samples"] == 3 and s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]
    c.lines.append("0, 1500, 2070, 800.0, 0x40, Active, Not Active, Not Active, Not Active")
    assert "hw_slowdown" in c.summary()["reasons"]


def test_clock_summary_without_samples():
    s = bench.Clocks(0).summary()
    assert s["samples"] == 0 and s["sm_mhz"] is None and s["reasons"] == []


def test_replica_rate_counts_every_rank():
    # 2 replicas, 1.3 GB each per step, the slowest step 0.25 ms -> 10.4 TB/s of work in all
    assert abs(bench.replica_rate(1.3e9, 2, 0.25) - 2 * 1.3e9 / 0.25e-3) < 1.0


def test_traffic_figure_needs_the_profiled_sources(monkeypatch):
    key, kernel = "paged_decode_qwen3", "paged_decode"
    if bench.profiled_traffic(kernel, key) is None:
        return  # the committed figure was taken on other sources: nothing to gate here
    monkeypatch.setattr(bench, "kernel_source_hash", lambda names: "0000000000000000")
    assert bench.profiled_traffic(kernel, key) is None
