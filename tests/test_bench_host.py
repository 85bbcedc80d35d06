"""Host-side helpers behind the benchmark's JSON line (no GPU)."""

import re

import bench


def test_clock_summary_median_max_and_reasons():
    # index, clocks.sm, clocks.max.sm, power.draw, reasons bitmask, then the
    # hw_slowdown, hw_thermal_slowdown, sw_thermal_slowdown, sw_power_cap flags
    text = "\n".join([
        "0, 2070, 2070, 900.1, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "0, 1980, 2070, 1390.5, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 2070, 2070, 950.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
        "0, [N/A], 2070, 0, 0x0, Not Active, Not Active, Not Active, Not Active",
    ])
    c = bench.summarize_clocks(text)
    assert c["samples"] == 3
    assert c["sm_mhz"] == 2070.0
    assert c["sm_max_mhz"] == 2070.0
    assert c["reasons"] == ["sw_power_cap"]


def test_clock_summary_flags_thermal_and_hw_slowdown():
    text = "0, 1200, 2070, 1400, 0x48, Active, Not Active, Active, Not Active"
    c = bench.summarize_clocks(text)
    assert c["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]
    assert bench.summarize_clocks("")["sm_mhz"] is None


def test_profiled_traffic_is_tied_to_the_kernel_sources(monkeypatch):
    """roofline.traffic comes from the committed ncu summary only while the
    kernel sources still hash to the value recorded beside it."""
    text = open(bench.os.path.join(bench.ROOT, "profiles", "paged_decode_qwen3_0p6b_decode.md")).read()
    recorded = float(re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text).group(1))
    src = re.search(r"kernel_source_sha256:\s*([0-9a-f]+)", text).group(1)
    monkeypatch.setattr(bench, "decode_source_hash", lambda sources=None: src)
    assert bench.profiled_traffic("qwen3_0p6b_decode") == recorded
    monkeypatch.setattr(bench, "decode_source_hash", lambda sources=None: "0" * 16)
    assert bench.profiled_traffic("qwen3_0p6b_decode") is None
    assert bench.profiled_traffic("no_such_workload") is None

