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



def test_config_selection_by_name_or_index():
    from paged_kv_cache_85_gb300 import workload as wl

    names = wl.CONFIG_NAMES
    assert bench.config_index(None, names, bench.DECODE_WORKLOAD) == names.index("max_concurrency")
    assert bench.config_index("vllm_bs16_8b_heads", names, "max_concurrency") == 2
    assert bench.config_index("1", names, "max_concurrency") == 1
    import pytest

    with pytest.raises(SystemExit):
        bench.config_index("no_such", names, "max_concurrency")
    with pytest.raises(SystemExit):
        bench.config_index("9", names, "max_concurrency")


def test_decode_config_describes_the_drawn_workload():
    """`config` comes from the workload itself (both arms print the same
    object), including its context-length distribution and padding slots."""
    from paged_kv_cache_85_gb300 import workload as wl

    w = wl.config_workload(0)
    cfg = bench.decode_config(w, "bf16", 1)
    assert cfg == bench.decode_config(w, "bf16", 1)
    assert cfg["workload"] == "tiny_paged_decode"
    assert cfg["context_lens"]["min"] == 1 and cfg["context_lens"]["max"] == 300
    assert cfg["context_lens"]["total_tokens"] == 1 + 17 + 40 + 300
    assert cfg["padding_slots"] == 0
    assert cfg["step_bytes"] == w.decode_bytes(2) + w.store_bytes(2)
    assert "unique_kv_bytes" not in cfg  # no shared blocks
    assert bench.decode_config(w, "fp8", 1)["kv_bytes"] == w.kv_bytes(1)


def test_unique_bytes_reported_for_shared_prefix_blocks():
    from paged_kv_cache_85_gb300 import workload as wl

    w = wl.make_workload("shared", B=3, Hq=2, Hkv=1, D=64, bs=16, context_lens=[40, 33, 64],
                         shared_prefix_tokens=32, rng=bench.np.random.default_rng(0))
    cfg = bench.decode_config(w, "bf16", 1)
    # 32 shared tokens counted once: 137 logical tokens, 137 - 2 * 32 distinct
    assert cfg["kv_bytes"] == 137 * 64 * 2 * 2
    assert cfg["unique_kv_bytes"] == (137 - 64) * 64 * 2 * 2


def test_cpu_baseline_runs_one_core_and_all_cores(monkeypatch):
    import oracle

    monkeypatch.setattr(oracle, "host_cores", lambda: 6)
    seen = []

    def timer(budget, threads):
        seen.append(threads)
        return {"value": float(threads), "unit": "GB/s", "cores": threads, "kind": "oracle",
                "sample": "fake"}

    top = bench.cpu_baselines(timer, budget_s=0.1)
    assert seen == [1, 6]
    assert top["cores"] == 6 and top["value"] == 6.0 and top["host_cores"] == 6
    assert [r["cores"] for r in top["by_cores"]] == [1, 6]
