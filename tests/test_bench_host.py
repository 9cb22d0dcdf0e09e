"""Host-side pieces of bench.py (no GPU): the clocks summary that vets a
timed run, and the algorithmic byte counts the roofline divides by."""
import os
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402
from speculative_decoding_eagle_gb300 import workloads as W  # noqa: E402


def _clocks(lines):
    c = bench.Clocks(0)
    c.lines = lines
    return c.summary()


def test_clocks_summary_median_and_reasons():
    s = _clocks(["0, 2070, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Not Active",
                 "0, 1980, 2070, 1100.0, 0x4, Not Active, Not Active, Not Active, Active",
                 "0, 2070, 2070, 950.0, 0x0, Not Active, Not Active, Not Active, Not Active"])
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0 and s["samples"] == 3
    assert s["reasons"] == ["sw_power_cap"]


def test_clocks_summary_flags_thermal_and_skips_garbage():
    s = _clocks(["garbage", "0, [N/A], 2070, 0, 0x0, Not Active, Not Active, Not Active, Not Active",
                 "0, 1500, 2070, 1300.0, 0x40, Active, Active, Not Active, Not Active"])
    assert s["samples"] == 1 and s["sm_mhz"] == 1500.0
    assert s["reasons"] == ["hw_slowdown", "hw_thermal_slowdown"]


def test_clocks_summary_without_samples():
    assert _clocks([])["reasons"] == ["unavailable"]


def test_clocks_without_nvidia_smi_or_csv(tmp_path):
    path = tmp_path / "clk.csv"
    with bench.Clocks(0, str(path)) as c:
        pass
    assert "reasons" in c.summary() and path.exists()


@pytest.mark.parametrize("name,prefix,want", [("llama2-7b", 1024, 18_776_064), ("llama2-13b", 4096, 86_384_640),
                                              ("llama2-70b", 8192, 36_540_416)])
def test_attention_bytes(name, prefix, want):
    """K/V prefix + tree K/V + Q + O per launch at batch 1."""
    wl = W.WORKLOADS[name]
    assert bench.attention_bytes(wl, [prefix]) == want


def test_step_spread_percentiles():
    s = bench.step_spread([0.5, 0.1, 0.4, 0.2, 0.3])  # order does not matter
    assert s == {"median_ms": 0.3, "p10_ms": 0.14, "p90_ms": 0.46}
    assert bench.step_spread([0.089] * 7) == {"median_ms": 0.089, "p10_ms": 0.089, "p90_ms": 0.089}
    assert bench.step_spread([])["median_ms"] is None


def test_recorded_attention_traffic_matches_the_kernel_sources():
    """The bench reports the attention kernel's DRAM traffic only while the
    committed ncu summary was taken on the same sources; the headline
    workload's summary must be current."""
    assert bench.recorded_attention_traffic("llama2-7b", 1, 1024) is not None
    assert bench.recorded_attention_traffic("llama2-7b", 1, 999) is None


def test_extras_child_failure_becomes_error_entries(monkeypatch):
    """The default bench runs its secondary sections in a child process; a child that fails (here: a command
    that exits non-zero at once) must leave an error entry in each section, not end the bench."""
    import types

    def fake_run(cmd, capture_output, text, timeout, env):
        assert "--extras" in cmd
        return types.SimpleNamespace(returncode=3, stdout="", stderr="CUDA error: unspecified launch failure")

    monkeypatch.setattr(bench.subprocess, "run", fake_run)
    ex = bench.run_extras_child(types.SimpleNamespace(steps=10))
    for key in ("tree_attention_shapes", "tree_attention_batched", "sweep_step"):
        assert ex[key] and "error" in ex[key][0] and "exited 3" in ex[key][0]["error"]


def test_extras_child_result_is_merged(monkeypatch):
    import json
    import types
    line = json.dumps({"tree_attention_shapes": [{"us_per_launch": 1.0}], "tree_attention_batched": [],
                       "sweep_step": [{"batch": 32}]})

    def fake_run(cmd, capture_output, text, timeout, env):
        return types.SimpleNamespace(returncode=0, stdout="noise\n" + line + "\n", stderr="")

    monkeypatch.setattr(bench.subprocess, "run", fake_run)
    ex = bench.run_extras_child(types.SimpleNamespace(steps=10))
    assert ex["tree_attention_shapes"] == [{"us_per_launch": 1.0}] and ex["sweep_step"] == [{"batch": 32}]
