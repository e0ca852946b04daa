"""The benchmark's clock sampler against a fake nvidia-smi (no GPU): the median
SM clock and every throttle reason seen active during the timed region must
reach the JSON line, since a run that saw a hardware or thermal slowdown is
rejected on them."""
import os
import stat
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

ROWS = [
    "0, 2070, 2070, 910.2, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
    "0, 1980, 2070, 1399.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
    "0, 2070, 2070, 1120.7, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
    "0, [N/A], 2070, 0, 0x0, Not Active, Not Active, Not Active, Not Active",
]


def _fake_smi(tmp_path, rows):
    exe = tmp_path / "nvidia-smi"
    body = "\n".join(f"echo '{r}'" for r in rows)
    exe.write_text(f"#!/bin/sh\n{body}\nexec sleep 30\n")
    exe.chmod(exe.stat().st_mode | stat.S_IXUSR)
    return str(tmp_path)


def test_median_clock_and_reasons(tmp_path, monkeypatch):
    monkeypatch.setenv("PATH", _fake_smi(tmp_path, ROWS) + os.pathsep + os.environ["PATH"])
    c = bench.Clocks(0)
    time.sleep(0.5)
    out = c.stop()
    assert out["samples"] == 3                  # the [N/A] row is skipped
    assert out["sm_mhz"] == 2070.0 and out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["sw_power_cap"]


def test_thermal_slowdown_is_reported(tmp_path, monkeypatch):
    rows = ["0, 1500, 2070, 1300.0, 0x40, Active, Not Active, Active, Not Active"]
    monkeypatch.setenv("PATH", _fake_smi(tmp_path, rows) + os.pathsep + os.environ["PATH"])
    c = bench.Clocks(0)
    time.sleep(0.5)
    out = c.stop()
    assert out["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]
    assert out["sm_mhz"] == 1500.0


def test_missing_tool(tmp_path, monkeypatch):
    monkeypatch.setenv("PATH", str(tmp_path))  # an empty directory: no nvidia-smi
    out = bench.Clocks(0).stop()
    assert out["reasons"] == ["nvidia-smi unavailable"]
