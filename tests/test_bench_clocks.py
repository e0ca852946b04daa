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


def test_sampler_names_the_gpu_it_was_given(tmp_path, monkeypatch):
    """The sampler passes nvidia-smi the id it was given (a UUID), not a CUDA
    ordinal, which nvidia-smi would read in its own (PCI) numbering."""
    log = tmp_path / "args.txt"
    exe = tmp_path / "nvidia-smi"
    exe.write_text(f"#!/bin/sh\necho \"$@\" > {log}\necho '{ROWS[0]}'\nexec sleep 30\n")
    exe.chmod(exe.stat().st_mode | stat.S_IXUSR)
    monkeypatch.setenv("PATH", str(tmp_path) + os.pathsep + os.environ["PATH"])
    c = bench.Clocks("GPU-7aebdb66-0000-4d0a-8503-96f012cef09c")
    time.sleep(0.5)
    c.stop()
    args = log.read_text().split()
    assert args[args.index("-i") + 1] == "GPU-7aebdb66-0000-4d0a-8503-96f012cef09c"


class _Props:
    def __init__(self, **kw):
        self.__dict__.update(kw)


def test_gpu_id_prefers_uuid_then_pci_bus(monkeypatch):
    import torch
    monkeypatch.setattr(torch.cuda, "get_device_properties",
                        lambda i: _Props(uuid="7aebdb66-67b0-4d0a-8503-96f012cef09c"))
    assert bench.smi_gpu_id(3) == "GPU-7aebdb66-67b0-4d0a-8503-96f012cef09c"
    monkeypatch.setattr(torch.cuda, "get_device_properties",
                        lambda i: _Props(uuid="GPU-abc", pci_bus_id=7))
    assert bench.smi_gpu_id(0) == "GPU-abc"
    monkeypatch.setattr(torch.cuda, "get_device_properties",
                        lambda i: _Props(pci_domain_id=0, pci_bus_id=0x1b, pci_device_id=0))
    assert bench.smi_gpu_id(0) == "00000000:1b:00.0"

    def boom(i):
        raise RuntimeError("no device")
    monkeypatch.setattr(torch.cuda, "get_device_properties", boom)
    assert bench.smi_gpu_id(5) == "5"


def test_host_description_and_numa_helpers():
    h = bench.host_info()
    assert h["nproc"] == os.cpu_count() and h["cpu_model"] and h["numa_nodes"] >= 1
    nodes = bench.cpu_numa_nodes()
    assert nodes and all(isinstance(n, int) for n in nodes)
    with bench.numa_bind(None) as bound:        # the default policy: nothing to bind
        assert bound is False
    import torch
    t = torch.empty(1 << 16, dtype=torch.uint8)
    t.fill_(1)
    assert bench.page_node(t.data_ptr()) in [-1] + nodes


def test_default_run_covers_the_four_roofline_workloads():
    a = bench.parse([])
    names = [a.workload] + [x for x in a.workloads.split(",") if x]
    assert names == ["llama3_8b_decode", "long_ctx_predict", "wide_budget", "fragmentation"]
    assert a.warmup >= 3
