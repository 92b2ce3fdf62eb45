"""Clock bookkeeping of bench.py on the host: how NVML and nvidia-smi samples
are merged into the line's `clocks` object (no GPU, no NVML needed)."""
import os

import bench


def _sampler(lines, nvml_samples, max_mhz=2070.0):
    c = bench.ClockSampler(0)
    c.lines = lines
    c.nvml_samples = nvml_samples

    class FakeNvml:
        pass

    c.nvml = FakeNvml()
    c.nvml.max_mhz = max_mhz
    return c


def test_unsampled_when_nothing_read():
    c = bench.ClockSampler(0)
    assert c.summary()["reasons"] == ["unsampled"]


def test_idle_nvml_samples_left_out_and_reasons_merged():
    smi = ["0, 1700, 2070, 1300.0, 0x4, Not Active, Not Active, Not Active, Active"]
    nv = [(2070.0, 0x1), (1650.0, 0x4 | 0x8), (1690.0, 0x0)]
    s = _sampler(smi, nv).summary()
    assert s["samples"] == 3
    assert s["sm_mhz"] == 1690.0
    assert s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["hw_slowdown", "sw_power_cap"]
    assert s["sources"] == {"nvml_2ms": 2, "nvidia_smi_200ms": 1}


def test_all_idle_samples_still_reported():
    s = _sampler([], [(345.0, 0x1), (345.0, 0x1)]).summary()
    assert s["samples"] == 2 and s["sm_mhz"] == 345.0


def test_thermal_reasons_from_nvidia_smi():
    smi = ["0, 1500, 2070, 900.0, 0x60, Not Active, Active, Active, Not Active"]
    s = _sampler(smi, []).summary()
    assert s["reasons"] == ["hw_thermal_slowdown", "sw_thermal_slowdown"]


def test_visible_devices_renumbering(monkeypatch):
    monkeypatch.setenv("CUDA_VISIBLE_DEVICES", "5,3")
    assert bench._smi_index(0) == 5 and bench._smi_index(1) == 3
    monkeypatch.setenv("CUDA_VISIBLE_DEVICES", "GPU-abc")
    assert bench._smi_index(1) == 1
    monkeypatch.delenv("CUDA_VISIBLE_DEVICES")
    assert bench._smi_index(2) == 2
