"""The bench's clock sampler on CPU, with a stand-in for nvidia-smi.

The sampler must start the timed region only once samples are flowing, count
only the samples taken inside the region, and report throttle reasons that were
active there.
"""
import os
import stat
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# one CSV row every 40 ms in the bench's field order: index, clocks.sm, clocks.max.sm,
# power.draw, active reasons, then hw_slowdown, hw_thermal, sw_thermal, sw_power_cap
_FAKE = """#!{py}
import sys, time
i = 0
while True:
    idle = i == 0
    mhz = 900 if idle else 2070
    cap = "Not Active" if idle or {cap_off} else "Active"
    print(f"0, {{mhz}}, 2070, 700.0, 0x4, Not Active, Not Active, Not Active, {{cap}}", flush=True)
    i += 1
    time.sleep(0.04)
"""


def _sampler(tmp_path, monkeypatch, cap_off=True):
    tool = tmp_path / "nvidia-smi"
    tool.write_text(_FAKE.format(py=sys.executable, cap_off=cap_off))
    tool.chmod(tool.stat().st_mode | stat.S_IXUSR)
    monkeypatch.setenv("PATH", f"{tmp_path}{os.pathsep}{os.environ['PATH']}")
    sys.path.insert(0, ROOT)
    import bench
    return bench.ClockSampler(0)


def test_samples_before_the_region_are_dropped(tmp_path, monkeypatch):
    with _sampler(tmp_path, monkeypatch) as clk:
        assert clk.skip >= 1        # the idle first sample was written before the region
        time.sleep(0.3)
    s = clk.summary()
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == [] and s["samples"] >= 3


def test_active_reasons_are_reported(tmp_path, monkeypatch):
    with _sampler(tmp_path, monkeypatch, cap_off=False) as clk:
        time.sleep(0.2)
    assert clk.summary()["reasons"] == ["sw_power_cap"]


def test_no_sampler_means_no_samples(monkeypatch):
    monkeypatch.setenv("PATH", "")
    sys.path.insert(0, ROOT)
    import bench
    with bench.ClockSampler(0) as clk:
        pass
    assert clk.summary() == dict(sm_mhz=None, sm_max_mhz=None, reasons=["no samples"], samples=0)
