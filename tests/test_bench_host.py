"""Host-side pieces of bench.py that need no GPU: the clock sampler, driven
by a stand-in nvidia-smi that prints canned samples."""
import os
import stat
import sys
import time

FAKE = """#!{python}
import sys, time
line = "0, 2070, 2070, 180.5, 0x0000000000000004, Not Active, Not Active, Not Active, Active"
while True:
    print(line, flush=True)
    time.sleep(0.05)
"""


def test_clock_sampler_waits_for_its_first_sample_and_parses(tmp_path, monkeypatch):
    import bench
    tool = tmp_path / "nvidia-smi"
    tool.write_text(FAKE.format(python=sys.executable))
    tool.chmod(tool.stat().st_mode | stat.S_IEXEC)
    monkeypatch.setenv("PATH", f"{tmp_path}{os.pathsep}{os.environ.get('PATH', '')}")
    sampler = bench.ClockSampler(0, str(tmp_path / "clocks.csv"))
    t0 = time.time()
    sampler.wait_first(timeout=10.0)
    assert os.path.getsize(tmp_path / "clocks.csv") > 0 and time.time() - t0 < 10.0
    time.sleep(0.3)
    res = sampler.stop()
    assert res["samples"] >= 2
    assert res["sm_mhz"] == 2070.0 and res["sm_max_mhz"] == 2070.0
    assert res["reasons"] == ["sw_power_cap"] and res["power_w_max"] == 180.5


def test_clock_sampler_without_nvidia_smi(tmp_path, monkeypatch):
    import bench
    monkeypatch.setenv("PATH", str(tmp_path))  # no nvidia-smi here
    sampler = bench.ClockSampler(0, str(tmp_path / "clocks.csv"))
    sampler.wait_first(timeout=0.1)
    assert sampler.stop()["reasons"] == ["nvidia-smi unavailable"]
