"""Host-side pieces of bench.py that need no GPU: the clock sampler, driven
by a stand-in nvidia-smi that prints canned samples."""
import os
import stat
import sys
import time

FAKE = """#!{python}
import sys, time
open({argv_file!r}, "w").write(" ".join(sys.argv[1:]))
line = "0, 2070, 2070, 180.5, 0x0000000000000004, Not Active, Not Active, Not Active, Active"
while True:
    print(line, flush=True)
    time.sleep(0.05)
"""


def test_clock_sampler_waits_for_its_first_sample_and_parses(tmp_path, monkeypatch):
    import bench
    tool = tmp_path / "nvidia-smi"
    argv_file = str(tmp_path / "argv.txt")
    tool.write_text(FAKE.format(python=sys.executable, argv_file=argv_file))
    tool.chmod(tool.stat().st_mode | stat.S_IEXEC)
    monkeypatch.setenv("PATH", f"{tmp_path}{os.pathsep}{os.environ.get('PATH', '')}")
    uuid = "GPU-8a7f3c52-0000-4000-8000-000000000001"
    sampler = bench.ClockSampler(uuid, str(tmp_path / "clocks.csv"))
    t0 = time.time()
    sampler.wait_first(timeout=10.0)
    assert os.path.getsize(tmp_path / "clocks.csv") > 0 and time.time() - t0 < 10.0
    time.sleep(0.3)
    res = sampler.stop()
    assert res["samples"] >= 2
    assert res["sm_mhz"] == 2070.0 and res["sm_max_mhz"] == 2070.0
    assert res["reasons"] == ["sw_power_cap"] and res["power_w_max"] == 180.5
    # the GPU is named by its UUID: nvidia-smi's indices ignore CUDA_VISIBLE_DEVICES
    assert f"--id={uuid}" in open(argv_file).read().split()


def test_smi_gpu_id_prefers_the_uuid(monkeypatch):
    import types
    import torch
    import bench
    props = types.SimpleNamespace(uuid="8a7f3c52-0000-4000-8000-000000000001")
    monkeypatch.setattr(torch.cuda, "get_device_properties", lambda d: props)
    assert bench.smi_gpu_id(torch.device("cuda", 3)) == "GPU-8a7f3c52-0000-4000-8000-000000000001"
    props.uuid = "GPU-1234"
    assert bench.smi_gpu_id(torch.device("cuda", 0)) == "GPU-1234"


def test_clock_sampler_without_nvidia_smi(tmp_path, monkeypatch):
    import bench
    monkeypatch.setenv("PATH", str(tmp_path))  # no nvidia-smi here
    sampler = bench.ClockSampler(0, str(tmp_path / "clocks.csv"))
    sampler.wait_first(timeout=0.1)
    assert sampler.stop()["reasons"] == ["nvidia-smi unavailable"]
