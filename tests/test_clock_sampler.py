"""bench.ClockSampler against a stand-in nvidia-smi on PATH (no GPU needed): it returns from
start() once the first sample is in, parses the samples and the throttle reasons, and does not
wait when the tool exits at once."""
import os
import stat
import time

import bench


def _fake_tool(tmp_path, body):
    d = tmp_path / "bin"
    d.mkdir()
    f = d / "nvidia-smi"
    f.write_text("#!/bin/sh\n" + body)
    f.chmod(f.stat().st_mode | stat.S_IEXEC)
    return str(d)


def test_sampler_parses_samples(tmp_path, monkeypatch):
    line = "2070, 2070, 950.5, 0x0, Not Active, Not Active, Not Active, Active"
    d = _fake_tool(tmp_path, f'while true; do echo "{line}"; sleep 0.05; done\n')
    monkeypatch.setenv("PATH", d + os.pathsep + os.environ["PATH"])
    s = bench.ClockSampler(0)
    t0 = time.perf_counter()
    s.start()
    assert time.perf_counter() - t0 < 5.0
    time.sleep(0.2)
    c = s.stop()
    assert c["sm_mhz"] == 2070.0 and c["sm_max_mhz"] == 2070.0 and c["samples"] >= 2
    assert c["reasons"] == ["sw_power_cap"]


def test_sampler_does_not_wait_for_a_tool_that_exits(tmp_path, monkeypatch):
    d = _fake_tool(tmp_path, "exit 9\n")
    monkeypatch.setenv("PATH", d + os.pathsep + os.environ["PATH"])
    s = bench.ClockSampler(0)
    t0 = time.perf_counter()
    s.start()
    assert time.perf_counter() - t0 < 5.0
    c = s.stop()
    assert c["sm_mhz"] is None and c["samples"] == 0
