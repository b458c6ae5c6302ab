"""The bench's clock sampler on the CPU, against a stand-in `nvidia-smi` that prints one timestamped
row every 100 ms: the samples it keeps are those taken during the timed region, plus one on each
side when the region is shorter than three intervals, and throttle reasons are read per column."""
import os
import stat
import sys
import textwrap
import time

import bench

FAKE = textwrap.dedent("""\
    #!{python}
    import datetime, sys, time
    reason = {reason!r}
    while True:
        now = datetime.datetime.now().strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        cols = [reason == r and "Active" or "Not Active"
                for r in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")]
        print(", ".join([now, "0", "2070", "2070", "350.5", "0x0"] + cols), flush=True)
        time.sleep(0.1)
    """)


def _fake_smi(tmp_path, monkeypatch, reason=""):
    path = tmp_path / "nvidia-smi"
    path.write_text(FAKE.format(python=sys.executable, reason=reason))
    path.chmod(path.stat().st_mode | stat.S_IXUSR)
    monkeypatch.setenv("PATH", str(tmp_path) + os.pathsep + os.environ["PATH"])


def test_samples_inside_a_long_region(tmp_path, monkeypatch):
    _fake_smi(tmp_path, monkeypatch)
    clocks = bench.ClockSampler(0).start()
    try:
        time.sleep(0.4)
        t0 = time.time()
        time.sleep(0.8)
        t1 = time.time()
        got = clocks.summary(t0, t1)
    finally:
        clocks.stop()
    assert got["window"] == "inside the timed region"
    # one row per 100 ms: at least 5 in 0.8 s, and no more than the region (however long the
    # sleep overran) can hold
    assert 5 <= got["samples"] <= (t1 - t0) / 0.1 + 2
    assert got["sm_mhz"] == 2070.0 and got["sm_max_mhz"] == 2070.0 and got["reasons"] == []


def test_short_region_keeps_a_neighbour_on_each_side(tmp_path, monkeypatch):
    _fake_smi(tmp_path, monkeypatch)
    clocks = bench.ClockSampler(0).start()
    try:
        time.sleep(0.5)
        t0 = time.time()
        time.sleep(0.01)
        t1 = time.time()
        got = clocks.summary(t0, t1)
    finally:
        clocks.stop()
    assert got["window"].startswith("inside the timed region, plus")
    assert 2 <= got["samples"] <= 3


def test_reason_columns(tmp_path, monkeypatch):
    _fake_smi(tmp_path, monkeypatch, reason="sw_power_cap")
    with bench.ClockSampler(0) as clocks:
        time.sleep(0.3)
        t0 = time.time()
        time.sleep(0.4)
        got = clocks.summary(t0, time.time())
    assert got["reasons"] == ["sw_power_cap"]


def test_no_nvidia_smi(tmp_path, monkeypatch):
    monkeypatch.setenv("PATH", str(tmp_path))
    with bench.ClockSampler(0) as clocks:
        assert clocks.summary(time.time(), time.time()) is None
