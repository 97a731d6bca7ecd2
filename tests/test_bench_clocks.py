"""bench.py's clock record and the check that rejects it, on the CPU with a stand-in nvidia-smi on PATH.

The bench samples SM clocks and throttle reasons during the timed region. A record showing a
hardware or thermal slowdown, or SM clocks held well below their maximum with no reason given,
rejects the timed region (the bench measures it once more); a power cap is kept and noted.
"""

from __future__ import annotations

import os
import stat
import sys
import time

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def fake_smi(tmp_path, sm: int, top: int, reasons: tuple[str, str, str, str]):
    """A stand-in that prints a sample every 20 ms in the queried CSV form until it is stopped."""
    hw, hwt, swt, cap = reasons
    script = tmp_path / "nvidia-smi"
    script.write_text(
        "#!/bin/bash\n"
        "while true; do\n"
        f'  echo "$(date +"%Y/%m/%d %H:%M:%S.%3N"), 0, {sm}, {top}, 950.00, 0x0, {hw}, {hwt}, {swt}, {cap}"\n'
        "  sleep 0.02\n"
        "done\n")
    script.chmod(script.stat().st_mode | stat.S_IEXEC)
    return str(tmp_path)


def record(tmp_path, monkeypatch, sm, top, reasons):
    monkeypatch.setenv("PATH", fake_smi(tmp_path, sm, top, reasons) + os.pathsep + os.environ["PATH"])
    c = bench.ClockSampler(0)
    c.start()
    t0 = time.time()
    time.sleep(0.3)
    t1 = time.time()
    early = c.summary(t0, t1, c.peek())  # while it runs, as the bench's check reads it
    c.stop()
    return early, c.summary(t0, t1)


NA, A = "Not Active", "Active"


def test_power_capped_record_is_kept(tmp_path, monkeypatch):
    early, final = record(tmp_path, monkeypatch, 1980, 2070, (NA, NA, NA, A))
    for s in (early, final):
        assert s["sm_mhz"] == 1980 and s["sm_max_mhz"] == 2070 and s["reasons"] == ["sw_power_cap"]
        assert s["samples"] >= 3 and s["window"] == "timed"
        assert bench.clock_rejection(s) is None


def test_hardware_slowdown_rejects(tmp_path, monkeypatch):
    early, final = record(tmp_path, monkeypatch, 1400, 2070, (A, NA, NA, NA))
    assert bench.clock_rejection(early) == "hw_slowdown" == bench.clock_rejection(final)


def test_thermal_slowdowns_reject(tmp_path, monkeypatch):
    _, final = record(tmp_path, monkeypatch, 1500, 2070, (NA, A, A, A))
    assert bench.clock_rejection(final) == "hw_thermal_slowdown, sw_thermal_slowdown"


def test_clock_held_low_without_reason_rejects(tmp_path, monkeypatch):
    _, final = record(tmp_path, monkeypatch, 1200, 2070, (NA, NA, NA, NA))
    assert final["reasons"] == []
    assert bench.clock_rejection(final) == "SM clock 1200 of 2070 MHz with no reason given"


def test_full_clock_and_no_samples_keep_the_measurement():
    assert bench.clock_rejection({"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 5}) is None
    none = bench.ClockSampler.summary(bench.ClockSampler.__new__(bench.ClockSampler), 0.0, 1.0, [])
    assert none["samples"] == 0 and bench.clock_rejection(none) is None


def test_parse_skips_malformed_lines():
    rows = bench.ClockSampler.parse("garbage\n2026/12/03 10:00:00.250, 0, 1980, 2070, 900, 0x0, "
                                    "Not Active, Not Active, Not Active, Active\n1, 2, 3\n")
    assert len(rows) == 1 and rows[0][1:3] == (1980.0, 2070.0) and rows[0][3][3] == "Active"


@pytest.mark.parametrize("line", ["2026/12/03 10:00:00, 0, [N/A], 2070, 900, 0x0, a, b, c, d"])
def test_parse_skips_unreadable_clocks(line):
    assert bench.ClockSampler.parse(line) == []
