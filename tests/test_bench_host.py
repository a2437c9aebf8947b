"""Host logic of bench.py that needs no GPU: the clock record built from nvidia-smi lines
and the DRAM traffic read from a committed ncu summary only for the matching build."""
import os
import sys
import types

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench   # noqa: E402


def _sampler(lines, times):
    c = bench.ClockSampler(0, period_ms=50)
    c.proc = types.SimpleNamespace(stdout=iter(lines))
    clock = iter(times)
    real = bench.time.time
    bench.time.time = lambda: next(clock)
    try:
        c._read()
    finally:
        bench.time.time = real
    return c


def test_clock_record_inside_the_timed_region():
    lines = ["0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active\n",
             "0, 1980, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active\n",
             "0, 2070, 2070, 950.0, 0x0, Not Active, Not Active, Not Active, Not Active\n",
             "garbage line\n"]
    c = _sampler(lines, [10.00, 10.05, 10.50])
    c.t0, c.t1 = 9.99, 10.06
    r = c.summary()
    assert r["samples"] == 2 and r["window"] == "inside timed region"
    assert r["sm_mhz"] == (2070 + 1980) / 2 and r["sm_max_mhz"] == 2070
    assert r["reasons"] == ["sw_power_cap"]


def test_clock_record_falls_back_to_the_nearest_sample():
    lines = ["0, 2070, 2070, 900.1, 0x0, Active, Not Active, Not Active, Not Active\n",
             "0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active\n"]
    c = _sampler(lines, [5.0, 7.0])
    c.t0, c.t1 = 6.9, 6.91
    r = c.summary()
    assert r["samples"] == 1 and r["window"].startswith("nearest") and r["reasons"] == []


def test_traffic_needs_the_matching_build(tmp_path, monkeypatch):
    (tmp_path / "k.md").write_text("summary\n\ntraffic_bytes_per_launch: 123456 (build abcdef0123456789)\n")
    monkeypatch.setattr(bench, "PROFILES", str(tmp_path))
    assert bench.traffic_from_profile("k.md", "abcdef0123456789") == 123456.0
    assert bench.traffic_from_profile("k.md", "0000000000000000") is None
    assert bench.traffic_from_profile("missing.md", "abcdef0123456789") is None
