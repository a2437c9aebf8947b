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


class _FakeNvml:
    """Stands in for libnvidia-ml: a clock and a clock-event reason mask per call."""

    def __init__(self, clocks, reasons):
        self.clocks, self.reasons = iter(clocks), iter(reasons)

    def nvmlDeviceGetClockInfo(self, h, kind, out):
        out._obj.value = next(self.clocks)
        return 0

    def nvmlDeviceGetCurrentClocksEventReasons(self, h, out):
        out._obj.value = next(self.reasons)
        return 0


def test_nvml_clock_record_and_reasons():
    c = bench.NvmlClocks.__new__(bench.NvmlClocks)
    c.period, c.samples, c.max_mhz, c.h = 0.0005, [], 2070.0, None
    c.lib = _FakeNvml([2070, 1965, 2070, 2070], [0x0, 0x4, 0x8 | 0x40, 0x1])
    c._reasons_fn = c.lib.nvmlDeviceGetCurrentClocksEventReasons
    clock = iter([1.0, 2.0, 3.0, 4.0])
    real = bench.time.time
    bench.time.time = lambda: next(clock)
    try:
        for _ in range(4):
            c._sample()
    finally:
        bench.time.time = real
    c.t0, c.t1 = 1.5, 3.5
    r = c.summary()
    assert r["samples"] == 2 and r["sm_mhz_min"] == 1965 and r["sm_max_mhz"] == 2070
    assert r["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_power_cap"]
    c.t0, c.t1 = 10.0, 11.0
    assert c.summary()["samples"] == 0


def test_spread_of_timings():
    r = bench.spread([1.0, 2.0, 3.0, 4.0, 5.0])
    assert r["us_median"] == 3000.0 and r["us_mean"] == 3000.0
    assert r["us_p10"] == 1400.0 and r["us_p90"] == 4600.0
    assert bench.spread([0.5])["us_p90"] == 500.0


def test_e2e_plans_the_next_step_while_the_gpu_runs():
    """Pipelined e2e: each step launches its copies and kernel, plans the next step's
    table on the host, then waits for its own result; every step has its copies."""
    log = []
    result_ready = types.SimpleNamespace(synchronize=lambda: log.append("wait result"))
    stream = types.SimpleNamespace(synchronize=lambda: log.append("sync"),
                                   record_event=lambda ev=None: result_ready)
    job = {"e2e": (lambda: log.append("plan"), lambda: log.append("launch")),
           "e2e_bytes": lambda: (100, 50), "numerator": 1e9, "scale": 1e9, "unit": "GB/s"}
    r = bench.e2e_run(job, steps=1, warmup=1, stream=stream)
    n = r["steps"]
    piped = log[3:3 + 1 + 3 * n + 1]     # after the warm-up's plan, launch, sync
    # each step waits for its own read-back (an event behind it), not for the next
    # step's plan upload; the stream is drained once at the end
    assert piped[0] == "plan" and piped[1:-1] == ["launch", "plan", "wait result"] * n
    assert piped[-1] == "sync"
    assert log[3 + 1 + 3 * n + 1:] == ["plan", "launch", "sync"] * n
    assert r["h2d_bytes_per_step"] == 100 and r["d2h_bytes_per_step"] == 50


def test_cascade_split_evens_out_the_levels():
    """The prefix level's SM share grows with its FLOPs and shrinks as the suffix's bytes
    grow, and always leaves both levels at least 8 SMs."""
    a = bench.cascade_prefix_sms(152, 34.4e9, 578e6)
    assert 8 <= a <= 144
    assert bench.cascade_prefix_sms(152, 2 * 34.4e9, 578e6) > a
    assert bench.cascade_prefix_sms(152, 34.4e9, 2 * 578e6) < a
    assert bench.cascade_prefix_sms(152, 1e3, 1e12) == 8
    assert bench.cascade_prefix_sms(152, 1e15, 1e3) == 144
