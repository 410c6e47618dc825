"""bench.py's clock record, on CPU: samples are time-stamped, and the
summary keeps those taken inside the busy window (the timed steps and the
per-kernel pass), with the median SM clock and every throttle reason seen
there; with none inside it falls back to every sample and says so."""
import datetime

import bench


def _line(t, sm, power_cap, thermal="Not Active"):
    ts = t.strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    return f"{ts}, 0, {sm}, 2070, 910.5, 0x0000000000000004, Not Active, {thermal}, Not Active, {power_cap}"


def _sampler(lines, window):
    c = bench.ClockSampler(0)
    c.lines = lines
    c.mark(*window)

    class _Done:  # a finished nvidia-smi process
        def terminate(self):
            pass

        def wait(self, timeout=None):
            return 0

    class _Thread:
        def join(self, timeout=None):
            pass

    c.proc, c.t = _Done(), _Thread()
    return c


def test_summary_keeps_the_busy_window(monkeypatch):
    monkeypatch.setattr(bench.time, "sleep", lambda s: None)
    t0 = datetime.datetime(2026, 1, 2, 3, 4, 5)
    ms = lambda v: t0 + datetime.timedelta(milliseconds=v)
    lines = [_line(ms(0), 1100, "Not Active"),          # idle, before
             _line(ms(120), 2070, "Active"),
             _line(ms(220), 2055, "Active"),
             _line(ms(320), 2070, "Not Active"),
             _line(ms(900), 1200, "Not Active", thermal="Active")]   # after
    clk = _sampler(lines, (ms(100), ms(400))).stop()
    assert clk["samples"] == 3
    assert clk["sm_mhz"] == 2070.0 and clk["sm_max_mhz"] == 2070.0
    assert clk["reasons"] == ["sw_power_cap"]
    assert clk["window_ms"] == 300.0


def test_summary_falls_back_to_every_sample(monkeypatch):
    monkeypatch.setattr(bench.time, "sleep", lambda s: None)
    t0 = datetime.datetime(2026, 1, 2, 3, 4, 5)
    lines = [_line(t0, 2070, "Not Active"), _line(t0 + datetime.timedelta(seconds=1), 2060, "Active")]
    window = (t0 + datetime.timedelta(milliseconds=300), t0 + datetime.timedelta(milliseconds=400))
    clk = _sampler(lines, window).stop()
    assert clk["samples"] == 2 and "no sample fell inside" in clk["window"]
    assert clk["reasons"] == ["sw_power_cap"]
