"""The bench's clock record: nvidia-smi samples (timestamped, every 50 ms)
kept only inside the timed window, with the throttle reasons seen there.
Runs on CPU with a recorded sample file in place of nvidia-smi."""
import datetime
import os
import sys
import tempfile

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


class _DoneProc:
    def poll(self):
        return 0

    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def _sampler(t_start, rows):
    """A ClockSampler whose nvidia-smi output is `rows` (seconds after t_start, MHz, power-cap active)."""
    fd, path = tempfile.mkstemp(suffix=".csv")
    with os.fdopen(fd, "w") as f:
        for dt, mhz, capped in rows:
            ts = datetime.datetime.fromtimestamp(t_start + dt).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
            cap = "Active" if capped else "Not Active"
            f.write("%s, 0, %d, 2070, 900.00, 0x0, Not Active, Not Active, Not Active, %s\n" % (ts, mhz, cap))
    c = bench.ClockSampler.__new__(bench.ClockSampler)
    c.proc, c.path, c.fh = _DoneProc(), path, open(os.devnull, "w")
    c.t0 = c.t1 = None
    return c


def test_only_samples_inside_the_window_count():
    t = 1.8e9
    rows = [(0.05 * i, 1500 if i < 4 else 2000 + i, i == 6) for i in range(12)]
    c = _sampler(t, rows)
    c.t0, c.t1 = t + 0.19, t + 0.41          # samples 4..8
    r = c.stop()
    assert r["samples"] == 5 and r["in_window"]
    assert r["sm_mhz"] == 2006 and r["sm_max_mhz"] == 2070
    assert r["reasons"] == ["sw_power_cap"]    # sample 6 only


def test_window_without_samples_takes_the_nearest():
    t = 1.8e9
    rows = [(0.0, 1900, False), (0.05, 1950, True), (0.10, 1990, False), (0.40, 2060, False)]
    c = _sampler(t, rows)
    c.t0, c.t1 = t + 0.06, t + 0.09           # between samples 1 and 2
    r = c.stop()
    assert not r["in_window"] and r["samples"] == 2
    assert r["sm_mhz"] == 1970 and r["reasons"] == ["sw_power_cap"]


def test_no_window_keeps_every_sample():
    t = 1.8e9
    c = _sampler(t, [(0.05 * i, 2000, False) for i in range(3)])
    r = c.stop()
    assert r["samples"] == 3 and r["reasons"] == []
