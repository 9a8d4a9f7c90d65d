"""The benchmark's reference arm (the oracle on the host cores) prints the one
JSON line the harness reads, for a sampled workload (Markov and RNN heads) and
for the greedy one (CPU only)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("config,head,extra,async_cap",
                         [("c2", "markov", [], False), ("greedy", "markov", [], False),
                          ("c2", "rnn", [], False), ("c2", "markov", ["--async-cap"], True),
                          ("c5", "markov", [], True), ("c5", "markov", ["--static-cap"], False)])
def test_reference_arm_json_line(config, head, extra, async_cap):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--config", config, "--steps", "3", "--warmup", "1", "--head", head,
                          *extra],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["metric"] == "draft+verified positions/s"
    assert line["value"] > 0 and line["unit"] == "positions/s" and line["higher_is_better"]
    assert line["steps"] == 3 and line["warmup"] == 1 and line["config"]["workload"] == config
    assert ("async_cap" in line["config"]) == async_cap
    for key in ("K", "logits", "factors", "parallelism"):  # the same config keys as our arm
        assert key in line["config"]
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    assert line["config"].get("head", "markov") == head


def test_workload_options():
    """--head and --async-cap reach the workload and the reported config; the
    verify-only greedy workload refuses both (it has no draft or schedule)."""
    import argparse
    import sys as _sys
    _sys.path.insert(0, ROOT)
    import bench

    def args(**kw):
        base = dict(config="c5", sched_mode="workload", sched_threshold=0.3, head="markov",
                    async_cap=False, static_cap=False)
        base.update(kw)
        return argparse.Namespace(**base)

    wl = bench._workload(args(head="rnn", async_cap=True))
    assert wl.head == "rnn" and wl.async_cap and wl.name == "c5"
    cfg = bench._sched_config(wl)
    assert cfg["sched_mode"] == "early_stop" and "async_cap" in cfg
    # c5's own cap is the asynchronous one; --static-cap keeps K fixed
    assert bench._workload(args()).async_cap
    assert not bench._workload(args(static_cap=True)).async_cap
    assert not bench._workload(args(config="c3")).async_cap
    wl = bench._workload(args(sched_mode="threshold", sched_threshold=0.25, static_cap=True))
    assert bench._sched_config(wl) == {"sched_mode": "threshold", "sched_threshold": 0.25}
    for kw in (dict(head="rnn"), dict(async_cap=True)):
        with pytest.raises(SystemExit):
            bench._workload(args(config="greedy", **kw))
    with pytest.raises(SystemExit):
        bench._workload(args(async_cap=True, static_cap=True))


def test_clock_sampler_keeps_the_timed_window(monkeypatch):
    """The clock record holds only the samples stamped inside the timed
    region, and reports the throttle reasons seen there (a stand-in for
    nvidia-smi writes the CSV)."""
    import datetime
    sys.path.insert(0, ROOT)
    import bench

    t0 = datetime.datetime(2026, 1, 2, 3, 4, 5, 100000)
    t1 = t0 + datetime.timedelta(milliseconds=40)

    def row(dt, mhz, reason):
        stamp = dt.strftime("%Y/%m/%d %H:%M:%S.") + f"{dt.microsecond // 1000:03d}"
        return (f"{stamp}, 0, {mhz} MHz, 2070 MHz, 600.00 W, 0x0, Not Active, Not Active, Not Active, "
                f"{reason}\n")

    class FakeProc:
        def terminate(self):
            pass

        def wait(self, timeout=None):
            return 0

        def kill(self):
            pass

    def fake_popen(cmd, stdout=None, stderr=None):
        assert cmd[0] == "nvidia-smi" and "-lms" in cmd
        stdout.write("timestamp, index, clocks.current.sm [MHz], ...\n")
        stdout.write(row(t0 - datetime.timedelta(milliseconds=30), 900, "Not Active"))  # idle, before
        for i, mhz in enumerate((2070, 2055, 2040)):
            stdout.write(row(t0 + datetime.timedelta(milliseconds=5 + 10 * i), mhz,
                             "Active" if i == 1 else "Not Active"))
        stdout.write(row(t1 + datetime.timedelta(milliseconds=8), 1000, "Not Active"))  # after
        stdout.flush()
        return FakeProc()

    monkeypatch.setattr(bench.subprocess, "Popen", fake_popen)
    clk = bench.ClockSampler(0).stop(t0, t1)
    assert clk["samples"] == 3 and clk["sm_mhz"] == 2055.0 and clk["sm_max_mhz"] == 2070.0
    assert clk["reasons"] == ["sw_power_cap"] and clk["interval_ms"] == 10 and clk["window_ms"] == 40.0
    # a window shorter than the interval takes the first sample after its start
    clk = bench.ClockSampler(0).stop(t0, t0 + datetime.timedelta(milliseconds=1))
    assert clk["samples"] == 1 and clk["sm_mhz"] == 2070.0
