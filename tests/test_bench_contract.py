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
