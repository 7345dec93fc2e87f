"""The reference arm (the oracle on the host cores) under each option of the
bench: the production scheduler, the fixed-threshold rule, the RNN head and
the observability pass, on the tiny workload (CPU only)."""
from __future__ import annotations

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("extra,key,val", [
    (["--scheduler", "dynamic"], "scheduler", "dynamic"),
    (["--scheduler", "threshold", "--tau", "0.6"], "tau", 0.6),
    (["--head", "rnn"], "head", "rnn"),
    (["--observe"], "observe", True),
])
def test_reference_arm_option(extra, key, val):
    cmd = [sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny_chain", "--steps", "2",
           "--warmup", "3"] + extra
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    out = json.loads(lines[0])
    assert out["impl"] == "reference" and out["value"] > 0
    got = out["config"][key]
    assert (abs(got - val) < 1e-6) if isinstance(val, float) else got == val


def test_reference_arm_reports_all_cores_and_one():
    """The default reference arm spreads single-request oracle cycles over
    every host core it may use and reports the single-threaded rate beside
    it; the oracle's own arithmetic is the same in both."""
    cmd = [sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny_chain", "--steps", "2",
           "--warmup", "3", "--cpu-seconds", "1"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    out = json.loads([l for l in r.stdout.splitlines() if l.startswith("{")][0])
    cb = out["cpu_baseline"]
    assert cb["cores"] == len(os.sched_getaffinity(0)) and cb["value"] == out["value"]
    assert cb["single_thread"]["cores"] == 1 and cb["single_thread"]["value"] > 0
    assert out["e2e"]["h2d_bytes_per_step"] == 0


def test_threaded_oracle_sample_commits_what_the_serial_one_does():
    """The all-core oracle sample runs the same per-request cycles as the
    single-threaded one: over the same requests it commits the same tokens."""
    sys.path.insert(0, ROOT)
    import bench
    from speculative_decoding_markov_gb300 import synthetic
    from speculative_decoding_markov_gb300.workloads import WORKLOADS

    w = WORKLOADS["tiny_chain"]
    inp = synthetic.generate(w, seed=0, device="cpu")
    h = bench.host_inputs(inp)
    serial = sum(bench.oracle_back(w, _front(bench, w, h, i)) for i in range(w.R))
    mt = bench.oracle_sample_threads(w, inp, 0.0, threads=3)
    assert mt["cores"] == 3 and mt["value"] > 0
    assert f"{w.R} of {w.R} requests" in mt["sample"] or mt["sample"].startswith("3 of")
    assert serial >= w.R


def _front(bench, w, h, i):
    st = bench.oracle_front(w, h, [i])
    bench.oracle_target(w, st)
    return st
