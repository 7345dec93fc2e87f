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
