"""GPU parity of the fixed-threshold verify length and the threshold sweep
([DSpark notes] sec. 5.2, sec. 8.3 Fig. 5) against the oracle: every output
bit-exact (integer counts; the expected count is an exact integer sum of
survivals in units of 2^-48 on both sides)."""
from __future__ import annotations

import json
import os

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_markov_gb300 import binding as sdm

pytestmark = pytest.mark.gpu
DEV = "cuda"
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def host(t):
    return t.detach().cpu().numpy()


def confidences(R, g, seed):
    """Random confidences with the edge values: exact thresholds, 0, 1, NaN."""
    rng = np.random.default_rng(seed)
    c = rng.random((R, g)).astype(np.float32) ** 0.3          # mostly high, as confidence heads are
    flat = c.reshape(-1)
    k = min(flat.size, 64)
    pos = rng.choice(flat.size, size=k, replace=False)
    flat[pos] = np.resize(np.array([0.5, 0.25, 0.9, 1.0, 0.0, np.nan], np.float32), k)
    return c


TAUS = np.array([0.0, 0.1, 0.25, 0.5, 0.5000001, 0.75, 0.9, 0.99, 1.0, 1.5], np.float32)


@pytest.mark.parametrize("R,g,seed", [(1, 1, 0), (3, 4, 1), (64, 7, 2), (256, 16, 3), (2000, 8, 4), (4096, 8, 5)])
def test_schedule_threshold(R, g, seed):
    conf = confidences(R, g, seed)
    for tau in (0.0, 0.5, 0.9, 1.0, 2.0):
        ref = oracle.schedule_threshold(conf, tau)
        out = sdm.schedule_threshold(dev(conf), tau)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(host(out["budget"]), ref["budget"])
        assert int(host(out["total_tokens"])[0]) == ref["total_tokens"]


@pytest.mark.parametrize("R,g,seed", [(1, 1, 0), (3, 4, 1), (64, 7, 2), (256, 16, 3), (2048, 16, 4), (1, 64, 5)])
def test_threshold_sweep(R, g, seed):
    conf = confidences(R, g, seed)
    ceiling = np.random.default_rng(seed + 100).integers(0, g + 1, R).astype(np.int32)
    ref = oracle.threshold_sweep(conf, TAUS, ceiling)
    out = sdm.threshold_sweep(dev(conf), dev(TAUS), dev(ceiling))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host(out["drafts"]), ref["drafts"])
    np.testing.assert_array_equal(host(out["accepted"]), ref["accepted"])
    np.testing.assert_array_equal(host(out["expected"]).view(np.uint64), ref["expected"].view(np.uint64))
    none = sdm.threshold_sweep(dev(conf), dev(TAUS))
    torch.cuda.synchronize()
    assert np.all(host(none["accepted"]) == -1)
    np.testing.assert_array_equal(host(none["drafts"]), ref["drafts"])


def test_threshold_worked_example_on_the_gpu():
    with open(os.path.join(GOLDEN, "threshold_sweep_worked_example.json")) as f:
        g = json.load(f)
    conf = np.array(g["conf"], np.float32)
    out = sdm.threshold_sweep(dev(conf), dev(np.array(g["taus"], np.float32)),
                              dev(np.array(g["ceiling"], np.int32)))
    one = sdm.schedule_threshold(dev(conf), 0.5)
    torch.cuda.synchronize()
    e = g["expected"]
    np.testing.assert_array_equal(host(out["drafts"]), e["drafts"])
    np.testing.assert_array_equal(host(out["accepted"]), e["accepted"])
    np.testing.assert_allclose(host(out["expected"]), e["expected"], atol=1e-6)
    np.testing.assert_array_equal(host(one["budget"]), e["budget_at_0.5"])
    assert int(host(one["total_tokens"])[0]) == e["total_tokens_at_0.5"]
