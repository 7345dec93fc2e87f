"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: known-answer
vectors, the worked example of the DSpark notes' Figure 1, closed forms
(losslessness: speculative greedy decoding equals target-only greedy
decoding), brute force on tiny inputs, special cases that reduce to a library
routine, and chi-square tests of the samplers.
"""
from __future__ import annotations

import itertools
import json
import math
import os

import numpy as np
import pytest
import torch
from scipy import special, stats

import oracle
from speculative_decoding_markov_gb300 import synthetic
from speculative_decoding_markov_gb300.workloads import BF16, FP32
from tests.helpers import (absolute_inputs, cycle_inputs, np_of, oracle_greedy_decode, small,
                           target_only_greedy)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------
# Philox4x32-10 and the uniforms
# ---------------------------------------------------------------------------
def test_philox_known_answers():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")) if l.strip() and l[0] != "#"]
    assert len(rows) == 3
    for row in rows:
        vals = [int(x, 16) for x in row]
        out = oracle.philox(vals[0:4], vals[4:6])
        assert [int(x) for x in out] == vals[6:10]


def test_uniform_grid_and_moments():
    us = np.array([oracle.uniform(7, 3, oracle.STREAM_DRAFT, i, 2, v) for i in range(40) for v in range(100)])
    assert np.all(us > 0) and np.all(us < 1)
    k = us * 2 ** 24
    assert np.all(k == np.round(k)) and np.all(np.round(k) % 2 == 1)      # odd multiples of 2^-24
    assert abs(us.mean() - 0.5) < 0.02 and abs(us.var() - 1 / 12) < 0.01
    # the four words of one block serve v = 4c .. 4c+3; a new block for each field
    assert oracle.uniform(1, 0, 0, 0, 0, 0) != oracle.uniform(1, 0, 0, 0, 0, 1)
    assert oracle.uniform(1, 0, 0, 0, 0, 0) != oracle.uniform(1, 0, 1, 0, 0, 0)
    assert oracle.uniform(1, 0, 0, 0, 0, 0) != oracle.uniform(1, 1, 0, 0, 0, 0)
    assert oracle.uniform(1, 0, 0, 0, 0, 0) != oracle.uniform(2, 0, 0, 0, 0, 0)


def test_uniform_uses_block_words_as_documented():
    blk = oracle.philox([1, 5, (oracle.STREAM_RESID << 16) | 3, 9], [11, 0])
    for w in range(4):
        u = oracle.uniform(11, 9, oracle.STREAM_RESID, 5, 3, 4 + w)
        assert u == (2 * (int(blk[w]) >> 9) + 1) / 2 ** 24


# ---------------------------------------------------------------------------
# Markov head and chain drafting
# ---------------------------------------------------------------------------
def _inputs(w, seed=0):
    return synthetic.generate(w, seed=seed)


def test_markov_product_exact_on_grid_and_flagged_off_grid():
    w = small(R=2, B=3, V=40, r=64)
    inp = _inputs(w)
    res = oracle.draft_chain(np_of(inp["L"]), np_of(inp["U"]), np_of(inp["W"]), np_of(inp["anchor"]))
    assert res["flags"] & oracle.FLAG_INEXACT_MARKOV == 0
    # a planted off-grid table (full-precision bf16 normals) must be caught
    U = np_of(torch.randn(40, 64, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16))
    Wt = np_of(torch.randn(64, 40, generator=torch.Generator().manual_seed(2)).to(torch.bfloat16))
    res = oracle.draft_chain(np_of(inp["L"]), U, Wt, np_of(inp["anchor"]))
    assert res["flags"] & oracle.FLAG_INEXACT_MARKOV


def test_chain_with_zero_markov_is_independent_argmax():
    """W = 0 turns the semi-AR head into the parallel drafter: y_d = argmax L_d."""
    for ldt in (FP32, BF16):
        w = small(R=5, B=6, V=333, r=32, l_dtype=ldt)
        inp = _inputs(w, seed=3)
        Wz = np.zeros((32, 333), np.uint16)
        res = oracle.draft_chain(np_of(inp["L"]), np_of(inp["U"]), Wz, np_of(inp["anchor"]))
        ref = torch.argmax(inp["L"].float(), dim=-1).numpy()
        np.testing.assert_array_equal(res["tokens"], ref)


def test_chain_zero_noise_target_accepts_everything():
    """sigma = 0 makes the target equal the drafter's logits: a correct chain
    draft (right previous token, right W orientation, L added) is accepted in
    full by greedy verification against the independent target stand-in."""
    for ldt in (FP32, BF16):
        w = small(R=6, B=7, V=97 * 8, r=64, l_dtype=ldt, target_dtype=FP32, sigma=(0.0,), l_std=1.0)
        inp = _inputs(w, seed=5)
        dr = oracle.draft_chain(np_of(inp["L"]), np_of(inp["U"]), np_of(inp["W"]), np_of(inp["anchor"]))
        tgt = synthetic.chain_target(inp, torch.as_tensor(dr["tokens"]), FP32)
        t_argmax = torch.argmax(tgt, dim=-1).numpy()
        np.testing.assert_array_equal(t_argmax[:, :-1], dr["tokens"])
        cu = np.arange(w.R + 1, dtype=np.int32) * (w.B + 1)
        vr = oracle.verify(oracle.STATIC, oracle.GREEDY, np_of(tgt.reshape(-1, w.V)), cu, np_of(inp["anchor"]),
                           dr["tokens"])
        np.testing.assert_array_equal(vr["accept"], np.full(w.R, w.B))
        np.testing.assert_array_equal(vr["out_tok"][:, -1], t_argmax[:, -1])


def test_chain_markov_term_changes_the_draft():
    """With a strong Markov term the draft follows z = L + U[y_{d-1}] W; the
    target's argmax along that prefix (computed by the stand-in) agrees."""
    w = small(R=4, B=5, V=64, r=64, l_std=0.05, sigma=(0.0,))
    inp = _inputs(w, seed=9)
    dr = oracle.draft_chain(np_of(inp["L"]), np_of(inp["U"]), np_of(inp["W"]), np_of(inp["anchor"]))
    tgt = synthetic.chain_target(inp, torch.as_tensor(dr["tokens"]), FP32)
    np.testing.assert_array_equal(torch.argmax(tgt, -1).numpy()[:, :-1], dr["tokens"])
    # and it differs from the parallel drafter's choice somewhere
    assert (dr["tokens"] != torch.argmax(inp["L"].float(), -1).numpy()).any()


def test_argmax_ties_take_lowest_id():
    V, r = 16, 8
    L = np.zeros((1, 2, V), np.float32)
    L[0, 0, [3, 9, 12]] = 2.0
    L[0, 1, [0, 15]] = 1.0
    U = np.zeros((V, r), np.uint16)
    W = np.zeros((r, V), np.uint16)
    res = oracle.draft_chain(L, U, W, np.array([5], np.int32))
    assert res["tokens"].tolist() == [[3, 0]]
    assert res["margin"][0, 0] == 0.0


def test_chain_lse_and_logq_match_library_logsumexp():
    """With W = 0, z = L: lse must equal scipy's logsumexp of L/T and
    logq = L[y]/T - lse."""
    w = small(R=3, B=4, V=200, r=16)
    inp = _inputs(w, seed=2)
    L = np_of(inp["L"])
    Wz = np.zeros((16, 200), np.uint16)
    for T in (1.0, 0.7):
        res = oracle.draft_chain(L, np_of(inp["U"]), Wz, np_of(inp["anchor"]), decode=oracle.SAMPLE,
                                 temperature=T, seed=4)
        ref = special.logsumexp(L.astype(np.float64) / T, axis=-1)
        np.testing.assert_allclose(res["lse"], ref, rtol=1e-13)
        y = res["tokens"]
        ly = np.take_along_axis(L.astype(np.float64), y[..., None], -1)[..., 0] / T
        np.testing.assert_allclose(res["logq"], ly - ref, rtol=1e-12, atol=1e-13)


def test_sampler_is_inverse_cdf_of_its_uniform():
    """Each sampled draft token is the inverse CDF of softmax(z/T) in
    vocabulary order at the one uniform of (stream 0, request, row d):
    numpy's searchsorted over the cumulative probabilities gives the same id,
    and the reported margin is the distance of u to the nearer bound."""
    V, R, B, T = 50, 40, 3, 0.7
    rng = np.random.default_rng(11)
    L = rng.normal(0, 1.5, (R, B, V)).astype(np.float32)
    U = np.zeros((V, 4), np.uint16)
    W = np.zeros((4, V), np.uint16)
    anchor = np.zeros(R, np.int32)
    res = oracle.draft_chain(L, U, W, anchor, decode=oracle.SAMPLE, temperature=T, seed=5, cycle=3)
    for i in range(R):
        for d in range(B):
            p = special.softmax(L[i, d].astype(np.float64) / T)
            c = np.cumsum(p)
            u = oracle.uniform(5, 3, oracle.STREAM_DRAFT, i, d + 1, 0)   # rows count drafts from 1
            y = int(np.searchsorted(c, u, side="right"))
            assert res["tokens"][i, d] == y
            lo = c[y - 1] if y else 0.0
            np.testing.assert_allclose(res["margin"][i, d], min(u - lo, c[y] - u), rtol=1e-9, atol=1e-14)


def test_sampler_follows_softmax():
    """The inverse-CDF sampler draws y ~ softmax(z/T): chi-square over many
    independent requests (distinct counters) that share one logit row."""
    V, n, T = 8, 1 << 15, 0.8
    rng = np.random.default_rng(0)
    row = rng.normal(0, 1.0, V).astype(np.float32)
    L = np.broadcast_to(row, (n, 1, V)).copy()
    U = np.zeros((V, 4), np.uint16)
    W = np.zeros((4, V), np.uint16)
    anchor = np.zeros(n, np.int32)
    res = oracle.draft_chain(L, U, W, anchor, decode=oracle.SAMPLE, temperature=T, seed=123)
    counts = np.bincount(res["tokens"][:, 0], minlength=V)
    p = special.softmax(row.astype(np.float64) / T)
    _, pval = stats.chisquare(counts, p * n)
    assert pval > 1e-4


# ---------------------------------------------------------------------------
# scheduler
# ---------------------------------------------------------------------------
def test_scheduler_fig1_budget():
    g = json.load(open(os.path.join(GOLDEN, "fig1_walkthrough.json")))
    conf = np.array([g["confidences"]], np.float32)
    cost = g["cost_a"] + g["cost_b"] * np.arange(1 * (len(g["confidences"]) + 1) + 1, dtype=np.float64)
    sc = oracle.schedule_budget(conf, cost)
    assert sc["budget"].tolist() == [g["expected_budget"]]
    # survival is the running product
    np.testing.assert_array_equal(sc["survival"][0], np.cumprod(conf[0], dtype=np.float32))


def _objective(S, n, cost):
    E = S.shape[0] + sum(float(S[i, :n[i]].astype(np.float64).sum()) for i in range(S.shape[0]))
    N = S.shape[0] + int(sum(n))
    return E / cost[N]


@pytest.mark.parametrize("seed", range(12))
def test_scheduler_matches_brute_force(seed):
    """Greedy over ranked survivals is the exact optimum of E/cost over every
    allocation (n_1..n_R) in [0, gamma]^R (notes sec. 5.2)."""
    rng = np.random.default_rng(seed)
    R = int(rng.integers(1, 5))
    g = int(rng.integers(1, 5))
    conf = rng.uniform(0.05, 1.0, (R, g)).astype(np.float32)
    a, b = float(rng.uniform(0.5, 3.0)), float(rng.uniform(0.01, 0.6))
    cost = a + b * np.arange(R * (g + 1) + 1, dtype=np.float64)
    sc = oracle.schedule_budget(conf, cost)
    S = np.cumprod(conf, axis=1, dtype=np.float32)
    best = max(_objective(S, n, cost) for n in itertools.product(range(g + 1), repeat=R))
    got = _objective(S, sc["budget"], cost)
    assert got == pytest.approx(best, rel=1e-15, abs=0)
    assert sc["total_tokens"] == R + int(sc["budget"].sum())
    assert sc["expected"] == R + sum(float(S[i, :sc["budget"][i]].astype(np.float64).sum()) for i in range(R))


def test_scheduler_prefix_closed_and_unimodal():
    rng = np.random.default_rng(7)
    R, g = 64, 8
    conf = rng.uniform(0.2, 1.0, (R, g)).astype(np.float32)
    cost = 2.0 + 0.004 * np.arange(R * (g + 1) + 1)
    sc = oracle.schedule_budget(conf, cost)
    S = np.cumprod(conf, axis=1, dtype=np.float32)
    # prefix-closed: every selected position k has all k' < k selected, and
    # every selected survival is >= every unselected one
    sel = np.array([[k < sc["budget"][i] for k in range(g)] for i in range(R)])
    assert S[sel].min() >= S[~sel].max()
    # f(m) over the ranked list rises then falls: early stop == global argmax
    order = sorted(((float(S[i, k]), i, k) for i in range(R) for k in range(g)), key=lambda t: (-t[0], t[1], t[2]))
    f = [(R + sum(o[0] for o in order[:m])) / cost[R + m] for m in range(len(order) + 1)]
    m_star = int(np.argmax(f))
    assert sc["m_star"] == m_star
    assert all(f[m] <= f[m + 1] for m in range(m_star)) and all(f[m] >= f[m + 1] for m in range(m_star, len(f) - 1))


# ---------------------------------------------------------------------------
# production scheduler (stale capacity, global search, current ranking)
# ---------------------------------------------------------------------------
def _cost_from(table, R, g):
    cost = np.zeros(R * (g + 1) + 1, np.float64)
    for n, c in table.items():
        cost[int(n)] = c
    cost[:R] = cost[R]
    return cost


def test_dynamic_scheduler_cliff_fixture():
    """The hand-worked example: the stepped table makes f fall after the
    first token, the early-stopping scheduler verifies nothing, the global
    search over the stale survivals finds K = 4, and the current ranking
    spends it on request 1."""
    g = json.load(open(os.path.join(GOLDEN, "sps_cliff_dynamic_scheduler.json")))
    R, gam = g["R"], g["gamma"]
    cost = _cost_from(g["cost_by_tokens"], R, gam)
    stale = np.array(g["conf_stale"], np.float32)
    now = np.array(g["conf_now"], np.float32)
    sd = oracle.schedule_dynamic(now, stale, cost)
    assert sd["capacity"] == g["expected_capacity"]
    assert sd["budget"].tolist() == g["expected_budget"]
    assert sd["total_tokens"] == g["expected_total_tokens"]
    assert abs(sd["expected"] - g["expected_E"]) < 1e-6
    assert oracle.schedule_budget(stale, cost)["m_star"] == g["expected_capacity_with_early_stop"]


@pytest.mark.parametrize("seed", range(6))
def test_dynamic_scheduler_equals_greedy_on_additive_tables(seed):
    """With current == stale confidences and an additive table (f rises then
    falls), the global search and the early-stopping greedy agree."""
    rng = np.random.default_rng(100 + seed)
    R, g = int(rng.integers(1, 40)), int(rng.integers(1, 9))
    conf = rng.uniform(0.1, 1.0, (R, g)).astype(np.float32)
    cost = float(rng.uniform(0.5, 3.0)) + float(rng.uniform(0.001, 0.5)) * np.arange(R * (g + 1) + 1)
    sd = oracle.schedule_dynamic(conf, conf, cost)
    sb = oracle.schedule_budget(conf, cost)
    np.testing.assert_array_equal(sd["budget"], sb["budget"])
    assert sd["capacity"] == sb["m_star"] and sd["expected"] == sb["expected"]
    np.testing.assert_array_equal(sd["survival"], sb["survival"])


def _allocations(R, g):
    return itertools.product(range(g + 1), repeat=R)


@pytest.mark.parametrize("seed", range(10))
def test_dynamic_scheduler_matches_brute_force(seed):
    """Over every allocation (n_1..n_R) in [0, gamma]^R: the capacity's value
    E'(K)/cost[R + K] on the stale survivals is the best any allocation
    reaches (stepped table), and among the allocations of the verified size
    none carries more current survival than the selection."""
    rng = np.random.default_rng(seed)
    R, g = int(rng.integers(1, 5)), int(rng.integers(1, 5))
    stale = rng.uniform(0.05, 1.0, (R, g)).astype(np.float32)
    now = rng.uniform(0.05, 1.0, (R, g)).astype(np.float32)
    tiers = np.sort(rng.choice(np.arange(R, R * (g + 1) + 1), size=min(3, R * g + 1), replace=False))
    N = np.arange(R * (g + 1) + 1)
    tier_of = np.array([tiers[np.searchsorted(tiers, n)] if n <= tiers[-1] else n for n in N])
    cost = float(rng.uniform(0.5, 2.0)) + float(rng.uniform(0.05, 0.6)) * tier_of.astype(np.float64)
    sd = oracle.schedule_dynamic(now, stale, cost)
    Ss = np.cumprod(stale, axis=1, dtype=np.float32).astype(np.float64)
    Sn = np.cumprod(now, axis=1, dtype=np.float32).astype(np.float64)

    def value(S, n):
        return R + sum(S[i, :n[i]].sum() for i in range(R))

    best = max(value(Ss, n) / cost[R + sum(n)] for n in _allocations(R, g))
    K = sd["capacity"]
    top_stale = sorted(Ss.reshape(-1), reverse=True)[:K]
    assert abs((R + sum(top_stale)) / cost[R + K] - best) <= 1e-12 * best
    size = sd["total_tokens"] - R
    assert size == min(K, R * g)
    best_now = max(value(Sn, n) for n in _allocations(R, g) if sum(n) == size)
    assert abs(sd["expected"] - best_now) <= 1e-12 * best_now
    assert int(sd["budget"].sum()) == size


# ---------------------------------------------------------------------------
# ragged pack
# ---------------------------------------------------------------------------
def test_pack_round_trip_and_tier():
    rng = np.random.default_rng(1)
    R, g = 37, 8
    anchor = rng.integers(0, 1000, R).astype(np.int32)
    draft = rng.integers(0, 1000, (R, g)).astype(np.int32)
    budget = rng.integers(0, g + 1, R).astype(np.int32)
    tiers = np.array([64, 128, 256, 512], np.int32)
    pk = oracle.pack_ragged(anchor, draft, budget, tiers)
    cu = pk["cu_seqlens"]
    np.testing.assert_array_equal(np.diff(cu), budget + 1)
    T = int(cu[-1])
    assert pk["tier"] == min(t for t in tiers if t >= T) and pk["flags"] == 0
    for row in range(T):
        i, p = pk["packed_req"][row], pk["packed_pos"][row]
        assert cu[i] + p == row
        assert pk["packed_tok"][row] == (anchor[i] if p == 0 else draft[i, p - 1])
    assert np.all(pk["packed_tok"][T:] == -1) and np.all(pk["packed_req"][T:] == -1)
    # static (budget = None) above every tier: uncaptured, tier = total
    pk = oracle.pack_ragged(anchor, draft, None, tiers[:3])
    assert pk["tier"] == R * (g + 1) and pk["flags"] == oracle.FLAG_TIER_UNCAPTURED
    # strict mode ([SGLang] ragged verify: only captured tiers run): the same
    # rows, reported as an overflow instead; a total inside a tier is no error
    st = oracle.pack_ragged(anchor, draft, None, tiers[:3], strict=True)
    assert st["flags"] == oracle.FLAG_TIER_OVERFLOW and st["tier"] == pk["tier"]
    for k in ("cu_seqlens", "packed_tok", "packed_req", "packed_pos"):
        np.testing.assert_array_equal(st[k], pk[k])
    assert oracle.pack_ragged(anchor, draft, budget, tiers, strict=True)["flags"] == 0


def test_pack_empty_windows():
    anchor = np.array([3, 4], np.int32)
    draft = np.array([[1, 2], [5, 6]], np.int32)
    pk = oracle.pack_ragged(anchor, draft, np.array([0, 0], np.int32), np.array([2, 4], np.int32))
    assert pk["cu_seqlens"].tolist() == [0, 1, 2] and pk["tier"] == 2
    assert pk["packed_tok"].tolist() == [3, 4]


# ---------------------------------------------------------------------------
# greedy verification
# ---------------------------------------------------------------------------
def _onehot_rows(ids, V, hi=5.0):
    t = np.zeros((len(ids), V), np.float32)
    for j, v in enumerate(ids):
        t[j, v] = hi
    return t


def test_verify_fig1_walkthrough():
    g = json.load(open(os.path.join(GOLDEN, "fig1_walkthrough.json")))
    V = len(g["vocab"])
    anchor = np.array([g["vocab"].index(g["anchor"])], np.int32)
    draft = np.array([g["draft_ids"]], np.int32)
    conf = np.array([g["confidences"]], np.float32)
    cost = g["cost_a"] + g["cost_b"] * np.arange(len(g["confidences"]) + 2, dtype=np.float64)
    sc = oracle.schedule_budget(conf, cost)
    pk = oracle.pack_ragged(anchor, draft, sc["budget"], np.array([8], np.int32))
    assert pk["packed_tok"][: pk["cu_seqlens"][-1]].tolist() == [3, 4, 5, 6]      # D E F G
    target = _onehot_rows(g["target_argmax_ids"][: pk["cu_seqlens"][-1]], V)
    target = np.concatenate([target, np.zeros((pk["tier"] - target.shape[0], V), np.float32)])
    vr = oracle.verify(oracle.COMPACT, oracle.GREEDY, target, pk["cu_seqlens"], anchor, draft)
    assert vr["accept"].tolist() == [g["expected_accept"]]
    assert vr["out_tok"][0, : vr["n_out"][0]].tolist() == g["expected_commit_ids"]
    assert vr["n_out"][0] == vr["accept"][0] + 1            # the bonus counts


def test_verify_accept_is_first_mismatch_and_bonus_is_target_token():
    rng = np.random.default_rng(3)
    R, g, V = 50, 6, 12
    anchor = rng.integers(0, V, R).astype(np.int32)
    draft = rng.integers(0, V, (R, g)).astype(np.int32)
    t_ids = draft.copy()
    flip = rng.random((R, g)) < 0.3
    t_ids[flip] = (t_ids[flip] + 1 + rng.integers(0, V - 1, flip.sum())) % V
    bonus = rng.integers(0, V, R)
    rows = np.concatenate([t_ids, bonus[:, None]], axis=1)
    target = _onehot_rows(rows.reshape(-1), V)
    cu = np.arange(R + 1, dtype=np.int32) * (g + 1)
    vr = oracle.verify(oracle.STATIC, oracle.GREEDY, target, cu, anchor, draft)
    for i in range(R):
        mism = np.nonzero(draft[i] != rows[i, :g])[0]
        a = int(mism[0]) if mism.size else g
        assert vr["accept"][i] == a
        assert vr["out_tok"][i, :a].tolist() == draft[i, :a].tolist()
        assert vr["out_tok"][i, a] == rows[i, a]


def test_greedy_speculative_decoding_equals_target_only_decoding():
    """Lossless: the committed stream of speculative greedy decoding is the
    target model's own greedy decode (PCTree article; notes sec. 1)."""
    for ldt, tdt in ((FP32, FP32), (BF16, BF16)):
        w = small(R=4, B=5, V=64, r=16, l_dtype=ldt, target_dtype=tdt, sigma=(0.3, 0.8), l_std=1.0)
        cycles = 6
        ab = absolute_inputs(w, positions=cycles * (w.B + 1) + w.B + 1, seed=11)
        seqs, recs = oracle_greedy_decode(w, ab, cycles)
        n = min(len(s) for s in seqs) - 1
        ref = target_only_greedy(ab, n, tdt)
        for i in range(w.R):
            assert seqs[i][: n + 1] == ref[i].tolist()
        acc = np.concatenate([r["verify"]["accept"] for r in recs])
        assert acc.min() == 0 and acc.max() >= 2        # a mix of accepts and rejections


def test_verify_modes_invariants():
    """cap-accept commits exactly what compact commits and reports a ceiling
    >= its accept; compact accept = min(static accept, n_i); static is compact
    with n_i = gamma (DSpark in SGLang, three verify modes)."""
    w = small(R=16, B=6, V=64, r=16, sigma=(0.2, 0.6, 1.2), target_dtype=BF16, l_dtype=BF16)
    inp = _inputs(w, seed=21)
    an = np_of(inp["anchor"])
    dr = oracle.draft_chain(np_of(inp["L"]), np_of(inp["U"]), np_of(inp["W"]), an)
    sc = oracle.schedule_budget(np_of(inp["conf"]), synthetic.cost_table(w).numpy())
    tgt = synthetic.chain_target(inp, torch.as_tensor(dr["tokens"]), w.target_dtype)
    res = {}
    for mode, budget in (("static", None), ("compact", sc["budget"]), ("cap", None)):
        pk = oracle.pack_ragged(an, dr["tokens"], budget, np.array(w.tiers, np.int32))
        packed = synthetic.gather_packed(tgt, torch.as_tensor(pk["packed_req"]), torch.as_tensor(pk["packed_pos"]))
        om = {"static": oracle.STATIC, "compact": oracle.COMPACT, "cap": oracle.CAP_ACCEPT}[mode]
        res[mode] = oracle.verify(om, oracle.GREEDY, np_of(packed), pk["cu_seqlens"], an, dr["tokens"],
                                  budget=sc["budget"])
    np.testing.assert_array_equal(res["cap"]["out_tok"], res["compact"]["out_tok"])
    np.testing.assert_array_equal(res["cap"]["n_out"], res["compact"]["n_out"])
    assert np.all(res["cap"]["ceiling"] >= res["cap"]["accept"])
    np.testing.assert_array_equal(res["cap"]["ceiling"], res["static"]["accept"])
    np.testing.assert_array_equal(res["compact"]["accept"], np.minimum(res["static"]["accept"], sc["budget"]))


# ---------------------------------------------------------------------------
# rejection sampling
# ---------------------------------------------------------------------------
def _sample_cycle(w, inp, anchor, seed, cycle, mode=oracle.STATIC, budget=None):
    U, W = np_of(inp["U"]), np_of(inp["W"])
    dr = oracle.draft_chain(np_of(inp["L"]), U, W, anchor, decode=oracle.SAMPLE, temperature=w.temperature,
                            seed=seed, cycle=cycle)
    tgt = synthetic.chain_target(inp | {"anchor": torch.as_tensor(anchor)}, torch.as_tensor(dr["tokens"]),
                                 w.target_dtype)
    R = anchor.shape[0]
    cu = np.arange(R + 1, dtype=np.int32) * (w.B + 1)
    vr = oracle.verify(mode, oracle.SAMPLE, np_of(tgt.reshape(R * (w.B + 1), -1)), cu, anchor, dr["tokens"],
                       budget=budget, logq=dr["logq"], lse_q=dr["lse"], L=np_of(inp["L"]), U=U, W=W,
                       temperature=w.temperature, seed=seed, cycle=cycle)
    return dr, tgt, vr


@pytest.mark.parametrize("sigma", [0.3, 2.0])
def test_rejection_sampling_first_token_follows_target(sigma):
    """u < min(1, p/q) with residual resampling keeps the target distribution:
    the first committed token ~ p_1(. | anchor) (chi-square, df = V-1)."""
    n, V = 1 << 16, 8
    w = small(R=n, B=3, V=V, r=4, sigma=(sigma,), l_std=1.0)
    base = _inputs(small(R=1, B=3, V=V, r=4, sigma=(sigma,), l_std=1.0), seed=2)
    inp = {k: (v.expand(n, *v.shape[1:]).contiguous() if k in ("L", "L_bonus", "eta", "anchor") else v)
           for k, v in base.items()}
    anchor = np.full(n, int(base["anchor"][0]), np.int32)
    dr, tgt, vr = _sample_cycle(w, inp, anchor, seed=77, cycle=1)
    p1 = torch.softmax(tgt[0, 0].double(), -1).numpy()
    counts = np.bincount(vr["out_tok"][:, 0], minlength=V)
    _, pval = stats.chisquare(counts, p1 * n)
    assert pval > 1e-4
    assert vr["accept"].min() == 0 and vr["accept"].max() == 3


def test_rejection_sampling_pairs_follow_target():
    """First two committed tokens ~ p_1(t1) p_2(t2 | t1) (df = V^2 - 1); a
    second cycle from the committed anchor supplies t2 when the first cycle
    commits one token only."""
    n, V, B = 1 << 16, 8, 3
    w = small(R=n, B=B, V=V, r=4, sigma=(0.8,), l_std=1.0)
    ab1 = absolute_inputs(small(R=1, B=B, V=V, r=4, sigma=(0.8,), l_std=1.0), positions=2 * B + 2, seed=5)
    ab = {k: (v.expand(n, *v.shape[1:]).contiguous() if k in ("L_abs", "eta_abs", "anchor", "conf_abs") else v)
          for k, v in ab1.items()}
    anchor = np.full(n, int(ab1["anchor"][0]), np.int32)
    ci = cycle_inputs(ab, np.zeros(n, np.int64), B)
    _, _, v1 = _sample_cycle(w, ci, anchor, seed=3, cycle=0)
    t1 = v1["out_tok"][:, 0]
    t2 = v1["out_tok"][:, 1].copy()
    need = v1["n_out"] == 1
    idx = np.nonzero(need)[0]
    ci2 = cycle_inputs({k: (v[idx] if k in ("L_abs", "eta_abs", "conf_abs") else v) for k, v in ab.items()},
                       np.ones(idx.size, np.int64), B)
    _, _, v2 = _sample_cycle(w, ci2, t1[idx].astype(np.int32), seed=3, cycle=1)
    t2[idx] = v2["out_tok"][:, 0]
    # reference joint distribution from the stand-in target
    one = {"L": ab1["L_abs"], "L_bonus": ab1["L_abs"][:, -1], "U": ab1["U"], "W": ab1["W"], "eta": ab1["eta_abs"]}
    r1 = synthetic.target_rows(one, torch.tensor([0]), torch.tensor([0]), ab1["anchor"][:1], w.target_dtype)
    p1 = torch.softmax(r1[0].double(), -1)
    r2 = synthetic.target_rows(one, torch.zeros(V, dtype=torch.long), torch.ones(V, dtype=torch.long),
                               torch.arange(V), w.target_dtype)
    p2 = torch.softmax(r2.double(), -1)
    joint = (p1.view(V, 1) * p2).numpy().reshape(-1)
    counts = np.bincount(t1 * V + t2, minlength=V * V)
    keep = joint * n >= 5
    obs = np.append(counts[keep], counts[~keep].sum())
    exp = np.append(joint[keep] * n, joint[~keep].sum() * n)
    _, pval = stats.chisquare(obs, exp)
    assert pval > 1e-4


def test_rejection_sampling_equal_distributions_accept_everything():
    w = small(R=40, B=5, V=64, r=16, sigma=(0.0,), l_std=1.5)
    inp = _inputs(w, seed=8)
    _, tgt, vr = _sample_cycle(w, inp, np_of(inp["anchor"]), seed=1, cycle=0)
    np.testing.assert_array_equal(vr["accept"], np.full(w.R, w.B))
    # the bonus token is the inverse CDF of p at row B, one uniform of stream 3
    for i in range(w.R):
        c = np.cumsum(special.softmax(tgt[i, w.B].double().numpy() / w.temperature))
        u = oracle.uniform(1, 0, oracle.STREAM_BONUS, i, w.B, 0)
        assert vr["out_tok"][i, w.B] == int(np.searchsorted(c, u, side="right"))


def test_residual_and_bonus_are_inverse_cdf_draws():
    """With the Markov term zero, q_d = softmax(L_d/T).  Where request i stops
    at row a < B the committed token is the inverse CDF of max(0, p_a - q_a)
    (normalised) at the uniform of (stream 2, i, a); where every draft is
    accepted it is the inverse CDF of p_B at (stream 3, i, B)."""
    R, B, V, T = 300, 3, 12, 0.9
    rng = np.random.default_rng(21)
    L = rng.normal(0, 1.0, (R, B, V)).astype(np.float32)
    U = np.zeros((V, 4), np.uint16)
    W = np.zeros((4, V), np.uint16)
    anchor = rng.integers(0, V, R).astype(np.int32)
    dr = oracle.draft_chain(L, U, W, anchor, decode=oracle.SAMPLE, temperature=T, seed=6, cycle=1)
    tgt = (L[:, np.r_[0:B, B - 1]] + rng.normal(0, 0.7, (R, B + 1, V))).astype(np.float32)
    cu = np.arange(R + 1, dtype=np.int32) * (B + 1)
    vr = oracle.verify(oracle.STATIC, oracle.SAMPLE, tgt.reshape(-1, V), cu, anchor, dr["tokens"],
                       logq=dr["logq"], lse_q=dr["lse"], L=L, U=U, W=W, temperature=T, seed=6, cycle=1)
    seen = set()
    for i in range(R):
        a = int(vr["accept"][i])
        p = special.softmax(tgt[i, a].astype(np.float64) / T)
        if a < B:
            w_ = np.maximum(p - special.softmax(L[i, a].astype(np.float64) / T), 0.0)
            u = oracle.uniform(6, 1, oracle.STREAM_RESID, i, a, 0)
        else:
            w_ = p
            u = oracle.uniform(6, 1, oracle.STREAM_BONUS, i, a, 0)
        c = np.cumsum(w_)
        assert vr["out_tok"][i, a] == int(np.searchsorted(c, u * c[-1], side="right"))
        seen.add(a)
    assert seen == set(range(B + 1))


def test_rejection_sampling_cap_accept_equals_compact():
    w = small(R=64, B=6, V=32, r=16, sigma=(1.0,), l_std=1.0)
    inp = _inputs(w, seed=4)
    an = np_of(inp["anchor"])
    budget = np.random.default_rng(0).integers(0, w.B + 1, w.R).astype(np.int32)
    U, W = np_of(inp["U"]), np_of(inp["W"])
    dr = oracle.draft_chain(np_of(inp["L"]), U, W, an, decode=oracle.SAMPLE, seed=9, cycle=2)
    tgt = synthetic.chain_target(inp, torch.as_tensor(dr["tokens"]), w.target_dtype)
    outs = {}
    for mode, bud in (("compact", budget), ("cap", None)):
        pk = oracle.pack_ragged(an, dr["tokens"], bud, np.array(w.tiers, np.int32))
        packed = synthetic.gather_packed(tgt, torch.as_tensor(pk["packed_req"]), torch.as_tensor(pk["packed_pos"]))
        om = oracle.COMPACT if mode == "compact" else oracle.CAP_ACCEPT
        outs[mode] = oracle.verify(om, oracle.SAMPLE, np_of(packed), pk["cu_seqlens"], an, dr["tokens"],
                                   budget=budget, logq=dr["logq"], lse_q=dr["lse"], L=np_of(inp["L"]), U=U, W=W,
                                   seed=9, cycle=2)
    np.testing.assert_array_equal(outs["cap"]["out_tok"], outs["compact"]["out_tok"])
    assert np.all(outs["cap"]["ceiling"] >= outs["cap"]["accept"])
    assert (outs["cap"]["ceiling"] > outs["cap"]["accept"]).any()


# ---------------------------------------------------------------------------
# PCTree
# ---------------------------------------------------------------------------
def test_tree_with_k1_is_the_chain():
    """k = 1, N = B: every level keeps one child, the tree is the greedy chain."""
    w = small(R=5, B=6, V=300, r=32, l_dtype=BF16)
    inp = _inputs(w, seed=13)
    args = (np_of(inp["L"]), np_of(inp["U"]), np_of(inp["W"]), np_of(inp["anchor"]))
    ch = oracle.draft_chain(*args)
    tr = oracle.draft_tree(*args, k=1, P=4, N=w.B)
    np.testing.assert_array_equal(tr["tok"][:, 1:], ch["tokens"])
    np.testing.assert_array_equal(tr["parent"][:, 1:], np.tile(np.arange(w.B), (w.R, 1)))
    np.testing.assert_array_equal(tr["depth"][:, 1:], np.tile(np.arange(1, w.B + 1), (w.R, 1)))
    assert np.all(tr["n_nodes"] == w.B + 1)


def _all_paths(L, U, W, anchor, B):
    """Brute force: every token path of length <= B with its score
    sum log pi(v | parent) (dict path -> score)."""
    V = L.shape[-1]
    Lf = L.astype(np.float32) if L.dtype != np.uint16 else (L.astype(np.uint32) << 16).view(np.float32)
    Uf = (U.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    Wf = (W.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    out = {}

    def rec(path, prev, s):
        d = len(path) + 1
        if d > B:
            return
        z = (Lf[d - 1] + (Uf[prev] @ Wf).astype(np.float32)).astype(np.float32)
        lse = special.logsumexp(z.astype(np.float64))
        for v in range(V):
            p2 = path + (v,)
            sc = s + (float(z[v]) - lse)
            out[p2] = (sc, float(z[v]))
            rec(p2, v, sc)

    rec((), int(anchor), 0.0)
    return out


def _beam_reference(paths, V, B, k, P, N):
    """Independent replay of PCTree's rules over the enumerated paths."""
    frontier = [()]
    pool = []
    for d in range(1, B + 1):
        cands = []
        for slot, par in enumerate(frontier):
            kids = sorted(range(V), key=lambda v: (-paths[par + (v,)][1], v))[:k]
            for rank, v in enumerate(kids):
                cands.append((paths[par + (v,)][0], slot, rank, par + (v,)))
        cands.sort(key=lambda c: (-c[0], c[1], c[2]))
        frontier = [c[3] for c in cands[:P]]
        pool.extend((paths[f][0], d, len(pool), f) for f in frontier)
    pool.sort(key=lambda t: (-t[0], t[1], t[2]))
    return [t[3] for t in pool[:N]]


def _tree_paths(tr, i):
    out = []
    for c in range(1, tr["n_nodes"][i]):
        p, a = [], c
        while a > 0:
            p.append(int(tr["tok"][i, a]))
            a = tr["parent"][i, a]
        out.append(tuple(reversed(p)))
    return out


@pytest.mark.parametrize("V,B,k,P,N", [(5, 3, 2, 3, 6), (4, 3, 3, 4, 9), (6, 2, 2, 2, 3), (3, 3, 2, 8, 10)])
def test_tree_matches_brute_force_beam(V, B, k, P, N):
    w = small(R=3, B=B, V=V, r=8, l_std=1.0)
    inp = _inputs(w, seed=V * 10 + B)
    L, U, W, an = np_of(inp["L"]), np_of(inp["U"]), np_of(inp["W"]), np_of(inp["anchor"])
    tr = oracle.draft_tree(L, U, W, an, k=k, P=P, N=N)
    for i in range(w.R):
        paths = _all_paths(L[i], U, W, an[i], B)
        ref = _beam_reference(paths, V, B, k, P, N)
        assert _tree_paths(tr, i) == ref
        for c in range(1, tr["n_nodes"][i]):
            assert tr["parent"][i, c] < c
            assert tr["score"][i, c] == pytest.approx(paths[_tree_paths(tr, i)[c - 1]][0], abs=1e-12)


def test_tree_without_pruning_maximises_path_mass():
    """k = V and P >= V^B: the selected N nodes maximise sum exp(s) over all
    ancestor-closed node sets of size N (top-N by path probability)."""
    V, B, N = 3, 3, 4
    w = small(R=2, B=B, V=V, r=8, l_std=1.2)
    inp = _inputs(w, seed=1)
    L, U, W, an = np_of(inp["L"]), np_of(inp["U"]), np_of(inp["W"]), np_of(inp["anchor"])
    tr = oracle.draft_tree(L, U, W, an, k=V, P=V ** B, N=N)
    for i in range(w.R):
        paths = _all_paths(L[i], U, W, an[i], B)
        nodes = list(paths)
        best = -1.0
        for sub in itertools.combinations(nodes, N):
            ss = set(sub)
            if all(p[:-1] in ss or len(p) == 1 for p in sub):
                best = max(best, sum(math.exp(paths[p][0]) for p in sub))
        got = sum(math.exp(paths[p][0]) for p in _tree_paths(tr, i))
        assert got == pytest.approx(best, rel=1e-12)


def test_tree_mask_is_ancestor_closure():
    w = small(R=4, B=4, V=50, r=16)
    inp = _inputs(w, seed=3)
    tr = oracle.draft_tree(np_of(inp["L"]), np_of(inp["U"]), np_of(inp["W"]), np_of(inp["anchor"]), k=3, P=4, N=10)
    S = 11
    for i in range(w.R):
        for c in range(S):
            bits = tr["mask"][i, c, 0]
            if c >= tr["n_nodes"][i]:
                assert bits == 0
                continue
            anc = set()
            a = c
            while a >= 0:
                anc.add(a)
                a = tr["parent"][i, a]
            assert {j for j in range(S) if bits >> j & 1} == anc


def test_tree_verify_walks_longest_accepted_path():
    # hand-built tree: root(5) -> {1: tok 2, 2: tok 3}; 1 -> {3: tok 4}; 2 -> {4: tok 4}
    V, B, N = 8, 3, 4
    tok = np.array([[5, 2, 3, 4, 4]], np.int32)
    parent = np.array([[-1, 0, 0, 1, 2]], np.int32)
    n_nodes = np.array([5], np.int32)
    # target argmax per slot: root -> 3 (accept slot 2), slot 2 -> 4 (accept slot 4), slot 4 -> 6 (bonus)
    am = [3, 0, 4, 0, 6]
    target = _onehot_rows(am, V).reshape(1, 5, V)
    vr = oracle.verify_tree(target, tok, parent, n_nodes, B)
    assert vr["accept"].tolist() == [2] and vr["out_tok"][0, :3].tolist() == [3, 4, 6]
    # a chain-shaped tree verifies like the chain
    w = small(R=6, B=5, V=64, r=16, sigma=(0.5,))
    inp = _inputs(w, seed=6)
    args = (np_of(inp["L"]), np_of(inp["U"]), np_of(inp["W"]), np_of(inp["anchor"]))
    tr = oracle.draft_tree(*args, k=1, P=2, N=w.B)
    tgt = synthetic.tree_target(inp, torch.as_tensor(tr["tok"]), torch.as_tensor(tr["depth"]),
                                torch.as_tensor(tr["n_nodes"]), FP32)
    vt = oracle.verify_tree(np_of(tgt), tr["tok"], tr["parent"], tr["n_nodes"], w.B)
    cu = np.arange(w.R + 1, dtype=np.int32) * (w.B + 1)
    vc = oracle.verify(oracle.STATIC, oracle.GREEDY, np_of(tgt.reshape(-1, w.V)), cu, args[3], tr["tok"][:, 1:])
    np.testing.assert_array_equal(vt["accept"], vc["accept"])
    np.testing.assert_array_equal(vt["out_tok"], vc["out_tok"])


# ---------------------------------------------------------------------------
# observability: the soft label 1 - TV(q, p) and the verify-cycle statistics
# ---------------------------------------------------------------------------
def test_tv_label_is_the_first_accept_probability():
    """Rejection sampling accepts y_1 ~ q_1 with probability sum_v min(q, p)
    ([DSpark notes] sec. 5.1, the soft label); position 2 is accepted, given
    y_1 was, with the label of row 1 along that y_1.  Both are checked
    against the accept frequencies of the oracle's own verify."""
    n, V, B = 1 << 15, 8, 3
    w = small(R=n, B=B, V=V, r=4, sigma=(0.9,), l_std=1.0, temperature=1.3)
    base = _inputs(small(R=1, B=B, V=V, r=4, sigma=(0.9,), l_std=1.0, temperature=1.3), seed=4)
    inp = {k: (v.expand(n, *v.shape[1:]).contiguous() if k in ("L", "L_bonus", "eta", "anchor") else v)
           for k, v in base.items()}
    anchor = np.full(n, int(base["anchor"][0]), np.int32)
    dr, tgt, vr = _sample_cycle(w, inp, anchor, seed=21, cycle=0)
    cu = np.arange(n + 1, dtype=np.int32) * (B + 1)
    lab = oracle.tv_label(np_of(tgt.reshape(n * (B + 1), -1)), cu, anchor, dr["tokens"], np_of(inp["L"]),
                          np_of(inp["U"]), np_of(inp["W"]), temperature=w.temperature)["label"]
    l0 = lab[0, 0]
    assert np.all(lab[:, 0] == l0) and 0.05 < l0 < 0.95
    f0 = np.mean(vr["accept"] >= 1)
    assert abs(f0 - l0) < 4.5 * math.sqrt(l0 * (1 - l0) / n)
    ok = vr["accept"] >= 1
    m = int(ok.sum())
    f1 = np.mean(vr["accept"][ok] >= 2)
    e1 = lab[ok, 1].mean()
    assert abs(f1 - e1) < 4.5 * math.sqrt(e1 * (1 - e1) / m)


def test_tv_label_two_token_closed_form_and_equal_rows():
    """V = 2: sum_v min(q_v, p_v) = 1 - |q_0 - p_0|; a target row equal to the
    draft's logits (no noise) gives 1; rows outside the window get -1."""
    w = small(R=6, B=4, V=2, r=4, sigma=(1.3,), l_std=1.2, temperature=0.7)
    inp = _inputs(w, seed=9)
    an = np_of(inp["anchor"])
    L, U, W = np_of(inp["L"]), np_of(inp["U"]), np_of(inp["W"])
    toks = np.random.default_rng(3).integers(0, 2, size=(w.R, w.B)).astype(np.int32)
    tgt = synthetic.chain_target(inp, torch.as_tensor(toks), w.target_dtype)
    win = np.array([4, 0, 2, 4, 1, 3])
    cu = np.zeros(w.R + 1, np.int32)
    rows = []
    for i in range(w.R):
        cu[i + 1] = cu[i] + win[i] + 1
        rows.append(np_of(tgt[i, : win[i] + 1]))
    packed = np.concatenate(rows)
    lab = oracle.tv_label(packed, cu, an, toks, L, U, W, temperature=w.temperature)["label"]
    u = torch.from_numpy(U.view(np.int16)).view(torch.bfloat16).double().numpy()
    wm = torch.from_numpy(W.view(np.int16)).view(torch.bfloat16).double().numpy()
    for i in range(w.R):
        for p in range(w.B):
            if p >= win[i]:
                assert lab[i, p] == -1.0
                continue
            prev = an[i] if p == 0 else toks[i, p - 1]
            z = (L[i, p].astype(np.float32) + (u[prev] @ wm).astype(np.float32)).astype(np.float64) / w.temperature
            q0 = 1.0 / (1.0 + math.exp(z[1] - z[0]))
            t = tgt[i, p].double().numpy() / w.temperature
            p0 = 1.0 / (1.0 + math.exp(t[1] - t[0]))
            assert abs(lab[i, p] - (1.0 - abs(q0 - p0))) < 1e-12
    # no target noise: p = q on every row
    w0 = small(R=3, B=3, V=40, r=8, sigma=(0.0,), l_std=1.0)
    inp0 = _inputs(w0, seed=2)
    toks0 = np.random.default_rng(4).integers(0, 40, size=(3, 3)).astype(np.int32)
    t0 = synthetic.chain_target(inp0, torch.as_tensor(toks0), w0.target_dtype)
    cu0 = np.arange(4, dtype=np.int32) * 4
    lab0 = oracle.tv_label(np_of(t0.reshape(12, -1)), cu0, np_of(inp0["anchor"]), toks0, np_of(inp0["L"]),
                           np_of(inp0["U"]), np_of(inp0["W"]), temperature=w0.temperature)["label"]
    np.testing.assert_allclose(lab0, 1.0, atol=1e-12)


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_observe_worked_example():
    g = _load("observe_worked_example.json")
    out = oracle.observe(np.array(g["conf"], np.float32), np.array(g["cu_seqlens"]), np.array(g["ceiling"]),
                         np.array(g["cls"]), g["n_class"], g["n_bins"])
    e = g["expected"]
    for k in ("hist", "reached", "hits", "bin_n", "bin_hit"):
        np.testing.assert_array_equal(out[k], np.array(e[k]), err_msg=k)
    np.testing.assert_allclose(out["bin_conf"], e["bin_conf"], atol=1e-6)
    assert abs(out["ece"] - e["ece"]) < 1e-6


def test_observe_single_bin_edges_and_counts():
    """One bin: ECE = |hits - sum conf| / N.  Confidence 1 and above fall in
    the top bin, NaN and negatives in bin 0 as 0.  With full windows the
    count reaching d+1 is the count of hits at d, and every class's
    histogram sums to its requests."""
    rng = np.random.default_rng(11)
    R, g, nc = 300, 6, 3
    conf = rng.random((R, g)).astype(np.float32)
    conf[0, 0], conf[1, 0], conf[2, 0], conf[3, 0] = 1.0, np.nan, 1.7, -0.2
    ceiling = rng.integers(0, g + 1, R).astype(np.int32)
    ceiling[:4] = 0
    cls = rng.integers(0, nc, R).astype(np.int32)
    cu = np.arange(R + 1, dtype=np.int32) * (g + 1)
    one = oracle.observe(conf, cu, ceiling, cls, nc, 1)
    N = one["bin_n"][0]
    assert N == one["reached"].sum() and one["bin_hit"][0] == one["hits"].sum()
    x = np.nan_to_num(conf, nan=0.0).clip(0, 1)
    obs = [(x[i, d - 1], d <= ceiling[i]) for i in range(R) for d in range(1, min(ceiling[i] + 1, g) + 1)]
    assert len(obs) == N
    assert abs(one["ece"] - abs(sum(h for _, h in obs) - sum(float(c) for c, _ in obs)) / N) < 1e-12
    ten = oracle.observe(conf, cu, ceiling, cls, nc, 10)
    assert ten["bin_n"][9] >= 2 and ten["bin_n"][0] >= 2                  # 1.0 and 1.7 on top; NaN, -0.2 at 0
    np.testing.assert_array_equal(ten["reached"][:, 1:], ten["hits"][:, :-1])
    np.testing.assert_array_equal(ten["hist"].sum(1), np.bincount(cls, minlength=nc))
    with pytest.raises(ValueError):
        oracle.observe(conf, cu, ceiling, np.full(R, nc, np.int32), nc, 4)


def test_observe_calibrated_confidence_has_small_ece():
    """Confidences equal to the true conditional accept probabilities (the
    soft labels) are calibrated against the observed outcomes; cubing them
    is not."""
    n, V, B = 1 << 13, 6, 3
    w = small(R=n, B=B, V=V, r=4, sigma=(1.0,), l_std=1.0)
    inp = _inputs(w, seed=12)
    an = np_of(inp["anchor"])
    dr, tgt, vr = _sample_cycle(w, inp, an, seed=5, cycle=0)
    cu = np.arange(n + 1, dtype=np.int32) * (B + 1)
    lab = oracle.tv_label(np_of(tgt.reshape(n * (B + 1), -1)), cu, an, dr["tokens"], np_of(inp["L"]),
                          np_of(inp["U"]), np_of(inp["W"]), temperature=w.temperature)["label"]
    cls = np.zeros(n, np.int32)
    good = oracle.observe(lab.astype(np.float32), cu, vr["ceiling"], cls, 1, 10)
    bad = oracle.observe((lab ** 3).astype(np.float32), cu, vr["ceiling"], cls, 1, 10)
    assert good["ece"] < 0.02 < 0.1 < bad["ece"]


# ---------------------------------------------------------------------------
# fixed-threshold verify length and the threshold sweep
# ---------------------------------------------------------------------------
def test_threshold_worked_example():
    g = _load("threshold_sweep_worked_example.json")
    conf = np.array(g["conf"], np.float32)
    out = oracle.threshold_sweep(conf, np.array(g["taus"], np.float32), np.array(g["ceiling"], np.int32))
    e = g["expected"]
    np.testing.assert_array_equal(out["drafts"], e["drafts"])
    np.testing.assert_array_equal(out["accepted"], e["accepted"])
    np.testing.assert_allclose(out["expected"], e["expected"], atol=1e-6)
    one = oracle.schedule_threshold(conf, 0.5)
    np.testing.assert_array_equal(one["budget"], e["budget_at_0.5"])
    assert one["total_tokens"] == e["total_tokens_at_0.5"]
    assert oracle.threshold_sweep(conf, [0.5])["accepted"][0] == -1       # no ceilings given


def test_threshold_zero_verifies_the_whole_block_and_sweep_is_monotone():
    """Threshold 0 is the fixed-length full verify (Fig. 5): every draft is
    sent and what is accepted is the static verify's count; raising the
    threshold never sends more drafts, and nothing above every confidence."""
    w = small(R=30, B=6, V=64, r=16, sigma=(0.6, 1.6), class_mix="alternate")
    inp = _inputs(w, seed=6)
    an = np_of(inp["anchor"])
    dr = oracle.draft_chain(np_of(inp["L"]), np_of(inp["U"]), np_of(inp["W"]), an)
    tgt = synthetic.chain_target(inp, torch.as_tensor(dr["tokens"]), w.target_dtype)
    cu = np.arange(w.R + 1, dtype=np.int32) * (w.B + 1)
    vr = oracle.verify(oracle.STATIC, oracle.GREEDY, np_of(tgt.reshape(w.R * (w.B + 1), -1)), cu, an, dr["tokens"])
    conf = np_of(inp["conf"])
    taus = np.linspace(0, 1, 21).astype(np.float32)
    sw = oracle.threshold_sweep(conf, taus, vr["accept"])
    assert sw["drafts"][0] == w.R * w.B and sw["accepted"][0] == vr["accept"].sum()
    assert np.all(np.diff(sw["drafts"]) <= 0) and np.all(np.diff(sw["accepted"]) <= 0)
    assert np.all(sw["accepted"] <= sw["drafts"]) and np.all(sw["expected"] <= sw["drafts"] + 1e-9)
    top = oracle.threshold_sweep(conf, [np.nextafter(conf.max(), np.float32(2))], vr["accept"])
    assert top["drafts"][0] == 0 and top["expected"][0] == 0.0
    # the single-threshold budgets are the sweep's lengths, and compact
    # verification with them commits min(ceiling, n) drafts
    for tau in (0.3, 0.6):
        b = oracle.schedule_threshold(conf, tau)["budget"]
        assert b.sum() == oracle.threshold_sweep(conf, [tau])["drafts"][0]
        pk = oracle.pack_ragged(an, dr["tokens"], b, np.array(w.tiers, np.int32))
        packed = synthetic.gather_packed(tgt, torch.as_tensor(pk["packed_req"]), torch.as_tensor(pk["packed_pos"]))
        vc = oracle.verify(oracle.COMPACT, oracle.GREEDY, np_of(packed), pk["cu_seqlens"], an, dr["tokens"])
        np.testing.assert_array_equal(vc["accept"], np.minimum(vr["accept"], b))


def test_threshold_expected_matches_rejection_sampling():
    """With each confidence the true accept probability of its drafted token,
    min(1, p(y)/q(y)), the survivals are the chances of accepting every draft
    up to d, so the expected accepted drafts at threshold 0 match what the
    oracle's rejection-sampling verify accepts (CLT bound from the exact
    variance of the accepted count)."""
    n, V, B = 1 << 13, 8, 4
    w = small(R=n, B=B, V=V, r=4, sigma=(0.8,), l_std=1.0)
    base = _inputs(small(R=1, B=B, V=V, r=4, sigma=(0.8,), l_std=1.0), seed=14)
    inp = {k: (v.expand(n, *v.shape[1:]).contiguous() if k in ("L", "L_bonus", "eta", "anchor") else v)
           for k, v in base.items()}
    anchor = np.full(n, int(base["anchor"][0]), np.int32)
    dr, tgt, vr = _sample_cycle(w, inp, anchor, seed=8, cycle=2)
    lp = torch.log_softmax(tgt[:, :B].double() / w.temperature, -1)
    lp_y = lp.gather(-1, torch.as_tensor(dr["tokens"]).long().unsqueeze(-1)).squeeze(-1).numpy()
    conf = np.minimum(1.0, np.exp(lp_y - dr["logq"])).astype(np.float32)
    sw = oracle.threshold_sweep(conf, [0.0], vr["ceiling"])
    S = np.cumprod(conf.astype(np.float64), axis=1)
    var = 0.0
    for i in range(n):      # A = sum_d 1[first d accepted]; E[1_d 1_e] = S_max(d, e)
        s = S[i]
        m2 = sum(s[max(d, e)] for d in range(B) for e in range(B))
        var += m2 - s.sum() ** 2
    assert abs(sw["accepted"][0] - sw["expected"][0]) < 4.5 * math.sqrt(var)
    assert abs(sw["expected"][0] - S.sum()) < 1e-6 * S.sum()


# ---------------------------------------------------------------------------
# RNN head
# ---------------------------------------------------------------------------
def _bf16_bits(x64):
    """Round doubles to bf16 bits through binary32, nearest-even (numpy)."""
    f = np.asarray(x64, np.float64).astype(np.float32)
    b = f.view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return b.astype(np.uint16)


def _f64_of_bf16(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("decode", [oracle.GREEDY, oracle.SAMPLE])
def test_rnn_without_memory_is_the_markov_head_on_tanh_table(decode):
    """A = 0 and x = 0 leave m_d = tanh(U[y_{d-1}]): the RNN draft is the
    Markov head's draft on the table bf16(tanh(U))."""
    w = small(R=12, B=5, V=300, r=16, sigma=(0.5,), l_std=1.0)
    inp = _inputs(w, seed=3)
    L, U, W, an = np_of(inp["L"]), np_of(inp["U"]), np_of(inp["W"]), np_of(inp["anchor"])
    A = np.zeros((w.r, w.r), np.uint16)
    X = np.zeros((w.R, w.B, w.r), np.uint16)
    U3 = _bf16_bits(_f64_of_bf16(U) * 4.0)                    # exact (a power of two), tanh well away from identity
    assert np.array_equal(_f64_of_bf16(U3), _f64_of_bf16(U) * 4.0)
    Ut = _bf16_bits(np.tanh(_f64_of_bf16(U3)))
    rnn = oracle.draft_chain_rnn(L, U3, W, A, X, an, decode=decode, temperature=0.9, seed=4, cycle=1)
    mk = oracle.draft_chain(L, Ut, W, an, decode=decode, temperature=0.9, seed=4, cycle=1)
    np.testing.assert_array_equal(rnn["tokens"], mk["tokens"])
    np.testing.assert_allclose(rnn["lse"], mk["lse"], rtol=0, atol=1e-12)


def test_rnn_zero_tables_draft_the_backbone_argmax():
    w = small(R=6, B=4, V=200, r=16, sigma=(0.5,))
    inp = _inputs(w, seed=5)
    L = np_of(inp["L"])
    rng = np.random.default_rng(0)
    A = _bf16_bits(rng.normal(0, 0.3, (w.r, w.r)))
    zero_u = np.zeros_like(np_of(inp["U"]))
    out = oracle.draft_chain_rnn(L, zero_u, np_of(inp["W"]), A, np.zeros((w.R, w.B, w.r), np.uint16),
                                 np_of(inp["anchor"]))
    np.testing.assert_array_equal(out["tokens"], L.argmax(-1))


def test_rnn_memo_small_signal_closed_form():
    """For small inputs tanh(v) = v - v^3/3 + ..., so the memo is the linear
    recurrence's closed form m_d = sum_k A^k (U[y_{d-1-k}] + x_{d-k}) to
    within the cubic terms carried through the recurrence (|A| < 1: at most
    d of them, each below max|v|^3 / 3)."""
    R, B, r, V = 5, 6, 16, 40
    rng = np.random.default_rng(7)
    eps = 2.0 ** -10
    A = _bf16_bits(rng.normal(0, 0.8 / math.sqrt(r), (r, r)))
    U = _bf16_bits(rng.normal(0, eps, (V, r)))
    X = _bf16_bits(rng.normal(0, eps, (R, B, r)))
    an = rng.integers(0, V, R).astype(np.int32)
    toks = rng.integers(0, V, (R, B)).astype(np.int32)
    memo = oracle.rnn_memo(A, U, X, an, toks)
    Af, Uf, Xf = _f64_of_bf16(A), _f64_of_bf16(U), _f64_of_bf16(X)
    powers = [np.eye(r)]
    for _ in range(B):
        powers.append(powers[-1] @ Af)
    for i in range(R):
        ys = np.concatenate([[an[i]], toks[i]])
        for d in range(1, B + 1):
            ref = sum(powers[k] @ (Uf[ys[d - 1 - k]] + Xf[i, d - 1 - k]) for k in range(d))
            err = np.abs(memo[i, d - 1] - ref).max()
            vmax = max(np.abs(memo[i, k]).max() for k in range(d)) * 1.01
            assert err <= d * vmax ** 3 / 3 + 1e-15, (i, d, err)
            assert err <= 1e-4 * np.abs(ref).max()


def test_rnn_memo_remembers_earlier_tokens():
    """With A != 0, m_3 depends on y_1; with A = 0 it depends only on y_2
    and x_3 (the Markov head's reach)."""
    R, B, r, V = 2, 3, 16, 30
    rng = np.random.default_rng(9)
    A = _bf16_bits(rng.normal(0, 0.5, (r, r)))
    U = _bf16_bits(rng.normal(0, 0.5, (V, r)))
    X = np.repeat(_bf16_bits(rng.normal(0, 0.5, (1, B, r))), R, axis=0)
    an = np.array([3, 3], np.int32)
    toks = np.array([[5, 7, 1], [6, 7, 1]], np.int32)          # differ at y_1 only
    m = oracle.rnn_memo(A, U, X, an, toks)
    assert np.abs(m[0, 2] - m[1, 2]).max() > 1e-3
    m0 = oracle.rnn_memo(np.zeros_like(A), U, X, an, toks)
    np.testing.assert_array_equal(m0[0, 2], m0[1, 2])
    np.testing.assert_array_equal(m0[0, 0], m0[1, 0])


def test_rnn_draft_follows_its_memo():
    """Every greedy draft token is the argmax of L_d + bf16(m_d) W with m_d
    the memo along the drafted tokens (the pinned recurrence above)."""
    w = small(R=8, B=5, V=120, r=16, sigma=(0.5,), l_std=0.5)
    inp = _inputs(w, seed=11)
    rnn = synthetic.rnn_inputs(w, seed=11)
    L, U, W, an = np_of(inp["L"]), np_of(inp["U"]), np_of(inp["W"]), np_of(inp["anchor"])
    A, X = np_of(rnn["A_rnn"]), np_of(rnn["X_rnn"])
    out = oracle.draft_chain_rnn(L, U, W, A, X, an)
    memo = oracle.rnn_memo(A, U, X, an, out["tokens"])
    mb = _f64_of_bf16(_bf16_bits(memo))
    z = L.astype(np.float32) + np.einsum("idr,rv->idv", mb, _f64_of_bf16(W)).astype(np.float32)
    np.testing.assert_array_equal(out["tokens"], z.argmax(-1))
    assert np.abs(memo).max() < 1.0 and np.abs(memo).max() > 0.3      # tanh range, not saturated away


@pytest.mark.parametrize("T", [1.0, 0.7])
def test_rnn_projection_of_a_given_memo_closed_forms(T):
    """The projection of a given memo (the GPU's memo enters the parity
    tests through it) reduces to library routines: a zero memo gives the
    backbone row's argmax and log-sum-exp (scipy), and a memo row c e_j (c a
    bf16 value) gives z = L + c W[j, :], whose argmax, log-sum-exp and
    inverse-CDF draw numpy forms directly."""
    R, B, V, r = 3, 4, 97 * 8, 16
    rng = np.random.default_rng(4)
    L = rng.normal(0, 1.5, (R, B, V)).astype(np.float32)
    W = _bf16_bits(rng.normal(0, 0.25, (r, V)))
    zero = np.zeros((R, B, r), np.float32)
    g = oracle.rnn_project(L, W, zero)
    np.testing.assert_array_equal(g["tokens"], L.argmax(-1))
    s = oracle.rnn_project(L, W, zero, decode=oracle.SAMPLE, temperature=T, seed=2, cycle=5)
    np.testing.assert_allclose(s["lse"], special.logsumexp(L.astype(np.float64) / T, axis=-1), rtol=1e-13)
    memo = np.zeros((R, B, r), np.float32)
    jj = rng.integers(0, r, (R, B))
    cc = _f64_of_bf16(_bf16_bits(rng.normal(0, 2.0, (R, B)))).astype(np.float32)
    for i in range(R):
        for d in range(B):
            memo[i, d, jj[i, d]] = cc[i, d]
    z = (L.astype(np.float32) + (cc[..., None].astype(np.float64) *
                                 _f64_of_bf16(W)[jj]).astype(np.float32)).astype(np.float32)
    g = oracle.rnn_project(L, W, memo)
    np.testing.assert_array_equal(g["tokens"], z.argmax(-1))
    s = oracle.rnn_project(L, W, memo, decode=oracle.SAMPLE, temperature=T, seed=2, cycle=5)
    zt = z.astype(np.float64) / T
    np.testing.assert_allclose(s["lse"], special.logsumexp(zt, axis=-1), rtol=1e-13)
    for i in range(R):
        for d in range(B):
            wts = np.exp(zt[i, d] - zt[i, d].max())
            u = oracle.uniform(2, 5, oracle.STREAM_DRAFT, i, d + 1, 0)
            y = int(np.searchsorted(np.cumsum(wts), u * wts.sum(), side="right"))
            assert s["tokens"][i, d] == y
            assert abs(s["logq"][i, d] - (zt[i, d, y] - s["lse"][i, d])) < 1e-12


def test_rnn_projection_follows_the_rnn_draft():
    """Fed the memo of the oracle's own RNN draft (rounded to fp32), the
    projection takes the same decisions as the draft, position by position."""
    w = small(R=6, B=5, V=400, r=32, sigma=(0.5,), l_std=1.0)
    inp = _inputs(w, seed=12)
    rnn = synthetic.rnn_inputs(w, seed=12)
    L, U, W, an = np_of(inp["L"]), np_of(inp["U"]), np_of(inp["W"]), np_of(inp["anchor"])
    A, X = np_of(rnn["A_rnn"]), np_of(rnn["X_rnn"])
    for dec in (oracle.GREEDY, oracle.SAMPLE):
        dr = oracle.draft_chain_rnn(L, U, W, A, X, an, decode=dec, temperature=0.8, seed=1, cycle=2)
        memo = oracle.rnn_memo(A, U, X, an, dr["tokens"])
        pj = oracle.rnn_project(L, W, memo.astype(np.float32), decode=dec, temperature=0.8, seed=1, cycle=2)
        same_bf16 = np.all(_bf16_bits(memo) == _bf16_bits(memo.astype(np.float32)), axis=-1)
        assert same_bf16.mean() > 0.9
        np.testing.assert_array_equal(pj["tokens"][same_bf16], dr["tokens"][same_bf16])
        np.testing.assert_allclose(pj["lse"][same_bf16], dr["lse"][same_bf16], rtol=1e-14)


def test_verify_margins_belong_to_their_decisions():
    """One margin per accept test and one for the final draw: the test of
    row p reports |ln u - ln(p/q)| with u the accept uniform of that row,
    rows past the rejection report none (infinity), and greedy decisions
    report none at all."""
    w = small(R=10, B=5, V=64, r=16, l_dtype=FP32, target_dtype=FP32, sigma=(0.8,), temperature=1.0)
    inp = _inputs(w, seed=8)
    an, U, W = np_of(inp["anchor"]), np_of(inp["U"]), np_of(inp["W"])
    dr = oracle.draft_chain(np_of(inp["L"]), U, W, an, decode=oracle.SAMPLE, seed=3, cycle=0)
    pk = oracle.pack_ragged(an, dr["tokens"], None, np.array([64], np.int32))
    tgt = synthetic.chain_target(inp, torch.as_tensor(dr["tokens"]), FP32)
    packed = np_of(synthetic.gather_packed(tgt, torch.as_tensor(pk["packed_req"]), torch.as_tensor(pk["packed_pos"])))
    ref = oracle.verify(oracle.STATIC, oracle.SAMPLE, packed, pk["cu_seqlens"], an, dr["tokens"], logq=dr["logq"],
                        lse_q=dr["lse"], L=np_of(inp["L"]), U=U, W=W, seed=3, cycle=0)
    assert ref["margin"].shape == (w.R, w.B + 1)
    cu = pk["cu_seqlens"]
    for i in range(w.R):
        A = ref["ceiling"][i]
        for p in range(w.B):
            if p > A or (p == A and A == w.B):
                assert ref["margin"][i, p] == np.inf
                continue
            row = packed[cu[i] + p].astype(np.float64)
            lp = row[dr["tokens"][i, p]] - special.logsumexp(row)
            lu = math.log(oracle.uniform(3, 0, oracle.STREAM_ACCEPT, i, p, 0))
            assert abs(ref["margin"][i, p] - abs(lu - (lp - dr["logq"][i, p]))) < 1e-9
            assert (lu < lp - dr["logq"][i, p]) == (p < A)
        assert 0 <= ref["margin"][i, w.B] < 1
    gr = oracle.verify(oracle.STATIC, oracle.GREEDY, packed, cu, an, dr["tokens"])
    assert np.all(gr["margin"] == np.inf)


def test_tree_margins_belong_to_their_decisions():
    """The tree's margins: level d's prune boundary gap equals the gap
    between the P-th and (P+1)-th candidate of a brute-force replay of that
    level (scores in double), the top-N gap and the ranking gap follow the
    output scores."""
    w = small(R=3, B=3, V=16, r=16, l_dtype=FP32, sigma=(0.5,), l_std=1.0)
    inp = _inputs(w, seed=6)
    L, U, W, an = np_of(inp["L"]), np_of(inp["U"]), np_of(inp["W"]), np_of(inp["anchor"])
    k, P, N = 3, 2, 5
    out = oracle.draft_tree(L, U, W, an, k=k, P=P, N=N)
    assert out["margin"].shape == (w.R, w.B + 2)
    Wf, Uf = _f64_of_bf16(W), _f64_of_bf16(U)
    for i in range(w.R):
        front = [(an[i], 0.0)]
        pool = []
        for d in range(w.B):
            cands = []
            for slot, (tok, s) in enumerate(front):
                z = (L[i, d].astype(np.float32) + (Uf[tok] @ Wf).astype(np.float32)).astype(np.float32)
                lse = special.logsumexp(z.astype(np.float64))
                order = sorted(range(w.V), key=lambda v: (-z[v], v))[:k]
                cands += [(s + float(z[v]) - lse, slot, c, v) for c, v in enumerate(order)]
            cands.sort(key=lambda c: (-c[0], c[1], c[2]))
            gap = cands[P - 1][0] - cands[P][0] if len(cands) > P else np.inf
            assert abs(out["margin"][i, d] - gap) < 1e-9 or gap == out["margin"][i, d]
            front = [(c[3], c[0]) for c in cands[:P]]
            pool += [c[0] for c in cands[:P]]
        pool.sort(reverse=True)
        assert abs(out["margin"][i, w.B] - (pool[N - 1] - pool[N])) < 1e-9
        sc = out["score"][i, 1:out["n_nodes"][i]]
        assert abs(out["margin"][i, w.B + 1] - np.min(sc[:-1] - sc[1:])) < 1e-12
