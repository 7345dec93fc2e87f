"""GPU parity: every C-ABI operation against the CPU oracle on the same seeded
inputs.

Integer results (token ids, accept lengths, budgets, packed offsets, tree
indices, masks) must match bit for bit; fp32 log-prob sums and scores within
1e-5 relative (|gpu - oracle| <= 1e-5 * max(1, |oracle|)).  Sampling and tree
pruning decide integers from exp/log values that the kernel computes in fp32
and the oracle in fp64: a mismatch there is only tolerated when the oracle's
decision margin is below 1e-5 (a tie-zone event, reported), and none is
expected at these seeds.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_markov_gb300 import binding as sdm
from speculative_decoding_markov_gb300 import synthetic
from speculative_decoding_markov_gb300.workloads import BF16, FP32, WORKLOADS
from tests.helpers import np_of, small, tree_first_decision, verify_first_decision

pytestmark = pytest.mark.gpu
DEV = "cuda"
TIE = 1e-5
FTOL = 1e-5


def dev(t):
    return t.to(DEV).contiguous()


def host(t):
    return t.detach().cpu().numpy()


def close(gpu, ref, tol=FTOL):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    return np.abs(gpu - ref) <= tol * np.maximum(1.0, np.abs(ref))


def compare_sequences(gpu_tok, orc_tok, orc_margin, what):
    """Exact per-request comparison up to a tie-zone flip (then the rest of
    that request depends on a different prefix and is not compared)."""
    events = 0
    for i in range(orc_tok.shape[0]):
        mism = np.nonzero(gpu_tok[i] != orc_tok[i])[0]
        if mism.size:
            d = int(mism[0])
            assert orc_margin[i, d] < TIE, f"{what}: request {i} position {d} differs at margin {orc_margin[i, d]}"
            events += 1
    return events


# ---------------------------------------------------------------------------
# draft_chain
# ---------------------------------------------------------------------------
CHAIN_CASES = [
    dict(R=4, B=7, V=1024, r=64, l_dtype=FP32),          # tiny chain workload shape
    dict(R=64, B=4, V=1000, r=256, l_dtype=BF16),        # ragged vocab tail (15 tiles + 40)
    dict(R=200, B=3, V=520, r=128, l_dtype=BF16),        # two M tiles, ragged rows
    dict(R=1, B=2, V=8, r=64, l_dtype=FP32),             # smallest shapes
    dict(R=130, B=2, V=4160, r=64, l_dtype=FP32),
]


@pytest.mark.parametrize("case", CHAIN_CASES, ids=lambda c: f"R{c['R']}B{c['B']}V{c['V']}r{c['r']}")
def test_draft_chain_greedy(case):
    w = small(sigma=(0.5,), **case)
    inp = synthetic.generate(w, seed=case["R"] + case["V"])
    ref = oracle.draft_chain(np_of(inp["L"]), np_of(inp["U"]), np_of(inp["W"]), np_of(inp["anchor"]))
    assert ref["flags"] == 0
    out = sdm.draft_chain(dev(inp["L"]), dev(inp["U"]), dev(inp["W"]), dev(inp["anchor"]))
    torch.cuda.synchronize()
    assert int(out["dev_status"].item()) == 0
    np.testing.assert_array_equal(host(out["tokens"]), ref["tokens"])


@pytest.mark.parametrize("case", CHAIN_CASES + [dict(R=3, B=4, V=151936, r=256, l_dtype=BF16),
                                                dict(R=2, B=3, V=50000, r=64, l_dtype=FP32)],
                         ids=lambda c: f"R{c['R']}B{c['B']}V{c['V']}r{c['r']}")
def test_draft_chain_greedy_prepared(case):
    """The bound-pruned greedy chain (prepared tables) against the oracle and
    bit for bit against the dense tensor-core path."""
    w = small(sigma=(0.5,), **case)
    inp = synthetic.generate(w, seed=case["R"] * 7 + case["V"])
    d = {k: dev(v) for k, v in inp.items()}
    prep = sdm.markov_prepare(d["U"], d["W"])
    pr = sdm.draft_chain(d["L"], d["U"], d["W"], d["anchor"], prepared=prep)
    dn = sdm.draft_chain(d["L"], d["U"], d["W"], d["anchor"])
    torch.cuda.synchronize()
    assert int(pr["dev_status"].item()) == 0
    ref = oracle.draft_chain(np_of(inp["L"]), np_of(inp["U"]), np_of(inp["W"]), np_of(inp["anchor"]))
    np.testing.assert_array_equal(host(pr["tokens"]), ref["tokens"])
    assert torch.equal(pr["tokens"], dn["tokens"])


def _prepared_views(raw, V, r):
    """The arrays of the prepared-tables buffer (each on a 256-byte boundary)."""
    def up(x):
        return (x + 255) // 256 * 256
    out, off = {}, 0
    for name, n, dt in (("wt", V * r * 2, torch.bfloat16), ("c", V * 4, torch.float32),
                        ("u_norm", V * 4, torch.float32), ("absmax", V * 4, torch.float32),
                        ("c_max", 4, torch.float32), ("n_max", 4, torch.float32), ("u_max", 4, torch.float32)):
        out[name] = raw[off: off + n].view(dt)
        off += up(n)
    out["wt"] = out["wt"].view(V, r)
    return out


def _check_bounds(c, U, W, ys, u_norm, n_max, r):
    """c(y) bounds max_v |U[y] . W[:, v]| (exact, fp64) from above, and by no
    more than the stated slack."""
    exact = (U[ys].double() @ W.double()).abs().max(dim=1).values
    slack = 4 * r * 2.0 ** -24 * u_norm[ys].double() * float(n_max) + 2.0 ** -20
    cy = c[ys].double()
    assert torch.all(cy >= exact), "bound below the exact maximum"
    assert torch.all(cy <= exact * (1 + 2.0 ** -10) * (1 + 1e-6) + slack + 1e-7), "bound looser than stated"


def test_markov_prepare_tables():
    w = small(R=1, B=1, V=1000, r=128, sigma=(0.5,))
    inp = synthetic.generate(w, seed=2)
    prep = sdm.markov_prepare(dev(inp["U"]), dev(inp["W"]))
    torch.cuda.synchronize()
    V, r = w.V, w.r
    t = _prepared_views(prep.cpu(), V, r)
    assert torch.equal(t["wt"], inp["W"].t().contiguous())
    u_ref = inp["U"].double().norm(dim=1)
    assert float(t["u_max"]) >= float(u_ref.max()) and float(t["u_max"]) <= float(u_ref.max()) * (1 + 1e-6)
    assert torch.all(t["u_norm"].double() >= u_ref) and torch.all(t["u_norm"].double() <= u_ref * (1 + 1e-6) + 1e-30)
    w_ref = inp["W"].double().norm(dim=0).max()
    assert float(t["n_max"]) >= float(w_ref) and float(t["n_max"]) <= float(w_ref) * (1 + 1e-6)
    _check_bounds(t["c"], inp["U"], inp["W"], torch.arange(V), t["u_norm"], t["n_max"], r)
    assert float(t["c_max"]) == float(t["c"].max())


def test_markov_prepare_bounds_full_vocab():
    """The absolute-maximum GEMM at the 152K vocabulary (1187 M tiles, every
    vocab tile): sampled tokens, and c_max against the sampled maxima."""
    w = small(R=1, B=1, V=151936, r=256, sigma=(0.5,))
    inp = synthetic.generate(w, seed=4)
    prep = sdm.markov_prepare(dev(inp["U"]), dev(inp["W"]))
    torch.cuda.synchronize()
    t = _prepared_views(prep.cpu(), w.V, w.r)
    g = torch.Generator().manual_seed(1)
    ys = torch.cat([torch.randint(0, w.V, (96,), generator=g), torch.tensor([0, 127, 128, w.V - 1])])
    _check_bounds(t["c"], inp["U"], inp["W"], ys, t["u_norm"], t["n_max"], w.r)
    assert float(t["c_max"]) == float(t["c"].max())
    assert float(t["c_max"]) < float(t["u_max"]) * float(t["n_max"])   # tighter than Cauchy-Schwarz


@pytest.mark.parametrize("kind", ["all_equal", "outlier", "ties", "wide_markov", "crowded", "crowded_mid",
                                  "crowded_long"])
def test_draft_chain_prepared_adversarial(kind):
    """Inputs that defeat the pruning bound (every id a candidate: many batches),
    exact ties (lowest id wins), a dominant Markov term, and crowded rows whose
    candidates overflow the shared-memory staging (later steps score from
    global memory; with 64 steps the lists themselves stay in global memory)."""
    R, B, V, r = 3, 3, 8192, 64
    if kind == "crowded":
        B = 24
    elif kind == "crowded_long":
        R, B = 2, 64
    w = small(R=R, B=B, V=V, r=r, l_dtype=BF16, sigma=(0.5,))
    inp = synthetic.generate(w, seed=9)
    L = inp["L"].clone()
    if kind == "all_equal":
        L[:] = 0.5
    elif kind == "outlier":
        L[:, :, 4321] = 50.0
    elif kind == "ties":
        L = torch.round(L.float() * 2).to(torch.bfloat16) / 2          # many exact ties
    elif kind == "wide_markov":
        L = (L.float() * 0.01).to(torch.bfloat16)                      # the Markov term decides
    elif kind == "crowded_mid":
        L = (L.float() * 0.5).to(torch.bfloat16)                       # lists around the pick's loaded head
    else:
        L = (L.float() * 0.3).to(torch.bfloat16)                       # ~60 candidates per step
    d = {k: dev(v) for k, v in inp.items()}
    d["L"] = dev(L)
    prep = sdm.markov_prepare(d["U"], d["W"])
    pr = sdm.draft_chain(d["L"], d["U"], d["W"], d["anchor"], prepared=prep)
    torch.cuda.synchronize()
    ref = oracle.draft_chain(np_of(L), np_of(inp["U"]), np_of(inp["W"]), np_of(inp["anchor"]))
    np.testing.assert_array_equal(host(pr["tokens"]), ref["tokens"])


@pytest.mark.parametrize("case,T", [(dict(R=40, B=5, V=2056, r=64, l_dtype=BF16), 0.7),
                                    (dict(R=150, B=2, V=512, r=128, l_dtype=FP32), 1.3),
                                    (dict(R=3, B=3, V=8, r=64, l_dtype=FP32), 1.0)])
def test_draft_chain_sample(case, T):
    w = small(sigma=(0.5,), **case)
    inp = synthetic.generate(w, seed=7)
    ref = oracle.draft_chain(np_of(inp["L"]), np_of(inp["U"]), np_of(inp["W"]), np_of(inp["anchor"]),
                             decode=oracle.SAMPLE, temperature=T, seed=99, cycle=5)
    out = sdm.draft_chain(dev(inp["L"]), dev(inp["U"]), dev(inp["W"]), dev(inp["anchor"]), decode=sdm.SAMPLE,
                          temperature=T, seed=99, cycle=5)
    torch.cuda.synchronize()
    tok = host(out["tokens"])
    events = compare_sequences(tok, ref["tokens"], ref["margin"], "sample chain")
    assert events == 0
    assert close(host(out["lse"]), ref["lse"]).all()
    assert close(host(out["logq"]), ref["logq"]).all()


def test_draft_chain_is_deterministic():
    w = small(R=96, B=3, V=4096, r=256, l_dtype=BF16, sigma=(0.5,))
    inp = {k: dev(v) for k, v in synthetic.generate(w, seed=3).items()}
    a = sdm.draft_chain(inp["L"], inp["U"], inp["W"], inp["anchor"], decode=sdm.SAMPLE, seed=1)
    b = sdm.draft_chain(inp["L"], inp["U"], inp["W"], inp["anchor"], decode=sdm.SAMPLE, seed=1)
    torch.cuda.synchronize()
    for key in ("tokens", "logq", "lse"):
        assert torch.equal(a[key], b[key])


def test_draft_chain_flags_bad_anchor_without_faulting():
    w = small(R=8, B=2, V=512, r=64, sigma=(0.5,))
    inp = synthetic.generate(w, seed=1)
    anchor = inp["anchor"].clone()
    anchor[3] = w.V + 17
    out = sdm.draft_chain(dev(inp["L"]), dev(inp["U"]), dev(inp["W"]), dev(anchor))
    torch.cuda.synchronize()
    assert int(out["dev_status"].item()) & sdm.DEV_BAD_TOKEN
    ok = [i for i in range(w.R) if i != 3]
    ref = oracle.draft_chain(np_of(inp["L"][ok]), np_of(inp["U"]), np_of(inp["W"]), np_of(inp["anchor"][ok]))
    np.testing.assert_array_equal(host(out["tokens"])[ok], ref["tokens"])


# ---------------------------------------------------------------------------
# schedule_budget
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("R,g,seed", [(1, 1, 0), (5, 7, 1), (64, 7, 2), (256, 8, 3), (512, 16, 4), (33, 16, 5)])
def test_schedule_budget(R, g, seed):
    rng = np.random.default_rng(seed)
    conf = rng.uniform(0.02, 1.0, (R, g)).astype(np.float32)
    conf[rng.random((R, g)) < 0.1] = 1.0                  # exact ties in S
    a, b = float(rng.uniform(0.5, 3.0)), float(rng.uniform(0.001, 0.2))
    cost = a + b * np.arange(R * (g + 1) + 1, dtype=np.float64)
    ref = oracle.schedule_budget(conf, cost)
    out = sdm.schedule_budget(dev(torch.from_numpy(conf)), dev(torch.from_numpy(cost)))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host(out["survival"]).view(np.uint32), ref["survival"].view(np.uint32))
    np.testing.assert_array_equal(host(out["budget"]), ref["budget"])
    if R * (g + 1) < 4096:                                 # fp64 sums exact in any order
        assert float(host(out["expected"])[0]) == ref["expected"]
    else:
        assert close(host(out["expected"]), [ref["expected"]], 1e-12).all()
    assert int(host(out["total_tokens"])[0]) == ref["total_tokens"]


def test_schedule_flushes_tiny_survivals_and_breaks_ties_by_request():
    R, g = 6, 5
    conf = np.full((R, g), 0.5, np.float32)
    conf[2] = 0.01                                         # S falls below 2^-18 by k = 3
    cost = 1.0 + 0.0001 * np.arange(R * (g + 1) + 1)
    ref = oracle.schedule_budget(conf, cost)
    out = sdm.schedule_budget(dev(torch.from_numpy(conf)), dev(torch.from_numpy(cost)))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host(out["budget"]), ref["budget"])
    assert ref["budget"][2] <= 2


def _tiered_cost(R, g, rng):
    """Step cost by total verify tokens: a + b * (the tier the total rounds up to)."""
    tiers = np.array([64, 128, 256, 512, 1024, 2048, 4096], np.int64)
    N = np.arange(R * (g + 1) + 1)
    t = np.array([tiers[np.searchsorted(tiers, n)] if n <= tiers[-1] else n for n in N], np.float64)
    return float(rng.uniform(0.5, 3.0)) + float(rng.uniform(0.001, 0.02)) * t


@pytest.mark.parametrize("R,g,seed", [(1, 4, 0), (4, 7, 1), (64, 7, 2), (256, 8, 3), (450, 8, 4), (37, 3, 5),
                                      (256, 16, 6), (512, 16, 7)])   # the rejection-sampling shape; R gamma = 8192
def test_schedule_dynamic(R, g, seed):
    """Capacity, budgets, survivals, E and N bit-exact against the oracle on a
    tiered cost table (E stays below 4096 at these shapes, so the fp64 sums of
    survivals >= 2^-18 are exact in any order); 450 x 8 sorts 4096 keys and
    512 x 16 the largest supported set, several per thread."""
    rng = np.random.default_rng(seed)
    now = rng.uniform(0.02, 1.0, (R, g)).astype(np.float32)
    stale = np.clip(now + rng.normal(0, 0.2, (R, g)), 0.02, 1.0).astype(np.float32)
    now[rng.random((R, g)) < 0.1] = 1.0                    # exact ties in S
    cost = _tiered_cost(R, g, rng)
    ref = oracle.schedule_dynamic(now, stale, cost)
    out = sdm.schedule_dynamic(dev(torch.from_numpy(now)), dev(torch.from_numpy(stale)), dev(torch.from_numpy(cost)))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host(out["survival"]).view(np.uint32), ref["survival"].view(np.uint32))
    assert int(host(out["capacity"])[0]) == ref["capacity"]
    np.testing.assert_array_equal(host(out["budget"]), ref["budget"])
    assert float(host(out["expected"])[0]) == ref["expected"]
    assert int(host(out["total_tokens"])[0]) == ref["total_tokens"]


def test_schedule_dynamic_cliff_fixture_and_additive_agreement():
    import json, os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "sps_cliff_dynamic_scheduler.json")))
    R, gam = g["R"], g["gamma"]
    cost = np.zeros(R * (gam + 1) + 1, np.float64)
    for n, c in g["cost_by_tokens"].items():
        cost[int(n)] = c
    cost[:R] = cost[R]
    out = sdm.schedule_dynamic(dev(torch.tensor(g["conf_now"], dtype=torch.float32)),
                               dev(torch.tensor(g["conf_stale"], dtype=torch.float32)), dev(torch.from_numpy(cost)))
    torch.cuda.synchronize()
    assert int(host(out["capacity"])[0]) == g["expected_capacity"]
    assert host(out["budget"]).tolist() == g["expected_budget"]
    assert int(host(out["total_tokens"])[0]) == g["expected_total_tokens"]
    # equal confidences, additive table: the same budgets as the early-stopping scheduler
    rng = np.random.default_rng(9)
    conf = dev(torch.from_numpy(rng.uniform(0.05, 1.0, (128, 8)).astype(np.float32)))
    add = dev(torch.from_numpy(2.0 + 0.004 * np.arange(128 * 9 + 1)))
    a = sdm.schedule_dynamic(conf, conf, add)
    b = sdm.schedule_budget(conf, add)
    torch.cuda.synchronize()
    assert torch.equal(a["budget"], b["budget"]) and torch.equal(a["expected"], b["expected"])


# ---------------------------------------------------------------------------
# pack_ragged
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("strict", [False, True], ids=["uncaptured", "strict"])
@pytest.mark.parametrize("R,g,seed,static", [(1, 1, 0, False), (37, 8, 1, False), (256, 8, 2, False),
                                             (256, 8, 3, True), (1500, 2, 4, False)])
def test_pack_ragged(R, g, seed, static, strict):
    rng = np.random.default_rng(seed)
    anchor = rng.integers(0, 5000, R).astype(np.int32)
    draft = rng.integers(0, 5000, (R, g)).astype(np.int32)
    budget = rng.integers(0, g + 1, R).astype(np.int32)
    budget[: max(1, R // 5)] = 0
    tiers = np.array([64, 128, 256, 512, 1024, 2048], np.int32)
    ref = oracle.pack_ragged(anchor, draft, None if static else budget, tiers, strict=strict)
    out = sdm.pack_ragged(dev(torch.from_numpy(anchor)), dev(torch.from_numpy(draft)),
                          None if static else dev(torch.from_numpy(budget)), dev(torch.from_numpy(tiers)),
                          strict=strict)
    torch.cuda.synchronize()
    t = ref["tier"]
    assert int(host(out["tier"])[0]) == t
    np.testing.assert_array_equal(host(out["cu_seqlens"]), ref["cu_seqlens"])
    for k in ("packed_tok", "packed_req", "packed_pos"):
        np.testing.assert_array_equal(host(out[k])[:t], ref[k])
    bits = int(out["dev_status"].item())
    assert bits == ref["flags"]                 # the same bit from both sides, nothing else
    # the status a caller maps the bits to: strict overflow is an error, uncaptured is not
    assert sdm.lib().sdm_status_of_device(bits) == (3 if ref["flags"] & oracle.FLAG_TIER_OVERFLOW else 0)
    if static and R * (g + 1) > 2048:
        assert ref["flags"] == (oracle.FLAG_TIER_OVERFLOW if strict else oracle.FLAG_TIER_UNCAPTURED)


# ---------------------------------------------------------------------------
# verify (greedy, all modes) on oracle-drafted inputs
# ---------------------------------------------------------------------------
def _oracle_chain_pipeline(w, seed, mode):
    inp = synthetic.generate(w, seed=seed)
    an = np_of(inp["anchor"])
    dr = oracle.draft_chain(np_of(inp["L"]), np_of(inp["U"]), np_of(inp["W"]), an)
    sc = oracle.schedule_budget(np_of(inp["conf"]), synthetic.cost_table(w).numpy())
    budget = sc["budget"]
    pk = oracle.pack_ragged(an, dr["tokens"], budget if mode == "compact" else None, np.array(w.tiers, np.int32))
    tgt = synthetic.chain_target(inp, torch.as_tensor(dr["tokens"]), w.target_dtype)
    packed = synthetic.gather_packed(tgt, torch.as_tensor(pk["packed_req"]), torch.as_tensor(pk["packed_pos"]))
    return inp, dr, budget, pk, packed


@pytest.mark.parametrize("mode", ["static", "compact", "cap_accept"])
@pytest.mark.parametrize("case", [dict(R=16, B=6, V=2048, r=64, l_dtype=BF16, target_dtype=BF16),
                                  dict(R=5, B=7, V=1024, r=64, l_dtype=FP32, target_dtype=FP32),
                                  dict(R=70, B=3, V=40008, r=64, l_dtype=BF16, target_dtype=BF16)],
                         ids=lambda c: f"R{c['R']}V{c['V']}")
def test_verify_greedy(mode, case):
    w = small(sigma=(0.1, 0.6, 1.5), class_mix="alternate", **case)
    inp, dr, budget, pk, packed = _oracle_chain_pipeline(w, 11, mode)
    om = {"static": oracle.STATIC, "compact": oracle.COMPACT, "cap_accept": oracle.CAP_ACCEPT}[mode]
    an = np_of(inp["anchor"])
    ref = oracle.verify(om, oracle.GREEDY, np_of(packed), pk["cu_seqlens"], an, dr["tokens"], budget=budget)
    gm = {"static": sdm.STATIC, "compact": sdm.COMPACT, "cap_accept": sdm.CAP_ACCEPT}[mode]
    out = sdm.verify(gm, sdm.GREEDY, dev(packed), dev(torch.from_numpy(pk["cu_seqlens"])), dev(inp["anchor"]),
                     dev(torch.from_numpy(dr["tokens"])), budget=dev(torch.from_numpy(budget)))
    torch.cuda.synchronize()
    assert int(out["dev_status"].item()) == 0
    for k in ("accept", "out_tok", "n_out"):
        np.testing.assert_array_equal(host(out[k]), ref[k])
    if mode == "cap_accept":
        np.testing.assert_array_equal(host(out["ceiling"]), ref["ceiling"])


def test_verify_greedy_empty_windows():
    """Budget 0 for every request: the window is the root only; the commit is
    the target token at row 0."""
    w = small(R=9, B=4, V=1024, r=64, l_dtype=BF16, target_dtype=BF16)
    inp = synthetic.generate(w, seed=2)
    an = np_of(inp["anchor"])
    dr = oracle.draft_chain(np_of(inp["L"]), np_of(inp["U"]), np_of(inp["W"]), an)
    budget = np.zeros(w.R, np.int32)
    pk = oracle.pack_ragged(an, dr["tokens"], budget, np.array([16], np.int32))
    tgt = synthetic.chain_target(inp, torch.as_tensor(dr["tokens"]), w.target_dtype)
    packed = synthetic.gather_packed(tgt, torch.as_tensor(pk["packed_req"]), torch.as_tensor(pk["packed_pos"]))
    ref = oracle.verify(oracle.COMPACT, oracle.GREEDY, np_of(packed), pk["cu_seqlens"], an, dr["tokens"])
    out = sdm.verify(sdm.COMPACT, sdm.GREEDY, dev(packed), dev(torch.from_numpy(pk["cu_seqlens"])),
                     dev(inp["anchor"]), dev(torch.from_numpy(dr["tokens"])))
    torch.cuda.synchronize()
    assert np.all(ref["accept"] == 0)
    np.testing.assert_array_equal(host(out["out_tok"]), ref["out_tok"])


def test_verify_greedy_flags_bad_windows_without_waiting():
    """A window without rows and a window past the packed rows are resolved
    as flagged failures (accept 0, one token 0); the other requests are
    verified as usual."""
    w = small(R=6, B=4, V=1024, r=64, l_dtype=BF16, target_dtype=BF16)
    inp = synthetic.generate(w, seed=4)
    an = np_of(inp["anchor"])
    dr = oracle.draft_chain(np_of(inp["L"]), np_of(inp["U"]), np_of(inp["W"]), an)
    pk = oracle.pack_ragged(an, dr["tokens"], None, np.array([64], np.int32))
    tgt = synthetic.chain_target(inp, torch.as_tensor(dr["tokens"]), w.target_dtype)
    rows = int(pk["cu_seqlens"][-1])
    packed = synthetic.gather_packed(tgt, torch.as_tensor(pk["packed_req"][:rows]),
                                     torch.as_tensor(pk["packed_pos"][:rows]))
    ref = oracle.verify(oracle.STATIC, oracle.GREEDY, np_of(packed), pk["cu_seqlens"], an, dr["tokens"])
    for bad, bit in (("inverted", sdm.DEV_BAD_WINDOW), ("past", sdm.DEV_CAPACITY)):
        cu = pk["cu_seqlens"].copy()
        if bad == "inverted":
            cu[3] = cu[2] - 1                    # request 2 inverted; request 3 grows
        else:
            cu[-1] = rows + 3                    # the last request runs past the buffer
        st = sdm.new_status(DEV)
        out = sdm.verify(sdm.STATIC, sdm.GREEDY, dev(packed), dev(torch.from_numpy(cu)), dev(inp["anchor"]),
                         dev(torch.from_numpy(dr["tokens"])), dev_status=st)
        torch.cuda.synchronize()
        assert int(st.item()) & bit
        flagged = 2 if bad == "inverted" else w.R - 1
        assert host(out["accept"])[flagged] == 0 and host(out["n_out"])[flagged] == 1
        assert host(out["out_tok"])[flagged, 0] == 0
        for i in range(w.R - 1):
            if bad == "inverted" and i in (2, 3):   # request 3 took request 2's rows
                continue
            assert host(out["accept"])[i] == ref["accept"][i]
            np.testing.assert_array_equal(host(out["out_tok"])[i], ref["out_tok"][i])


def _non_monotone_cu(cu):
    """cu[R] moved down to cu[2]: requests 2 .. R-2 end past cu[R] (the
    streams write rows below cu[R] only) and request R-1 has no rows."""
    bad = cu.copy()
    bad[-1] = bad[2]
    return bad


@pytest.mark.parametrize("decode", ["greedy", "sample"])
def test_verify_flags_windows_past_the_packed_total(decode):
    """A non-monotone cu_seqlens whose total cu[R] lies below a request's
    end: that request is flagged (SDM_DEV_BAD_WINDOW) and commits one token
    (0) instead of reading partials this call never wrote; requests inside
    the total are verified as usual.  Run after a larger call on the same
    workspace, so stale partials would be there to read."""
    w = small(R=6, B=4, V=2048, r=64, l_dtype=BF16, target_dtype=BF16, sigma=(0.5,), temperature=1.0)
    inp = synthetic.generate(w, seed=17)
    an = np_of(inp["anchor"])
    U, W = np_of(inp["U"]), np_of(inp["W"])
    samp = decode == "sample"
    dr = oracle.draft_chain(np_of(inp["L"]), U, W, an, decode=oracle.SAMPLE if samp else oracle.GREEDY, seed=4,
                            cycle=1)
    pk = oracle.pack_ragged(an, dr["tokens"], None, np.array([64], np.int32))
    tgt = synthetic.chain_target(inp, torch.as_tensor(dr["tokens"]), w.target_dtype)
    packed = dev(synthetic.gather_packed(tgt, torch.as_tensor(pk["packed_req"]), torch.as_tensor(pk["packed_pos"])))
    kw = {}
    okw = {}
    if samp:
        logq32, lse32 = dr["logq"].astype(np.float32), dr["lse"].astype(np.float32)
        kw = dict(logq=dev(torch.from_numpy(logq32)), lse_q=dev(torch.from_numpy(lse32)), L=dev(inp["L"]),
                  U=dev(inp["U"]), W=dev(inp["W"]), seed=4, cycle=1)
        okw = dict(logq=logq32.astype(np.float64), lse_q=lse32.astype(np.float64), L=np_of(inp["L"]), U=U, W=W,
                   seed=4, cycle=1)
    dec = sdm.SAMPLE if samp else sdm.GREEDY
    ref = oracle.verify(oracle.STATIC, oracle.SAMPLE if samp else oracle.GREEDY, np_of(packed.cpu()),
                        pk["cu_seqlens"], an, dr["tokens"], **okw)
    tokens = dev(torch.from_numpy(dr["tokens"]))
    ws = sdm.workspace(sdm.OP_VERIFY, w.R, w.B, w.V, w.r, packed.shape[0], device=DEV)
    full = sdm.verify(sdm.STATIC, dec, packed, dev(torch.from_numpy(pk["cu_seqlens"])), dev(inp["anchor"]), tokens,
                      ws=ws, **kw)
    st = sdm.new_status(DEV)
    cu = _non_monotone_cu(pk["cu_seqlens"])
    out = sdm.verify(sdm.STATIC, dec, packed, dev(torch.from_numpy(cu)), dev(inp["anchor"]), tokens,
                     ws=ws, dev_status=st, **kw)
    torch.cuda.synchronize()
    assert int(full["dev_status"].item()) == 0
    assert int(st.item()) & sdm.DEV_BAD_WINDOW
    assert not int(st.item()) & sdm.DEV_CAPACITY
    for i in range(w.R):
        if i < 2:
            first = verify_first_decision(ref, i, host(out["accept"])[i], host(out["ceiling"])[i],
                                          host(out["out_tok"])[i])
            assert first is None, f"request {i} differs at decision {first}"
        else:
            assert host(out["accept"])[i] == 0 and host(out["n_out"])[i] == 1, i
            assert host(out["out_tok"])[i, 0] == 0 and np.all(host(out["out_tok"])[i, 1:] == -1), i


# ---------------------------------------------------------------------------
# verify (rejection sampling)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("mode", ["static", "compact", "cap_accept"])
@pytest.mark.parametrize("case,T", [(dict(R=48, B=5, V=2048, r=64, l_dtype=BF16, target_dtype=FP32), 1.0),
                                    (dict(R=20, B=4, V=1000, r=128, l_dtype=FP32, target_dtype=BF16), 0.8)],
                         ids=["bf16L_fp32T", "fp32L_bf16T"])
def test_verify_sample(mode, case, T):
    w = small(sigma=(0.3, 1.0), class_mix="alternate", temperature=T, **case)
    inp = synthetic.generate(w, seed=21)
    an = np_of(inp["anchor"])
    U, W = np_of(inp["U"]), np_of(inp["W"])
    dr = oracle.draft_chain(np_of(inp["L"]), U, W, an, decode=oracle.SAMPLE, temperature=T, seed=5, cycle=3)
    logq32 = dr["logq"].astype(np.float32)
    lse32 = dr["lse"].astype(np.float32)
    budget = np.random.default_rng(1).integers(0, w.B + 1, w.R).astype(np.int32)
    pk = oracle.pack_ragged(an, dr["tokens"], budget if mode == "compact" else None, np.array(w.tiers, np.int32))
    tgt = synthetic.chain_target(inp, torch.as_tensor(dr["tokens"]), w.target_dtype)
    packed = synthetic.gather_packed(tgt, torch.as_tensor(pk["packed_req"]), torch.as_tensor(pk["packed_pos"]))
    om = {"static": oracle.STATIC, "compact": oracle.COMPACT, "cap_accept": oracle.CAP_ACCEPT}[mode]
    ref = oracle.verify(om, oracle.SAMPLE, np_of(packed), pk["cu_seqlens"], an, dr["tokens"], budget=budget,
                        logq=logq32.astype(np.float64), lse_q=lse32.astype(np.float64), L=np_of(inp["L"]), U=U, W=W,
                        temperature=T, seed=5, cycle=3)
    gm = {"static": sdm.STATIC, "compact": sdm.COMPACT, "cap_accept": sdm.CAP_ACCEPT}[mode]
    out = sdm.verify(gm, sdm.SAMPLE, dev(packed), dev(torch.from_numpy(pk["cu_seqlens"])), dev(inp["anchor"]),
                     dev(torch.from_numpy(dr["tokens"])), budget=dev(torch.from_numpy(budget)),
                     logq=dev(torch.from_numpy(logq32)), lse_q=dev(torch.from_numpy(lse32)), L=dev(inp["L"]),
                     U=dev(inp["U"]), W=dev(inp["W"]), temperature=T, seed=5, cycle=3)
    torch.cuda.synchronize()
    assert int(out["dev_status"].item()) == 0
    events = 0
    for i in range(w.R):
        first = verify_first_decision(ref, i, host(out["accept"])[i], host(out["ceiling"])[i], host(out["out_tok"])[i])
        if first is not None:   # only a decision inside the tie zone may differ, and none is expected
            assert first[1] < TIE, f"request {i} differs at decision {first[0]}, margin {first[1]}"
            events += 1
    assert events == 0, f"{events} tie-zone events"
    if mode == "cap_accept":
        np.testing.assert_array_equal(host(out["ceiling"]), ref["ceiling"])


def test_verify_sample_flags_windows_past_the_buffer():
    """A window whose rows run past the packed buffer is flagged and commits
    one token (0) with accept 0; the other requests are verified as usual."""
    w = small(R=8, B=4, V=2048, r=64, l_dtype=BF16, target_dtype=FP32, sigma=(0.5,), temperature=1.0)
    inp = synthetic.generate(w, seed=13)
    an = np_of(inp["anchor"])
    U, W = np_of(inp["U"]), np_of(inp["W"])
    dr = oracle.draft_chain(np_of(inp["L"]), U, W, an, decode=oracle.SAMPLE, seed=2, cycle=0)
    logq32, lse32 = dr["logq"].astype(np.float32), dr["lse"].astype(np.float32)
    pk = oracle.pack_ragged(an, dr["tokens"], None, np.array([64], np.int32))
    rows = int(pk["cu_seqlens"][-1])
    tgt = synthetic.chain_target(inp, torch.as_tensor(dr["tokens"]), w.target_dtype)
    packed = synthetic.gather_packed(tgt, torch.as_tensor(pk["packed_req"][:rows]),
                                     torch.as_tensor(pk["packed_pos"][:rows]))
    ref = oracle.verify(oracle.STATIC, oracle.SAMPLE, np_of(packed), pk["cu_seqlens"], an, dr["tokens"],
                        logq=logq32.astype(np.float64), lse_q=lse32.astype(np.float64), L=np_of(inp["L"]), U=U, W=W,
                        seed=2, cycle=0)
    cu = pk["cu_seqlens"].copy()
    cu[-1] = rows + 5                            # the last request runs past the buffer
    st = sdm.new_status(DEV)
    out = sdm.verify(sdm.STATIC, sdm.SAMPLE, dev(packed), dev(torch.from_numpy(cu)), dev(inp["anchor"]),
                     dev(torch.from_numpy(dr["tokens"])), logq=dev(torch.from_numpy(logq32)),
                     lse_q=dev(torch.from_numpy(lse32)), L=dev(inp["L"]), U=dev(inp["U"]), W=dev(inp["W"]),
                     seed=2, cycle=0, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & sdm.DEV_CAPACITY
    last = w.R - 1
    assert host(out["accept"])[last] == 0 and host(out["n_out"])[last] == 1 and host(out["out_tok"])[last, 0] == 0
    for i in range(w.R - 1):
        first = verify_first_decision(ref, i, host(out["accept"])[i], host(out["ceiling"])[i],
                                      host(out["out_tok"])[i])
        assert first is None, f"request {i} differs at decision {first}"


# ---------------------------------------------------------------------------
# PCTree
# ---------------------------------------------------------------------------
TREE_CASES = [dict(R=4, B=4, V=1000, r=64, k=4, P=8, N=16),
              dict(R=3, B=3, V=64, r=64, k=2, P=4, N=6),
              dict(R=20, B=5, V=2048, r=128, k=4, P=8, N=32),     # 160 GEMM rows: two M tiles
              dict(R=2, B=6, V=520, r=64, k=1, P=2, N=6)]         # k = 1: the chain


def check_tree(out, ref, w, what):
    """GPU tree against the oracle: identical trees (a differing one only at a
    tie-zone decision, and none is expected), masks bit for bit, scores within
    1e-5 relative."""
    events = 0
    for i in range(w.R):
        first = tree_first_decision(ref, i, host(out["tok"])[i], host(out["parent"])[i], host(out["depth"])[i],
                                    int(host(out["n_nodes"])[i]), w.B)
        if first is not None:
            assert first[1] < TIE, f"{what}: request {i} tree differs at {first[0]}, margin {first[1]}"
            events += 1
            continue
        assert host(out["n_nodes"])[i] == ref["n_nodes"][i]
        np.testing.assert_array_equal(host(out["mask"])[i].view(np.uint32), ref["mask"][i])
        assert close(host(out["score"])[i], ref["score"][i]).all(), what
    assert events == 0, f"{what}: {events} tie-zone events"


@pytest.mark.parametrize("case", TREE_CASES, ids=lambda c: f"R{c['R']}B{c['B']}k{c['k']}P{c['P']}N{c['N']}")
def test_draft_tree_bound_pruned(case):
    """The level by bound pruning (prepared tables): the scan's lists, the
    GEMM's log-sum-exp partials and the per-request exact top-k give the
    oracle's tree, and the same tree as the record path."""
    w = small(R=case["R"], B=case["B"], V=case["V"], r=case["r"], l_dtype=BF16, sigma=(0.5,), l_std=2.0)
    inp = synthetic.generate(w, seed=case["V"])
    args = (np_of(inp["L"]), np_of(inp["U"]), np_of(inp["W"]), np_of(inp["anchor"]))
    ref = oracle.draft_tree(*args, k=case["k"], P=case["P"], N=case["N"])
    U, W = dev(inp["U"]), dev(inp["W"])
    prep = sdm.markov_prepare(U, W)
    out = sdm.draft_tree(dev(inp["L"]), U, W, dev(inp["anchor"]), case["k"], case["P"], case["N"], prepared=prep)
    rec = sdm.draft_tree(dev(inp["L"]), U, W, dev(inp["anchor"]), case["k"], case["P"], case["N"])
    torch.cuda.synchronize()
    assert int(out["dev_status"].item()) == 0
    check_tree(out, ref, w, "pruned")
    for k in ("tok", "parent", "depth", "n_nodes", "mask"):
        assert torch.equal(out[k], rec[k]), k
    assert close(host(out["score"]), host(rec["score"])).all()


@pytest.mark.parametrize("kind", ["constant_rows", "few_large", "fp32_L"])
def test_draft_tree_bound_pruned_adversarial(kind):
    """Rows whose lists overflow (every logit equal: the chunk lists cannot
    hold them) take the exhaustive top-k; rows with only a few large logits
    test the k-th-largest ladder; fp32 L uses the 8192-id chunks.  Every
    tree equals the oracle's."""
    l_dtype = FP32 if kind == "fp32_L" else BF16
    w = small(R=5, B=3, V=20000, r=64, l_dtype=l_dtype, sigma=(0.5,), l_std=2.0)
    inp = synthetic.generate(w, seed=77)
    L = inp["L"].clone()
    if kind == "constant_rows":
        L[1] = 0.5                                   # every logit of request 1 equal (ties by id)
        L[3, 1] = -1.0                               # one level of request 3
    elif kind == "few_large":
        L[:] = -30.0
        g = torch.Generator().manual_seed(3)
        for i in range(w.R):
            for d in range(w.B):
                ids = torch.randperm(w.V, generator=g)[:3]   # fewer than k outstanding logits
                L[i, d, ids] = torch.tensor([9.0, 8.5, 8.0]).to(L.dtype)
    args = (np_of(L), np_of(inp["U"]), np_of(inp["W"]), np_of(inp["anchor"]))
    k, P, N = 4, 4, 10
    ref = oracle.draft_tree(*args, k=k, P=P, N=N)
    U, W = dev(inp["U"]), dev(inp["W"])
    prep = sdm.markov_prepare(U, W)
    out = sdm.draft_tree(dev(L), U, W, dev(inp["anchor"]), k, P, N, prepared=prep)
    torch.cuda.synchronize()
    assert int(out["dev_status"].item()) == 0
    check_tree(out, ref, w, kind)


@pytest.mark.parametrize("case", TREE_CASES, ids=lambda c: f"R{c['R']}B{c['B']}k{c['k']}P{c['P']}N{c['N']}")
def test_draft_tree(case):
    w = small(R=case["R"], B=case["B"], V=case["V"], r=case["r"], l_dtype=BF16, sigma=(0.5,), l_std=2.0)
    inp = synthetic.generate(w, seed=case["V"])
    args = (np_of(inp["L"]), np_of(inp["U"]), np_of(inp["W"]), np_of(inp["anchor"]))
    ref = oracle.draft_tree(*args, k=case["k"], P=case["P"], N=case["N"])
    out = sdm.draft_tree(dev(inp["L"]), dev(inp["U"]), dev(inp["W"]), dev(inp["anchor"]), case["k"], case["P"],
                         case["N"])
    torch.cuda.synchronize()
    assert int(out["dev_status"].item()) == 0
    events = 0
    for i in range(w.R):
        first = tree_first_decision(ref, i, host(out["tok"])[i], host(out["parent"])[i], host(out["depth"])[i],
                                    int(host(out["n_nodes"])[i]), w.B)
        if first is not None:   # only a decision inside the tie zone may differ, and none is expected
            assert first[1] < TIE, f"request {i} tree differs at {first[0]}, margin {first[1]}"
            events += 1
            continue
        assert host(out["n_nodes"])[i] == ref["n_nodes"][i]
        np.testing.assert_array_equal(host(out["mask"])[i].view(np.uint32), ref["mask"][i])
        assert close(host(out["score"])[i], ref["score"][i]).all()
    assert events == 0, f"{events} tie-zone events"
    if case["k"] == 1:
        ch = oracle.draft_chain(*args)
        np.testing.assert_array_equal(host(out["tok"])[:, 1:], ch["tokens"])


def test_verify_tree():
    case = dict(R=6, B=4, V=2048, r=64, k=3, P=4, N=12)
    w = small(R=case["R"], B=case["B"], V=case["V"], r=case["r"], l_dtype=BF16, target_dtype=BF16, sigma=(0.4,),
              l_std=2.0)
    inp = synthetic.generate(w, seed=4)
    args = (np_of(inp["L"]), np_of(inp["U"]), np_of(inp["W"]), np_of(inp["anchor"]))
    tr = oracle.draft_tree(*args, k=case["k"], P=case["P"], N=case["N"])
    tgt = synthetic.tree_target(inp, torch.as_tensor(tr["tok"]), torch.as_tensor(tr["depth"]),
                                torch.as_tensor(tr["n_nodes"]), w.target_dtype)
    ref = oracle.verify_tree(np_of(tgt), tr["tok"], tr["parent"], tr["n_nodes"], w.B)
    out = sdm.verify_tree(dev(tgt), dev(torch.from_numpy(tr["tok"])), dev(torch.from_numpy(tr["parent"])),
                          dev(torch.from_numpy(tr["n_nodes"])), w.B)
    torch.cuda.synchronize()
    for k in ("accept", "out_tok", "n_out"):
        np.testing.assert_array_equal(host(out[k]), ref[k])
    assert ref["accept"].max() >= 1


# ---------------------------------------------------------------------------
# failure detection: a bounded wait that runs out
# ---------------------------------------------------------------------------
def test_a_wait_that_runs_out_is_reported_and_the_stream_stays_usable():
    """The Markov GEMM with its loads withheld and a 50 us limit on every
    wait: every wait runs out, the kernel records SDM_DEV_TIMEOUT, drains
    what it had in flight and returns; the next ordinary calls on the same
    stream give the oracle's tokens."""
    w = small(R=40, B=4, V=4160, r=128, l_dtype=BF16, sigma=(0.5,), l_std=2.0)
    inp = synthetic.generate(w, seed=31)
    L, U, W, an = dev(inp["L"]), dev(inp["U"]), dev(inp["W"]), dev(inp["anchor"])
    st = sdm.check_timeout_path(L, U, W, an, 50_000)
    torch.cuda.synchronize()
    assert int(st.item()) == sdm.DEV_TIMEOUT
    assert sdm.lib().sdm_status_of_device(int(st.item())) == 7           # SDM_ERR_TIMEOUT
    ref = oracle.draft_chain(np_of(inp["L"]), np_of(inp["U"]), np_of(inp["W"]), np_of(inp["anchor"]))
    for _ in range(2):
        out = sdm.draft_chain(L, U, W, an)
        torch.cuda.synchronize()
        assert int(out["dev_status"].item()) == 0
        np.testing.assert_array_equal(host(out["tokens"]), ref["tokens"])
    st2 = sdm.check_timeout_path(L, U, W, an, 1_000_000)                  # a second run, a longer limit
    out = sdm.draft_chain(L, U, W, an)
    torch.cuda.synchronize()
    assert int(st2.item()) == sdm.DEV_TIMEOUT and int(out["dev_status"].item()) == 0
    np.testing.assert_array_equal(host(out["tokens"]), ref["tokens"])


# ---------------------------------------------------------------------------
# the draft that fills the ragged layout
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("case", [dict(R=64, B=7, V=151936, r=256), dict(R=37, B=5, V=4104, r=64)],
                         ids=["headline_shape", "ragged"])
def test_draft_chain_packed_fills_the_layout(case):
    """The layout made from the budgets alone (pack_ragged without drafts, on
    a second stream) and filled by the draft's pick equals pack_ragged with
    the drafts; the drafts equal sdm_draft_chain's."""
    w = small(l_dtype=BF16, sigma=(0.5,), l_std=2.0, **case)
    inp = {k: dev(v) for k, v in synthetic.generate(w, seed=case["R"]).items()}
    prep = sdm.markov_prepare(inp["U"], inp["W"])
    ref = sdm.draft_chain(inp["L"], inp["U"], inp["W"], inp["anchor"], prepared=prep)
    budget = dev(torch.from_numpy(np.random.default_rng(3).integers(0, w.B + 1, w.R).astype(np.int32)))
    tiers = dev(torch.tensor([64, 128, 256, 512, 1024], dtype=torch.int32))
    full = sdm.pack_ragged(inp["anchor"], ref["tokens"], budget, tiers)
    side = torch.cuda.Stream()
    ready = torch.cuda.Event()
    main = torch.cuda.current_stream()
    side.wait_stream(main)
    with torch.cuda.stream(side):
        lay = sdm.pack_ragged(inp["anchor"], None, budget, tiers, gamma=w.B)
        ready.record(side)
    out = sdm.draft_chain_packed(inp["L"], inp["U"], inp["W"], inp["anchor"], prep, lay["cu_seqlens"],
                                 lay["packed_tok"], layout_ready=ready)
    main.wait_stream(side)
    torch.cuda.synchronize()
    assert int(out["dev_status"].item()) == 0 and int(lay["dev_status"].item()) & ~sdm.DEV_TIER_UNCAPTURED == 0
    assert torch.equal(out["tokens"], ref["tokens"])
    for k in ("cu_seqlens", "packed_tok", "packed_req", "packed_pos", "tier"):
        assert torch.equal(lay[k], full[k]), k


@pytest.mark.parametrize("case", [dict(R=64, B=7, V=8200, r=128), dict(R=5, B=3, V=2056, r=64),
                                  dict(R=300, B=6, V=4104, r=64), dict(R=37, B=16, V=8200, r=256)])
@pytest.mark.parametrize("use_budget", [True, False])
def test_draft_chain_front_equals_the_three_calls(case, use_budget):
    """The greedy draft with the scheduler and the layout in its own launches
    (the scan's extra CTA) gives, bit for bit, schedule_budget, then
    pack_ragged with the drafts (budgets for compact, all B for static), and
    sdm_draft_chain's tokens."""
    w = small(l_dtype=BF16, sigma=(0.5,), l_std=2.0, conf="sigmoid", cost=(2.0, 0.004), **case)
    inp = {k: dev(v) for k, v in synthetic.generate(w, seed=case["R"] + 1).items()}
    prep = sdm.markov_prepare(inp["U"], inp["W"])
    ref = sdm.draft_chain(inp["L"], inp["U"], inp["W"], inp["anchor"], prepared=prep)
    sc = sdm.schedule_budget(inp["conf"], inp["cost"])
    full = sdm.pack_ragged(inp["anchor"], ref["tokens"], sc["budget"] if use_budget else None, inp["tiers"])
    out = sdm.draft_chain_front(inp["L"], inp["U"], inp["W"], inp["anchor"], prep, inp["conf"], inp["cost"],
                                inp["tiers"], use_budget=use_budget, capacity=full["packed_tok"].numel())
    torch.cuda.synchronize()
    assert int(out["dev_status"].item()) & ~sdm.DEV_TIER_UNCAPTURED == 0
    assert int(out["dev_status"].item()) == int(full["dev_status"].item()) | int(ref["dev_status"].item())
    assert torch.equal(out["tokens"], ref["tokens"])
    for k in ("survival", "budget", "expected", "total_tokens"):
        assert torch.equal(out["sched"][k], sc[k]), k
    for k in ("cu_seqlens", "packed_tok", "packed_req", "packed_pos", "tier"):
        assert torch.equal(out["pk"][k], full[k]), k


def test_pack_layout_alone_holds_the_anchors():
    """Without drafts the layout's window rows hold the anchor first and -1
    where the drafts go; the offsets and row maps are those of the full pack."""
    R, g = 9, 4
    rng = np.random.default_rng(5)
    anchor = rng.integers(0, 1000, R).astype(np.int32)
    draft = rng.integers(0, 1000, (R, g)).astype(np.int32)
    budget = rng.integers(0, g + 1, R).astype(np.int32)
    tiers = np.array([16, 32, 64], np.int32)
    ref = oracle.pack_ragged(anchor, draft, budget, tiers)
    out = sdm.pack_ragged(dev(torch.from_numpy(anchor)), None, dev(torch.from_numpy(budget)), dev(torch.from_numpy(tiers)),
                          gamma=g)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host(out["cu_seqlens"]), ref["cu_seqlens"])
    t = ref["tier"]
    np.testing.assert_array_equal(host(out["packed_req"])[:t], ref["packed_req"])
    np.testing.assert_array_equal(host(out["packed_pos"])[:t], ref["packed_pos"])
    tok = host(out["packed_tok"])[:t]
    pos = ref["packed_pos"]
    np.testing.assert_array_equal(tok[pos == 0], anchor)
    assert np.all(tok[pos > 0] == -1)
