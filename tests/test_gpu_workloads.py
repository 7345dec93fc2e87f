"""The five workloads at full size on the GPU, in the launch configuration the
benchmark times, checked against the oracle on sampled requests (requests
are independent in drafting and verification; the scheduler and the pack
couple them and are checked over all requests)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_markov_gb300 import binding as sdm
from speculative_decoding_markov_gb300 import synthetic
from speculative_decoding_markov_gb300.workloads import WORKLOADS
from tests.helpers import np_of, oracle_map, tree_first_decision, verify_first_decision

pytestmark = pytest.mark.gpu
TIE = 1e-5


def host(t):
    return t.detach().cpu().numpy()


def close(gpu, ref, tol=1e-5):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    return np.abs(gpu - ref) <= tol * np.maximum(1.0, np.abs(ref))


def sub_inputs(inp, idx):
    t = torch.as_tensor(idx, dtype=torch.long, device=inp["L"].device)
    d = {k: inp[k].index_select(0, t).cpu() for k in ("L", "L_bonus", "eta", "anchor")}
    d["U"], d["W"] = inp["U"].cpu(), inp["W"].cpu()
    return d


def run_chain_workload(name, idx, modes=None):
    w = WORKLOADS[name]
    inp = synthetic.generate(w, seed=0, device="cuda")
    sample = w.decode == "sample"
    prepared = None if sample else sdm.markov_prepare(inp["U"], inp["W"])
    dr = sdm.draft_chain(inp["L"], inp["U"], inp["W"], inp["anchor"], decode=sdm.SAMPLE if sample else sdm.GREEDY,
                         temperature=w.temperature, seed=0, cycle=0, prepared=prepared)
    if not sample:   # the bound-pruned chain equals the dense tensor-core chain bit for bit
        dense = sdm.draft_chain(inp["L"], inp["U"], inp["W"], inp["anchor"])
        torch.cuda.synchronize()
        assert torch.equal(dense["tokens"], dr["tokens"])
    sc = sdm.schedule_budget(inp["conf"], inp["cost"])
    target = synthetic.chain_target(inp, dr["tokens"], w.target_dtype)
    torch.cuda.synchronize()
    assert int(dr["dev_status"].item()) == 0

    # oracle on the sampled requests
    sub = sub_inputs(inp, idx)
    ids = np.asarray(idx, np.int32)
    U, W = np_of(sub["U"]), np_of(sub["W"])
    Ls, ans = np_of(sub["L"]), np_of(sub["anchor"])

    def one(j):   # one request per oracle call, the calls spread over the host cores
        return oracle.draft_chain(Ls[j:j + 1], U, W, ans[j:j + 1], decode=oracle.SAMPLE if sample else oracle.GREEDY,
                                  temperature=w.temperature, seed=0, cycle=0, req_ids=ids[j:j + 1])

    parts = oracle_map(one, range(len(idx)))
    odr = {k: np.concatenate([q[k] for q in parts]) for k in ("tokens", "logq", "lse", "margin")}
    gtok = host(dr["tokens"])[idx]
    for i in range(len(idx)):
        mism = np.nonzero(gtok[i] != odr["tokens"][i])[0]
        assert mism.size == 0 or odr["margin"][i, mism[0]] < TIE, f"request {idx[i]} draft differs"
        assert mism.size == 0, f"tie-zone event at request {idx[i]}"
    if sample:
        assert close(host(dr["lse"])[idx], odr["lse"]).all()
        assert close(host(dr["logq"])[idx], odr["logq"]).all()

    # scheduler over every request
    osc = oracle.schedule_budget(np_of(inp["conf"]), np_of(inp["cost"]))
    np.testing.assert_array_equal(host(sc["budget"]), osc["budget"])
    np.testing.assert_array_equal(host(sc["survival"]).view(np.uint32), osc["survival"].view(np.uint32))
    assert int(host(sc["total_tokens"])[0]) == osc["total_tokens"]

    results = {}
    for mode in (modes or w.modes):
        budget_all = sc["budget"]
        pk = sdm.pack_ragged(inp["anchor"], dr["tokens"], budget_all if mode == "compact" else None, inp["tiers"])
        packed = synthetic.gather_packed(target, pk["packed_req"], pk["packed_pos"])
        gm = {"static": sdm.STATIC, "compact": sdm.COMPACT, "cap_accept": sdm.CAP_ACCEPT}[mode]
        kw = {}
        if sample:
            kw = dict(logq=dr["logq"], lse_q=dr["lse"], L=inp["L"], U=inp["U"], W=inp["W"])
        vr = sdm.verify(gm, sdm.SAMPLE if sample else sdm.GREEDY, packed, pk["cu_seqlens"], inp["anchor"],
                        dr["tokens"], budget=budget_all, temperature=w.temperature, seed=0, cycle=0, **kw)
        torch.cuda.synchronize()
        st = int(pk["dev_status"].item())
        assert st & ~sdm.DEV_TIER_UNCAPTURED == 0 and int(vr["dev_status"].item()) == 0

        # pack: offsets over all requests, rows of the sampled ones
        opk_all = oracle.pack_ragged(np_of(inp["anchor"]), np.zeros((w.R, w.B), np.int32),
                                     osc["budget"] if mode == "compact" else None, np_of(inp["tiers"]))
        np.testing.assert_array_equal(host(pk["cu_seqlens"]), opk_all["cu_seqlens"])
        assert int(host(pk["tier"])[0]) == opk_all["tier"]
        cu = host(pk["cu_seqlens"])
        bsub = osc["budget"][ids]
        opk = oracle.pack_ragged(np_of(sub["anchor"]), odr["tokens"], bsub if mode == "compact" else None,
                                 np.array([1 << 20], np.int32))
        for j, i in enumerate(idx):
            a, b = cu[i], cu[i + 1]
            oa, ob = opk["cu_seqlens"][j], opk["cu_seqlens"][j + 1]
            np.testing.assert_array_equal(host(pk["packed_tok"])[a:b], opk["packed_tok"][oa:ob])
            np.testing.assert_array_equal(host(pk["packed_pos"])[a:b], opk["packed_pos"][oa:ob])

        # verify on the sampled requests, target rows built from the oracle's drafts
        otgt = synthetic.chain_target(sub, torch.as_tensor(odr["tokens"]), w.target_dtype)
        opacked = synthetic.gather_packed(otgt, torch.as_tensor(opk["packed_req"][: opk["cu_seqlens"][-1]]),
                                          torch.as_tensor(opk["packed_pos"][: opk["cu_seqlens"][-1]]))
        om = {"static": oracle.STATIC, "compact": oracle.COMPACT, "cap_accept": oracle.CAP_ACCEPT}[mode]
        okw = {}
        if sample:
            okw = dict(logq=odr["logq"], lse_q=odr["lse"], L=np_of(sub["L"]), U=U, W=W, temperature=w.temperature,
                       seed=0, cycle=0)
        ovr = oracle.verify(om, oracle.SAMPLE if sample else oracle.GREEDY, np_of(opacked), opk["cu_seqlens"],
                            np_of(sub["anchor"]), odr["tokens"], budget=bsub, req_ids=ids, **okw)
        for j, i in enumerate(idx):
            first = verify_first_decision(ovr, j, host(vr["accept"])[i], host(vr["ceiling"])[i],
                                          host(vr["out_tok"])[i])
            assert first is None or first[1] < TIE, f"{mode}: request {i} differs at decision {first}"
            assert first is None, f"{mode}: tie-zone event at request {i} ({first})"
        results[mode] = dict(accept=host(vr["accept"]), n_out=host(vr["n_out"]), out_tok=host(vr["out_tok"]),
                             ceiling=host(vr["ceiling"]))
    return w, results, osc


def test_tiny_chain_full():
    w = WORKLOADS["tiny_chain"]
    run_chain_workload("tiny_chain", list(range(w.R)))


def test_qwen3_8b_chain():
    w, res, _ = run_chain_workload("qwen3_8b_chain", [0, 1, 17, 31, 38, 50, 62, 63])
    assert res["compact"]["n_out"].sum() > w.R          # some drafts accepted


def test_rejection_sampling():
    # both M tiles of the GEMMs (requests 0-127 and 128-255), their edges included
    w, res, _ = run_chain_workload("rejection_sampling", [0, 37, 100, 127, 128, 131, 200, 255])
    assert res["static"]["accept"].max() > 0


def test_mixed_traffic_modes():
    w, res, osc = run_chain_workload("mixed_traffic", [0, 100, 127, 128, 200, 254])
    np.testing.assert_array_equal(res["cap_accept"]["out_tok"], res["compact"]["out_tok"])
    np.testing.assert_array_equal(res["cap_accept"]["ceiling"], res["static"]["accept"])
    np.testing.assert_array_equal(res["compact"]["accept"], np.minimum(res["static"]["accept"], osc["budget"]))


def test_pctree():
    w = WORKLOADS["pctree"]
    inp = synthetic.generate(w, seed=0, device="cuda")
    prep = sdm.markov_prepare(inp["U"], inp["W"])
    tr = sdm.draft_tree(inp["L"], inp["U"], inp["W"], inp["anchor"], w.k, w.P, w.N, prepared=prep)
    rec = sdm.draft_tree(inp["L"], inp["U"], inp["W"], inp["anchor"], w.k, w.P, w.N)   # the record path
    torch.cuda.synchronize()
    for key in ("tok", "parent", "depth", "n_nodes", "mask"):   # the two level paths agree on every request
        assert torch.equal(tr[key], rec[key]), key
    assert close(host(tr["score"]), host(rec["score"])).all()
    tgt = synthetic.tree_target(inp, tr["tok"], tr["depth"], tr["n_nodes"], w.target_dtype)
    vt = sdm.verify_tree(tgt, tr["tok"], tr["parent"], tr["n_nodes"], w.B)
    torch.cuda.synchronize()
    assert int(tr["dev_status"].item()) == 0 and int(vt["dev_status"].item()) == 0
    assert np.all(host(tr["n_nodes"]) == w.N + 1)
    # frontier rows of requests 0-15 fill the level GEMM's first M tile, 16-31 its second
    idx = [5, 15, 16, 30]
    sub = sub_inputs(inp, idx)
    Ls, Us, Ws, ans = np_of(sub["L"]), np_of(sub["U"]), np_of(sub["W"]), np_of(sub["anchor"])
    parts = oracle_map(lambda j: oracle.draft_tree(Ls[j:j + 1], Us, Ws, ans[j:j + 1], w.k, w.P, w.N),
                       range(len(idx)))
    otr = {k: np.concatenate([q[k] for q in parts]) for k in ("tok", "parent", "depth", "score", "mask", "n_nodes",
                                                              "margin")}
    for j, i in enumerate(idx):
        first = tree_first_decision(otr, j, host(tr["tok"])[i], host(tr["parent"])[i], host(tr["depth"])[i],
                                    int(host(tr["n_nodes"])[i]), w.B)
        assert first is None or first[1] < TIE, f"tree of request {i} differs at {first}"
        assert first is None, f"tie-zone event in the tree of request {i} ({first})"
    for key in ("tok", "parent", "depth", "n_nodes"):
        np.testing.assert_array_equal(host(tr[key])[idx], otr[key])
    np.testing.assert_array_equal(host(tr["mask"])[idx].view(np.uint32), otr["mask"])
    assert close(host(tr["score"])[idx], otr["score"]).all()
    otgt = synthetic.tree_target(sub, torch.as_tensor(otr["tok"]), torch.as_tensor(otr["depth"]),
                                 torch.as_tensor(otr["n_nodes"]), w.target_dtype)
    ovt = oracle.verify_tree(np_of(otgt), otr["tok"], otr["parent"], otr["n_nodes"], w.B)
    for key in ("accept", "out_tok", "n_out"):
        np.testing.assert_array_equal(host(vt[key])[idx], ovt[key])
    # every tree is ancestor-closed and topologically ordered
    par = host(tr["parent"])
    assert np.all(par[:, 1:] < np.arange(1, w.N + 1)[None, :]) and np.all(par[:, 1:] >= 0)
