"""GPU parity of the observability entries against the oracle: the soft label
1 - TV(q, p) of every verified window row (DSpark notes sec. 5.1) and the
verify-cycle statistics (SGLang "observability").

Label tolerance: 1e-5 relative.  The label is a sum of positive terms
min(q_v, p_v), so its relative error is at most the largest relative error of
one term plus the summation's: each q_v and p_v is an fp32 exponential of an
argument within about 30 of zero (relative error below 3e-6, the fp32
log-sum-exp it subtracts included), a thread sums at most a few hundred terms
in fp32 and the per-thread partials are added in fp64.  The oracle works in
fp64.  Counts of the statistics are exact; the confidence sums per bin are
fp64 atomic adds (order not fixed), compared within 1e-12.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_markov_gb300 import binding as sdm
from speculative_decoding_markov_gb300 import synthetic
from speculative_decoding_markov_gb300.workloads import BF16, FP32, WORKLOADS
from tests.helpers import np_of, small

pytestmark = pytest.mark.gpu
DEV = "cuda"
LABEL_TOL = 1e-5   # relative


def dev(t):
    if isinstance(t, np.ndarray):
        t = torch.from_numpy(t)
    return t.to(DEV).contiguous()


def host(t):
    return t.detach().cpu().numpy()


def packed_rows(tgt, win, pad=0):
    """Front-packed window rows of tgt [R, B+1, V] (w_i + 1 rows each), with
    `pad` spare rows after them, and cu_seqlens."""
    R = tgt.shape[0]
    cu = np.zeros(R + 1, np.int32)
    rows = []
    for i in range(R):
        cu[i + 1] = cu[i] + int(win[i]) + 1
        rows.append(tgt[i, : int(win[i]) + 1])
    if pad:
        rows.append(tgt[0, :1].expand(pad, -1))
    return torch.cat(rows).contiguous(), cu


def check_labels(gpu, ref):
    outside = ref == -1.0
    np.testing.assert_array_equal(gpu[outside], -1.0)
    inside = ref[~outside]
    assert np.all(inside > 0)
    err = np.abs(gpu[~outside].astype(np.float64) - inside) / inside
    assert err.size == 0 or err.max() <= LABEL_TOL, f"max relative label error {err.max()}"
    return err


# ---------------------------------------------------------------------------
# soft label
# ---------------------------------------------------------------------------
LABEL_CASES = [
    # ragged vocab tail; q's log-sum-exp from the sampling draft; compact windows; spare rows
    (dict(R=4, B=5, V=1000, r=64, l_dtype=BF16, target_dtype=BF16), 0.8, "sample", "compact"),
    # greedy draft: q's log-sum-exp computed by the extra pass; full windows
    (dict(R=6, B=7, V=2056, r=128, l_dtype=FP32, target_dtype=FP32), 1.0, "greedy", "static"),
    # up to 320 listed rows: three M tiles, the last one ragged
    (dict(R=40, B=8, V=4104, r=64, l_dtype=BF16, target_dtype=FP32), 1.3, "greedy", "compact"),
    # smallest shapes
    (dict(R=1, B=1, V=8, r=64, l_dtype=FP32, target_dtype=FP32), 1.0, "sample", "static"),
    # every window empty: every label -1
    (dict(R=3, B=4, V=520, r=256, l_dtype=BF16, target_dtype=BF16), 1.0, "greedy", "empty"),
]


@pytest.mark.parametrize("case,T,decode,windows", LABEL_CASES,
                         ids=lambda c: c if isinstance(c, str) else (f"{c:g}" if isinstance(c, float) else
                                                                     f"R{c['R']}B{c['B']}V{c['V']}r{c['r']}"))
def test_tv_label(case, T, decode, windows):
    w = small(sigma=(0.4, 1.5), class_mix="alternate", temperature=T, **case)
    inp = synthetic.generate(w, seed=case["R"] * 7 + case["V"])
    rng = np.random.default_rng(case["V"])
    lse = None
    if decode == "sample":
        dr = sdm.draft_chain(dev(inp["L"]), dev(inp["U"]), dev(inp["W"]), dev(inp["anchor"]), decode=sdm.SAMPLE,
                             temperature=T, seed=3, cycle=1)
        torch.cuda.synchronize()
        tokens = host(dr["tokens"])
        lse = dr["lse"]
    else:
        tokens = rng.integers(0, w.V, size=(w.R, w.B)).astype(np.int32)
    win = {"static": np.full(w.R, w.B), "compact": rng.integers(0, w.B + 1, w.R),
           "empty": np.zeros(w.R, np.int64)}[windows]
    tgt = synthetic.chain_target(inp, torch.as_tensor(tokens), w.target_dtype)
    packed, cu = packed_rows(tgt, win, pad=5 if windows == "compact" else 0)
    ref = oracle.tv_label(np_of(packed[: cu[-1]]), cu, np_of(inp["anchor"]), tokens, np_of(inp["L"]),
                          np_of(inp["U"]), np_of(inp["W"]), temperature=T)
    assert ref["flags"] == 0
    st = sdm.new_status(DEV)
    out = sdm.tv_label(dev(packed), dev(cu), dev(inp["anchor"]), dev(tokens), dev(inp["L"]), dev(inp["U"]),
                       dev(inp["W"]), lse_q=lse, temperature=T, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    check_labels(host(out), ref["label"])


def test_tv_label_given_and_computed_lse_agree():
    """The sampling draft's log-sum-exp and the label's own pass give the
    same labels (both fp32 paths over the same logits)."""
    w = small(R=24, B=6, V=3000, r=128, l_dtype=BF16, target_dtype=BF16, sigma=(0.8,), temperature=0.9)
    inp = synthetic.generate(w, seed=5)
    dr = sdm.draft_chain(dev(inp["L"]), dev(inp["U"]), dev(inp["W"]), dev(inp["anchor"]), decode=sdm.SAMPLE,
                         temperature=0.9, seed=1, cycle=0)
    tgt = synthetic.chain_target({k: dev(v) for k, v in inp.items()}, dr["tokens"], w.target_dtype)
    packed, cu = packed_rows(tgt, np.full(w.R, w.B))
    args = (packed, dev(cu), dev(inp["anchor"]), dr["tokens"], dev(inp["L"]), dev(inp["U"]), dev(inp["W"]))
    a = sdm.tv_label(*args, lse_q=dr["lse"], temperature=0.9)
    b = sdm.tv_label(*args, lse_q=None, temperature=0.9)
    torch.cuda.synchronize()
    assert torch.max(torch.abs(a - b) / b).item() < 2 * LABEL_TOL
    assert torch.all((a > 0) & (a <= 1 + 1e-5))


def test_tv_label_is_deterministic():
    w = small(R=40, B=8, V=4104, r=64, l_dtype=BF16, target_dtype=FP32, sigma=(1.0,))
    inp = {k: dev(v) for k, v in synthetic.generate(w, seed=2).items()}
    toks = torch.randint(0, w.V, (w.R, w.B), dtype=torch.int32, device=DEV)
    tgt = synthetic.chain_target(inp, toks, w.target_dtype)
    packed, cu = packed_rows(tgt, np.full(w.R, w.B))
    args = (packed, dev(cu), inp["anchor"], toks, inp["L"], inp["U"], inp["W"])
    a = sdm.tv_label(*args)
    b = sdm.tv_label(*args)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_tv_label_flags_bad_rows_without_faulting():
    """A previous token outside [0, V) is flagged on the device; its row keeps
    -1 and the others are still labelled."""
    w = small(R=4, B=3, V=512, r=64, l_dtype=FP32, target_dtype=FP32, sigma=(0.5,))
    inp = synthetic.generate(w, seed=3)
    toks = np.random.default_rng(0).integers(0, w.V, size=(w.R, w.B)).astype(np.int32)
    tgt = synthetic.chain_target(inp, torch.as_tensor(toks), w.target_dtype)
    packed, cu = packed_rows(tgt, np.full(w.R, w.B))
    bad = toks.copy()
    bad[1, 0] = w.V + 3                          # previous token of row 1 of request 1
    st = sdm.new_status(DEV)
    out = host(sdm.tv_label(dev(packed), dev(cu), dev(inp["anchor"]), dev(bad), dev(inp["L"]), dev(inp["U"]),
                            dev(inp["W"]), dev_status=st))
    torch.cuda.synchronize()
    assert int(st.item()) & sdm.DEV_BAD_TOKEN
    ref = oracle.tv_label(np_of(packed), cu, np_of(inp["anchor"]), toks, np_of(inp["L"]), np_of(inp["U"]),
                          np_of(inp["W"]))["label"]
    assert out[1, 1] == -1.0
    keep = np.ones_like(out, bool)
    keep[1, 1] = False
    assert (np.abs(out[keep] - ref[keep]) / ref[keep]).max() <= LABEL_TOL


def _full_label_case(name, idx, given_lse):
    w = WORKLOADS[name]
    inp = synthetic.generate(w, seed=0, device=DEV)
    sample = w.decode == "sample"
    dr = sdm.draft_chain(inp["L"], inp["U"], inp["W"], inp["anchor"], decode=sdm.SAMPLE if sample else sdm.GREEDY,
                         temperature=w.temperature, seed=0, cycle=0)
    tgt = synthetic.chain_target(inp, dr["tokens"], w.target_dtype)
    sc = sdm.schedule_budget(inp["conf"], inp["cost"])
    pk = sdm.pack_ragged(inp["anchor"], dr["tokens"], sc["budget"], inp["tiers"])
    packed = synthetic.gather_packed(tgt, pk["packed_req"], pk["packed_pos"])
    st = sdm.new_status(DEV)
    lab = sdm.tv_label(packed, pk["cu_seqlens"], inp["anchor"], dr["tokens"], inp["L"], inp["U"], inp["W"],
                       lse_q=dr["lse"] if (sample and given_lse) else None, temperature=w.temperature, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    cu = host(pk["cu_seqlens"])
    lab = host(lab)
    toks = host(dr["tokens"])
    pk_np = np_of(packed[: cu[-1]].cpu())
    L = np_of(inp["L"].index_select(0, torch.as_tensor(idx, device=DEV)).cpu())
    an = host(inp["anchor"])[idx]
    rows = np.concatenate([pk_np[cu[i]: cu[i + 1]] for i in idx])
    sub_cu = np.concatenate([[0], np.cumsum([cu[i + 1] - cu[i] for i in idx])]).astype(np.int32)
    ref = oracle.tv_label(rows, sub_cu, an, toks[idx], L, np_of(inp["U"].cpu()), np_of(inp["W"].cpu()),
                          temperature=w.temperature)["label"]
    err = check_labels(lab[idx], ref)
    # rows past every sampled window are -1 on the device too, for all requests
    win = cu[1:] - cu[:-1] - 1
    for i in range(w.R):
        assert np.all(lab[i, win[i]:] == -1.0) and np.all(lab[i, : win[i]] >= 0.0)
    return err


def test_tv_label_rejection_sampling_full_size():
    """256 requests x 16 positions at V = 151,936, r = 256, compact windows,
    q's log-sum-exp from the sampling draft; 3 requests checked row by row."""
    _full_label_case("rejection_sampling", [0, 101, 255], given_lse=True)


def test_tv_label_headline_full_size_computed_lse():
    """64 requests x 7 positions at V = 151,936 (greedy draft): the label's own
    log-sum-exp pass; 4 requests checked row by row."""
    _full_label_case("qwen3_8b_chain", [0, 17, 40, 63], given_lse=False)


# ---------------------------------------------------------------------------
# verify-cycle statistics
# ---------------------------------------------------------------------------
def _stats_inputs(R, g, nc, nb, seed):
    rng = np.random.default_rng(seed)
    conf = rng.random((R, g)).astype(np.float32)
    flat = conf.reshape(-1)
    # edge values: exact bin edges k / nb (fp32), 0, 1, above 1, below 0, NaN
    edges = (np.arange(nb + 1, dtype=np.float32) / np.float32(nb)).astype(np.float32)
    k = min(flat.size, 3 * (nb + 1))
    pos = rng.choice(flat.size, size=k, replace=False)
    flat[pos] = np.resize(edges, k)
    if flat.size > 8:
        flat[rng.choice(flat.size, size=4, replace=False)] = [1.5, -0.25, np.nan, 1.0]
    win = rng.integers(0, g + 1, R)
    cu = np.concatenate([[0], np.cumsum(win + 1)]).astype(np.int32)
    ceiling = np.array([rng.integers(0, x + 1) for x in win], np.int32)
    cls = rng.integers(0, nc, R).astype(np.int32)
    return conf, cu, ceiling, cls


def check_stats(out, ref):
    for k in ("hist", "reached", "hits", "bin_n", "bin_hit"):
        np.testing.assert_array_equal(host(out[k]), ref[k], err_msg=k)
    np.testing.assert_allclose(host(out["bin_conf"]), ref["bin_conf"], rtol=1e-12, atol=1e-12)
    assert abs(float(host(out["ece"])[0]) - ref["ece"]) <= 1e-12


@pytest.mark.parametrize("R,g,nc,nb,seed", [(1, 1, 1, 1, 0), (7, 5, 3, 10, 1), (256, 16, 3, 15, 2),
                                            (2000, 8, 5, 64, 3), (64, 7, 1, 10, 4), (5000, 3, 2, 7, 5)])
def test_observe(R, g, nc, nb, seed):
    conf, cu, ceiling, cls = _stats_inputs(R, g, nc, nb, seed)
    ref = oracle.observe(conf, cu, ceiling, cls, nc, nb)
    out = sdm.observe(dev(conf), dev(cu), dev(ceiling), dev(cls), nc, nb)
    torch.cuda.synchronize()
    assert int(out["dev_status"].item()) == 0
    check_stats(out, ref)


def test_observe_on_a_verify_cycle_and_bad_class():
    """Ceilings from the cap-accept verify of a mixed-class workload; a class
    id out of range is flagged and its request left out."""
    w = small(R=60, B=6, V=2048, r=64, l_dtype=BF16, target_dtype=BF16, sigma=(0.2, 0.8, 2.0),
              class_mix="alternate")
    inp = {k: dev(v) for k, v in synthetic.generate(w, seed=9).items()}
    dr = sdm.draft_chain(inp["L"], inp["U"], inp["W"], inp["anchor"])
    sc = sdm.schedule_budget(inp["conf"], inp["cost"])
    pk = sdm.pack_ragged(inp["anchor"], dr["tokens"], None, inp["tiers"])
    tgt = synthetic.chain_target(inp, dr["tokens"], w.target_dtype)
    packed = synthetic.gather_packed(tgt, pk["packed_req"], pk["packed_pos"])
    vr = sdm.verify(sdm.CAP_ACCEPT, sdm.GREEDY, packed, pk["cu_seqlens"], inp["anchor"], dr["tokens"],
                    budget=sc["budget"])
    cls = (torch.arange(w.R, device=DEV) % 3).to(torch.int32)
    out = sdm.observe(inp["conf"], pk["cu_seqlens"], vr["ceiling"], cls, 3, 10)
    torch.cuda.synchronize()
    ref = oracle.observe(host(inp["conf"]), host(pk["cu_seqlens"]), host(vr["ceiling"]), host(cls), 3, 10)
    check_stats(out, ref)
    assert ref["hist"].sum() == w.R and ref["reached"][:, 0].sum() == w.R
    bad = cls.clone()
    bad[5] = 3
    out = sdm.observe(inp["conf"], pk["cu_seqlens"], vr["ceiling"], bad, 3, 10)
    torch.cuda.synchronize()
    assert int(out["dev_status"].item()) & sdm.DEV_BAD_CLASS
    keep = np.arange(w.R) != 5
    cu = host(pk["cu_seqlens"])
    win = (cu[1:] - cu[:-1])[keep]
    cu_k = np.concatenate([[0], np.cumsum(win)]).astype(np.int32)
    ref = oracle.observe(host(inp["conf"])[keep], cu_k, host(vr["ceiling"])[keep], host(cls)[keep], 3, 10)
    check_stats(out, ref)
