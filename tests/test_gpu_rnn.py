"""GPU parity of the chain draft with the RNN head against the oracle.

The kernel keeps the memo in fp32 (the oracle in fp64) and rounds it to bf16
where it enters the vocabulary projection, so the comparison has three
parts, each at 1e-5:
  1. the GPU's fp32 memo against the oracle's memo along the GPU's tokens;
  2. every decision, lse and logq against the oracle's projection of the
     GPU's own memo (z_d = L_d + bf16(m_d) W): tokens exact unless that
     decision's margin is below 1e-5 (a tie-zone event; none is expected),
     lse and logq within 1e-5 relative (|x| >= 1) or absolute;
  3. the tokens against the oracle's own draft: they may part only at a
     position where the two memos' bf16 roundings differ at or before it.
"""
from __future__ import annotations

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
TIE = 1e-5
FTOL = 1e-5
MEMO_TOL = 1e-5


def dev(t):
    return t.to(DEV).contiguous()


def host(t):
    return t.detach().cpu().numpy()


def bf16_bits(x):
    """Round to bf16 through binary32, nearest-even (as the kernel's memo rows)."""
    b = np.asarray(x, np.float64).astype(np.float32).view(np.uint32).astype(np.uint64)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)


def close(gpu, ref, tol=FTOL):
    gpu, ref = np.asarray(gpu, np.float64), np.asarray(ref, np.float64)
    return np.abs(gpu - ref) <= tol * np.maximum(1.0, np.abs(ref))


def check(gpu, ref, L, W, anchor, A, U, X, decode, T, seed, cycle):
    gtok = host(gpu["tokens"])
    gmemo = host(gpu["memo"]).astype(np.float32)
    memo = oracle.rnn_memo(A, U, X, anchor, gtok)
    assert np.abs(gmemo - memo).max() <= MEMO_TOL
    pj = oracle.rnn_project(L, W, gmemo, decode=decode, temperature=T, seed=seed, cycle=cycle)
    events = 0
    for i in range(gtok.shape[0]):
        mism = np.nonzero(gtok[i] != pj["tokens"][i])[0]
        for d in mism:   # each position's decision stands alone given the GPU's memo
            assert pj["margin"][i, d] < TIE, f"request {i} position {d} differs at margin {pj['margin'][i, d]}"
            events += 1
    assert events == 0, f"{events} tie-zone events"
    if decode == oracle.SAMPLE:
        assert close(host(gpu["lse"]), pj["lse"]).all()
        assert close(host(gpu["logq"]), pj["logq"]).all()
    flips = np.any(bf16_bits(gmemo) != bf16_bits(memo), axis=-1)   # [R, B]: a memo element rounds apart
    for i in range(gtok.shape[0]):
        mism = np.nonzero(gtok[i] != ref["tokens"][i])[0]
        if mism.size:
            d = int(mism[0])
            assert flips[i, : d + 1].any(), f"request {i} parts from the oracle's draft at {d} with equal memos"


CASES = [
    (dict(R=4, B=7, V=1024, r=64, l_dtype=FP32), "greedy", 1.0),
    (dict(R=64, B=4, V=1000, r=256, l_dtype=BF16), "greedy", 1.0),     # ragged vocab tail
    (dict(R=130, B=3, V=4160, r=128, l_dtype=BF16), "sample", 0.8),    # two M tiles, ragged rows
    (dict(R=40, B=5, V=2056, r=64, l_dtype=FP32), "sample", 1.3),
    (dict(R=1, B=2, V=8, r=64, l_dtype=FP32), "sample", 1.0),          # smallest shapes
]


@pytest.mark.parametrize("case,decode,T", CASES,
                         ids=lambda c: c if isinstance(c, str) else (f"T{c:g}" if isinstance(c, float) else
                                                                     f"R{c['R']}B{c['B']}V{c['V']}r{c['r']}"))
def test_draft_chain_rnn(case, decode, T):
    w = small(sigma=(0.5,), l_std=1.0, **case)
    inp = synthetic.generate(w, seed=case["R"] + case["V"])
    rnn = synthetic.rnn_inputs(w, seed=case["V"])
    sample = decode == "sample"
    L, U, W, an = np_of(inp["L"]), np_of(inp["U"]), np_of(inp["W"]), np_of(inp["anchor"])
    A, X = np_of(rnn["A_rnn"]), np_of(rnn["X_rnn"])
    od = oracle.SAMPLE if sample else oracle.GREEDY
    ref = oracle.draft_chain_rnn(L, U, W, A, X, an, decode=od, temperature=T, seed=6, cycle=2)
    out = sdm.draft_chain_rnn(dev(inp["L"]), dev(inp["U"]), dev(inp["W"]), dev(rnn["A_rnn"]), dev(rnn["X_rnn"]),
                              dev(inp["anchor"]), decode=sdm.SAMPLE if sample else sdm.GREEDY, temperature=T,
                              seed=6, cycle=2, memo=True)
    torch.cuda.synchronize()
    assert int(out["dev_status"].item()) == 0
    check(out, ref, L, W, an, A, U, X, od, T, 6, 2)


def test_rnn_without_memory_matches_the_markov_draft_on_the_gpu():
    """A = 0, x = 0: the GPU's RNN draft equals its Markov draft on the table
    bf16(tanh U) (both through the same tensor-core projection)."""
    w = small(R=48, B=5, V=2048, r=64, l_dtype=BF16, sigma=(0.5,))
    inp = {k: dev(v) for k, v in synthetic.generate(w, seed=2).items()}
    A = torch.zeros((w.r, w.r), dtype=torch.bfloat16, device=DEV)
    X = torch.zeros((w.R, w.B, w.r), dtype=torch.bfloat16, device=DEV)
    U4 = (inp["U"].float() * 4).to(torch.bfloat16)
    Ut = torch.tanh(U4.float()).to(torch.bfloat16)           # fp32 tanh, as the memo kernel forms it
    for dec in (sdm.GREEDY, sdm.SAMPLE):
        a = sdm.draft_chain_rnn(inp["L"], U4, inp["W"], A, X, inp["anchor"], decode=dec, temperature=0.9, seed=3)
        b = sdm.draft_chain(inp["L"], Ut, inp["W"], inp["anchor"], decode=dec, temperature=0.9, seed=3)
        torch.cuda.synchronize()
        assert torch.equal(a["tokens"], b["tokens"])
        if dec == sdm.SAMPLE:
            assert torch.max(torch.abs(a["lse"] - b["lse"])).item() < 1e-5


def test_draft_chain_rnn_headline_full_size():
    """64 requests x 7 positions at V = 151,936, r = 256 (bf16 L), greedy;
    3 requests checked against the oracle."""
    w = WORKLOADS["qwen3_8b_chain"]
    inp = synthetic.generate(w, seed=0, device=DEV)
    rnn = synthetic.rnn_inputs(w, seed=0, device=DEV)
    out = sdm.draft_chain_rnn(inp["L"], inp["U"], inp["W"], rnn["A_rnn"], rnn["X_rnn"], inp["anchor"], memo=True)
    torch.cuda.synchronize()
    assert int(out["dev_status"].item()) == 0
    idx = [0, 31, 63]
    t = torch.as_tensor(idx, device=DEV)
    L = np_of(inp["L"].index_select(0, t).cpu())
    U, W, A = np_of(inp["U"].cpu()), np_of(inp["W"].cpu()), np_of(rnn["A_rnn"].cpu())
    X = np_of(rnn["X_rnn"].index_select(0, t).cpu())
    an = host(inp["anchor"])[idx]
    ref = oracle.draft_chain_rnn(L, U, W, A, X, an)
    sub = dict(tokens=out["tokens"][t], memo=out["memo"][t])
    check(sub, ref, L, W, an, A, U, X, oracle.GREEDY, 1.0, 0, 0)
