"""Greedy verification for callers that cannot allocate: sdm_verify_greedy_static.

Some callers cannot hand the library scratch memory (a server that reserved
all device memory at start-up, a framework whose allocator must account for
every byte, a loop that cannot afford the device synchronisation of
cudaMalloc).  This entry point keeps its scratch in a fixed array in the
library's own device memory.  The test calls it through the C-ABI twice in a
row and checks every output against sdm_verify (caller workspace) on the same
inputs; integer outputs must match exactly.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

from speculative_decoding_markov_gb300 import binding as sdm
from speculative_decoding_markov_gb300 import synthetic
from speculative_decoding_markov_gb300.workloads import BF16, FP32, Workload

pytestmark = pytest.mark.gpu


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _static_verify(mode, packed, cu, draft, budget, R, gamma, V, rows=None):
    out = dict(accept=torch.full((R,), -9, dtype=torch.int32, device="cuda"),
               ceiling=torch.full((R,), -9, dtype=torch.int32, device="cuda"),
               out_tok=torch.full((R, gamma + 1), -9, dtype=torch.int32, device="cuda"),
               n_out=torch.full((R,), -9, dtype=torch.int32, device="cuda"),
               dev_status=torch.zeros(1, dtype=torch.int32, device="cuda"))
    rows = packed.shape[0] if rows is None else rows
    st = sdm.lib().sdm_verify_greedy_static(
        mode, _ptr(packed), 0 if packed.dtype == torch.bfloat16 else 1, rows, _ptr(cu), _ptr(draft), _ptr(budget),
        R, gamma, V, _ptr(out["accept"]), _ptr(out["ceiling"]), _ptr(out["out_tok"]), _ptr(out["n_out"]),
        _ptr(out["dev_status"]), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st, out


@pytest.mark.parametrize("tdt", [BF16, FP32])
def test_static_scratch_verify_matches_workspace_verify(tdt):
    w = Workload(name="no_alloc", R=24, B=7, V=151936, r=64, l_dtype=BF16, l_std=2.0, sigma=(0.3, 1.0),
                 target_dtype=tdt)
    inp = {k: v.cuda() for k, v in synthetic.generate(w, seed=5).items()}
    dr = sdm.draft_chain(inp["L"], inp["U"], inp["W"], inp["anchor"])
    sc = sdm.schedule_budget(inp["conf"], inp["cost"])
    target = synthetic.chain_target(inp, dr["tokens"], tdt)
    for mode in (sdm.COMPACT, sdm.CAP_ACCEPT, sdm.STATIC):
        pk = sdm.pack_ragged(inp["anchor"], dr["tokens"], sc["budget"] if mode == sdm.COMPACT else None,
                             inp["tiers"])
        packed = synthetic.gather_packed(target, pk["packed_req"], pk["packed_pos"])
        ref = sdm.verify(mode, sdm.GREEDY, packed, pk["cu_seqlens"], inp["anchor"], dr["tokens"],
                         budget=sc["budget"])
        torch.cuda.synchronize()
        for call in range(2):   # the shared array is reused by consecutive calls
            st, out = _static_verify(mode, packed, pk["cu_seqlens"], dr["tokens"], sc["budget"], w.R, w.B, w.V)
            torch.cuda.synchronize()
            assert st == 0, sdm.lib().sdm_status_str(st)
            assert int(out["dev_status"].item()) == 0
            for k in ("accept", "out_tok", "n_out"):
                assert torch.equal(out[k], ref[k]), (mode, call, k)
            if mode == sdm.CAP_ACCEPT:
                assert torch.equal(out["ceiling"], ref["ceiling"])
        assert ref["accept"].max() > 0


def test_static_scratch_rejects_what_does_not_fit():
    V, R, gamma = 151936, 4, 7
    packed = torch.zeros((8, V), dtype=torch.bfloat16, device="cuda")
    cu = torch.arange(0, 2 * (R + 1), 2, dtype=torch.int32, device="cuda")
    draft = torch.zeros((R, gamma), dtype=torch.int32, device="cuda")
    # 20000 rows x 10 chunks of partial keys exceed the 1 MiB array
    st, out = _static_verify(sdm.COMPACT, packed, cu, draft, None, R, gamma, V, rows=20000)
    torch.cuda.synchronize()
    assert st == 5                                       # SDM_ERR_WORKSPACE, nothing launched
    assert torch.all(out["accept"] == -9)


def test_static_scratch_never_reads_partials_of_an_earlier_call():
    """The array keeps the last call's partial keys.  A later call whose
    cu_seqlens ends (cu[R]) before one of its requests' windows must not read
    them: such a request is flagged and commits one token (0), the requests
    inside the total match the workspace entry point."""
    w = Workload(name="no_alloc", R=6, B=4, V=2048, r=64, l_dtype=BF16, l_std=2.0, sigma=(0.5,),
                 target_dtype=BF16)
    inp = {k: v.cuda() for k, v in synthetic.generate(w, seed=9).items()}
    dr = sdm.draft_chain(inp["L"], inp["U"], inp["W"], inp["anchor"])
    pk = sdm.pack_ragged(inp["anchor"], dr["tokens"], None, inp["tiers"])
    target = synthetic.chain_target(inp, dr["tokens"], BF16)
    packed = synthetic.gather_packed(target, pk["packed_req"], pk["packed_pos"])
    ref = sdm.verify(sdm.STATIC, sdm.GREEDY, packed, pk["cu_seqlens"], inp["anchor"], dr["tokens"])
    st, first = _static_verify(sdm.STATIC, packed, pk["cu_seqlens"], dr["tokens"], None, w.R, w.B, w.V)
    torch.cuda.synchronize()
    assert st == 0 and int(first["dev_status"].item()) == 0
    bad = pk["cu_seqlens"].clone()
    bad[-1] = bad[2]                          # requests 2 .. R-1 end past the packed total
    st, out = _static_verify(sdm.STATIC, packed, bad, dr["tokens"], None, w.R, w.B, w.V)
    torch.cuda.synchronize()
    assert st == 0
    assert int(out["dev_status"].item()) & sdm.DEV_BAD_WINDOW
    for k in ("accept", "out_tok", "n_out"):
        assert torch.equal(out[k][:2], ref[k][:2]), k
    assert torch.all(out["accept"][2:] == 0) and torch.all(out["n_out"][2:] == 1)
    assert torch.all(out["out_tok"][2:, 0] == 0) and torch.all(out["out_tok"][2:, 1:] == -1)
