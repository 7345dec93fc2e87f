"""Python access to the CPU oracle (TEST INFRASTRUCTURE ONLY).

The oracle is plain single-threaded C (oracle.c) restating the method from
its pages.  Only tests, the smoke check and the benchmark's CPU-baseline leg
may import this module; the CUDA library never does.  Arrays are numpy;
bf16 data is passed as its uint16 bit pattern.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
HDR = os.path.join(HERE, "oracle.h")
LIB = os.path.join(HERE, "liboracle.so")

BF16, FP32 = 0, 1
GREEDY, SAMPLE = 0, 1
STATIC, COMPACT, CAP_ACCEPT = 0, 1, 2
STREAM_DRAFT, STREAM_ACCEPT, STREAM_RESID, STREAM_BONUS = 0, 1, 2, 3
FLAG_TIER_UNCAPTURED = 2
FLAG_TIER_OVERFLOW = 64
FLAG_INEXACT_MARKOV = 16

_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc (-O2 -ffp-contract=off, single-threaded)."""
    newest = max(os.path.getmtime(SRC), os.path.getmtime(HDR))
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < newest:
        tmp = LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11",
                               "-fPIC", "-shared", "-o", tmp, SRC, "-lm"])
        os.replace(tmp, LIB)
    return LIB


def lib():
    global _lib
    if _lib is None:
        build()
        _lib = ctypes.CDLL(LIB)
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _dt(arr) -> int:
    return BF16 if arr.dtype == np.uint16 else FP32


def philox(ctr, key):
    out = np.zeros(4, np.uint32)
    lib().orc_philox4x32_10(_p(_c(ctr, np.uint32)), _p(_c(key, np.uint32)), _p(out))
    return out


def uniform(seed, cycle, stream, req, row, v) -> float:
    f = lib().orc_uniform
    f.restype = ctypes.c_double
    return f(ctypes.c_uint64(seed), ctypes.c_uint64(cycle), ctypes.c_int(stream),
             ctypes.c_uint32(req), ctypes.c_uint32(row), ctypes.c_uint32(v))


def draft_chain(L, U, W, anchor, decode=GREEDY, temperature=1.0, seed=0, cycle=0, req_ids=None):
    """L [R,B,V] (uint16 bf16 bits or float32), U [V,r], W [r,V] uint16."""
    R, B, V = L.shape
    r = U.shape[1]
    L = np.ascontiguousarray(L)
    tokens = np.zeros((R, B), np.int32)
    logq = np.zeros((R, B), np.float64)
    lse = np.zeros((R, B), np.float64)
    margin = np.zeros((R, B), np.float64)
    ids = None if req_ids is None else _c(req_ids, np.int32)
    flags = lib().orc_draft_chain(
        _p(L), _dt(L), _p(_c(U, np.uint16)), _p(_c(W, np.uint16)), _p(_c(anchor, np.int32)), _p(ids),
        R, B, V, r, decode, ctypes.c_double(temperature), ctypes.c_uint64(seed), ctypes.c_uint64(cycle),
        _p(tokens), _p(logq), _p(lse), _p(margin))
    return dict(tokens=tokens, logq=logq, lse=lse, margin=margin, flags=flags)


def draft_tree(L, U, W, anchor, k, P, N):
    R, B, V = L.shape
    r = U.shape[1]
    L = np.ascontiguousarray(L)
    S = N + 1
    words = (S + 31) // 32
    tok = np.zeros((R, S), np.int32)
    parent = np.zeros((R, S), np.int32)
    depth = np.zeros((R, S), np.int32)
    score = np.zeros((R, S), np.float64)
    mask = np.zeros((R, S, words), np.uint32)
    n_nodes = np.zeros(R, np.int32)
    margin = np.zeros((R, B + 2), np.float64)
    flags = lib().orc_draft_tree(
        _p(L), _dt(L), _p(_c(U, np.uint16)), _p(_c(W, np.uint16)), _p(_c(anchor, np.int32)),
        R, B, V, r, k, P, N, _p(tok), _p(parent), _p(depth), _p(score), _p(mask), _p(n_nodes), _p(margin))
    return dict(tok=tok, parent=parent, depth=depth, score=score, mask=mask, n_nodes=n_nodes,
                margin=margin, flags=flags)


def schedule_budget(conf, cost):
    R, g = conf.shape
    survival = np.zeros((R, g), np.float32)
    budget = np.zeros(R, np.int32)
    expected = np.zeros(1, np.float64)
    total = np.zeros(1, np.int32)
    m_star = np.zeros(1, np.int32)
    lib().orc_schedule_budget(_p(_c(conf, np.float32)), R, g, _p(_c(cost, np.float64)), _p(survival),
                              _p(budget), _p(expected), _p(total), _p(m_star))
    return dict(survival=survival, budget=budget, expected=float(expected[0]), total_tokens=int(total[0]),
                m_star=int(m_star[0]))


def schedule_dynamic(conf, conf_stale, cost):
    R, g = conf.shape
    assert conf_stale.shape == (R, g)
    survival = np.zeros((R, g), np.float32)
    budget = np.zeros(R, np.int32)
    expected = np.zeros(1, np.float64)
    total = np.zeros(1, np.int32)
    capacity = np.zeros(1, np.int32)
    lib().orc_schedule_dynamic(_p(_c(conf, np.float32)), _p(_c(conf_stale, np.float32)), R, g,
                               _p(_c(cost, np.float64)), _p(survival), _p(budget), _p(expected), _p(total),
                               _p(capacity))
    return dict(survival=survival, budget=budget, expected=float(expected[0]), total_tokens=int(total[0]),
                capacity=int(capacity[0]))


def pack_ragged(anchor, draft, budget, tiers, strict=False):
    R, g = draft.shape
    tiers = _c(tiers, np.int32)
    cap = max(int(tiers.max()) if tiers.size else 0, R * (g + 1))
    cu = np.zeros(R + 1, np.int32)
    ptok = np.full(cap, -7, np.int32)
    preq = np.full(cap, -7, np.int32)
    ppos = np.full(cap, -7, np.int32)
    tier = np.zeros(1, np.int32)
    flags = np.zeros(1, np.int32)
    b = None if budget is None else _c(budget, np.int32)
    rc = lib().orc_pack_ragged(_p(_c(anchor, np.int32)), _p(_c(draft, np.int32)), _p(b), R, g,
                               _p(tiers), tiers.size, 1 if strict else 0, _p(cu), _p(ptok), _p(preq), _p(ppos),
                               _p(tier), _p(flags))
    if rc != 0:
        raise ValueError("pack_ragged: budget out of range")
    t = int(tier[0])
    return dict(cu_seqlens=cu, packed_tok=ptok[:t], packed_req=preq[:t], packed_pos=ppos[:t], tier=t,
                flags=int(flags[0]))


def verify(mode, decode, target, cu_seqlens, anchor, draft, budget=None, logq=None, lse_q=None,
           L=None, U=None, W=None, temperature=1.0, seed=0, cycle=0, req_ids=None):
    """target [rows, V] packed (uint16 bf16 bits or float32)."""
    R, g = draft.shape
    V = target.shape[-1]
    target = np.ascontiguousarray(target)
    accept = np.zeros(R, np.int32)
    ceiling = np.zeros(R, np.int32)
    out_tok = np.zeros((R, g + 1), np.int32)
    n_out = np.zeros(R, np.int32)
    margin = np.zeros((R, g + 1), np.float64)
    r = 0 if U is None else U.shape[1]
    Lc = None if L is None else np.ascontiguousarray(L)
    flags = lib().orc_verify(
        mode, decode, ctypes.c_double(temperature), ctypes.c_uint64(seed), ctypes.c_uint64(cycle),
        _p(None if req_ids is None else _c(req_ids, np.int32)), _p(target), _dt(target), _p(_c(cu_seqlens, np.int32)), _p(_c(anchor, np.int32)), _p(_c(draft, np.int32)),
        _p(None if budget is None else _c(budget, np.int32)),
        _p(None if logq is None else _c(logq, np.float64)), _p(None if lse_q is None else _c(lse_q, np.float64)),
        _p(Lc), 0 if Lc is None else _dt(Lc), _p(None if U is None else _c(U, np.uint16)),
        _p(None if W is None else _c(W, np.uint16)), r, R, g, V,
        _p(accept), _p(ceiling), _p(out_tok), _p(n_out), _p(margin))
    return dict(accept=accept, ceiling=ceiling, out_tok=out_tok, n_out=n_out, margin=margin, flags=flags)


def verify_tree(target, tok, parent, n_nodes, B):
    R, S, V = target.shape
    target = np.ascontiguousarray(target)
    accept = np.zeros(R, np.int32)
    out_tok = np.zeros((R, B + 1), np.int32)
    n_out = np.zeros(R, np.int32)
    lib().orc_verify_tree(_p(target), _dt(target), _p(_c(tok, np.int32)), _p(_c(parent, np.int32)),
                          _p(_c(n_nodes, np.int32)), R, S - 1, B, V, _p(accept), _p(out_tok), _p(n_out))
    return dict(accept=accept, out_tok=out_tok, n_out=n_out)


def tv_label(target, cu_seqlens, anchor, draft, L, U, W, temperature=1.0):
    """label [R, gamma] (float64): 1 - TV(q, p) per verified window row, -1 outside."""
    R, g = draft.shape
    V = target.shape[-1]
    target = np.ascontiguousarray(target)
    L = np.ascontiguousarray(L)
    label = np.zeros((R, g), np.float64)
    flags = lib().orc_tv_label(ctypes.c_double(temperature), _p(target), _dt(target), _p(_c(cu_seqlens, np.int32)),
                               _p(_c(anchor, np.int32)), _p(_c(draft, np.int32)), _p(L), _dt(L),
                               _p(_c(U, np.uint16)), _p(_c(W, np.uint16)), U.shape[1], R, g, V, _p(label))
    return dict(label=label, flags=flags)


def observe(conf, cu_seqlens, ceiling, cls, n_class, n_bins):
    """Verify-cycle statistics (see orc_observe)."""
    R, g = conf.shape
    hist = np.zeros((n_class, g + 1), np.int32)
    reached = np.zeros((n_class, g), np.int32)
    hits = np.zeros((n_class, g), np.int32)
    bin_n = np.zeros(n_bins, np.int32)
    bin_hit = np.zeros(n_bins, np.int32)
    bin_conf = np.zeros(n_bins, np.float64)
    ece = np.zeros(1, np.float64)
    rc = lib().orc_observe(_p(_c(conf, np.float32)), _p(_c(cu_seqlens, np.int32)), _p(_c(ceiling, np.int32)),
                           _p(_c(cls, np.int32)), R, g, n_class, n_bins, _p(hist), _p(reached), _p(hits),
                           _p(bin_n), _p(bin_hit), _p(bin_conf), _p(ece))
    if rc != 0:
        raise ValueError("class id out of range")
    return dict(hist=hist, reached=reached, hits=hits, bin_n=bin_n, bin_hit=bin_hit, bin_conf=bin_conf,
                ece=float(ece[0]))


def schedule_threshold(conf, tau):
    R, g = conf.shape
    budget = np.zeros(R, np.int32)
    total = np.zeros(1, np.int32)
    lib().orc_schedule_threshold(_p(_c(conf, np.float32)), R, g, ctypes.c_float(tau), _p(budget), _p(total))
    return dict(budget=budget, total_tokens=int(total[0]))


def threshold_sweep(conf, taus, ceiling=None):
    R, g = conf.shape
    taus = _c(taus, np.float32)
    K = taus.size
    drafts = np.zeros(K, np.int32)
    accepted = np.zeros(K, np.int32)
    expected = np.zeros(K, np.float64)
    lib().orc_threshold_sweep(_p(_c(conf, np.float32)), _p(None if ceiling is None else _c(ceiling, np.int32)), R, g,
                              _p(taus), K, _p(drafts), _p(accepted), _p(expected))
    return dict(drafts=drafts, accepted=accepted, expected=expected)


def rnn_memo(A, U, X, anchor, tokens):
    """Memo trajectory [R, B, r] (float64) of the RNN head along tokens."""
    R, B, r = X.shape
    memo = np.zeros((R, B, r), np.float64)
    lib().orc_rnn_memo(_p(_c(A, np.uint16)), _p(_c(U, np.uint16)), _p(_c(X, np.uint16)), _p(_c(anchor, np.int32)),
                       _p(_c(tokens, np.int32)), R, B, r, _p(memo))
    return memo


def draft_chain_rnn(L, U, W, A, X, anchor, decode=GREEDY, temperature=1.0, seed=0, cycle=0, req_ids=None):
    """Chain draft with the RNN head; outputs as draft_chain."""
    R, B, V = L.shape
    r = U.shape[1]
    L = np.ascontiguousarray(L)
    tokens = np.zeros((R, B), np.int32)
    logq = np.zeros((R, B), np.float64)
    lse = np.zeros((R, B), np.float64)
    margin = np.zeros((R, B), np.float64)
    ids = None if req_ids is None else _c(req_ids, np.int32)
    flags = lib().orc_draft_chain_rnn(
        _p(L), _dt(L), _p(_c(U, np.uint16)), _p(_c(W, np.uint16)), _p(_c(A, np.uint16)), _p(_c(X, np.uint16)),
        _p(_c(anchor, np.int32)), _p(ids), R, B, V, r, decode, ctypes.c_double(temperature), ctypes.c_uint64(seed),
        ctypes.c_uint64(cycle), _p(tokens), _p(logq), _p(lse), _p(margin))
    return dict(tokens=tokens, logq=logq, lse=lse, margin=margin, flags=flags)


def rnn_project(L, W, memo, decode=GREEDY, temperature=1.0, seed=0, cycle=0, req_ids=None):
    """The RNN head's projection and decision for a given fp32 memo [R, B, r]
    (z_d = L_d + bf16(memo_d) W); outputs as draft_chain, each margin that of
    its own position's decision."""
    R, B, V = L.shape
    r = memo.shape[2]
    L = np.ascontiguousarray(L)
    tokens = np.zeros((R, B), np.int32)
    logq = np.zeros((R, B), np.float64)
    lse = np.zeros((R, B), np.float64)
    margin = np.zeros((R, B), np.float64)
    ids = None if req_ids is None else _c(req_ids, np.int32)
    lib().orc_rnn_project(_p(L), _dt(L), _p(_c(W, np.uint16)), _p(_c(memo, np.float32)), _p(ids), R, B, V, r, decode,
                          ctypes.c_double(temperature), ctypes.c_uint64(seed), ctypes.c_uint64(cycle), _p(tokens),
                          _p(logq), _p(lse), _p(margin))
    return dict(tokens=tokens, logq=logq, lse=lse, margin=margin)
