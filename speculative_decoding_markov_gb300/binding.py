"""Python binding of libsdm.so (ctypes): argument marshalling only.

`sdm_*` are the raw C entry points (pointers and sizes).  The lower-case
helpers take torch CUDA tensors, allocate outputs and the workspace with
torch (device memory is all torch provides here), call the C entry point on
the current stream and return the outputs.  Every computation happens in the
library's CUDA kernels; there is no fallback: if libsdm.so is missing or no
GPU is present the calls raise.
"""
from __future__ import annotations

import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libsdm.so")

BF16, FP32 = 0, 1
GREEDY, SAMPLE = 0, 1
STATIC, COMPACT, CAP_ACCEPT = 0, 1, 2
OP_DRAFT_CHAIN, OP_DRAFT_TREE, OP_SCHEDULE, OP_PACK, OP_VERIFY, OP_VERIFY_TREE, OP_TV_LABEL, OP_DRAFT_CHAIN_RNN = range(8)
DEV_BAD_TOKEN, DEV_TIER_UNCAPTURED, DEV_TIMEOUT, DEV_BAD_WINDOW, DEV_CAPACITY, DEV_BAD_CLASS = 1, 2, 4, 8, 16, 32
DEV_TIER_OVERFLOW = 64

EXPORTS = ("sdm_workspace_size", "sdm_markov_prepared_size", "sdm_markov_prepare", "sdm_draft_chain",
           "sdm_draft_tree", "sdm_schedule_budget", "sdm_pack_ragged", "sdm_verify", "sdm_verify_tree",
           "sdm_verify_greedy_static", "sdm_schedule_dynamic", "sdm_tv_label", "sdm_observe", "sdm_schedule_threshold",
           "sdm_threshold_sweep", "sdm_draft_chain_rnn", "sdm_status_str", "sdm_status_of_device", "sdm_check_timeout_path",
           "sdm_draft_chain_packed", "sdm_draft_chain_front",
           "sdm_version")


class SdmRng(ctypes.Structure):
    _fields_ = [("seed", ctypes.c_uint64), ("cycle", ctypes.c_uint64)]


_lib = None
_VP, _I, _F, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t


def _declare(lib):
    lib.sdm_workspace_size.restype = _SZ
    lib.sdm_workspace_size.argtypes = [_I] * 8
    lib.sdm_status_str.restype = ctypes.c_char_p
    lib.sdm_status_str.argtypes = [_I]
    lib.sdm_version.restype = _I
    lib.sdm_markov_prepared_size.restype = _SZ
    lib.sdm_markov_prepared_size.argtypes = [_I, _I]
    lib.sdm_markov_prepare.restype = _I
    lib.sdm_markov_prepare.argtypes = [_VP, _VP, _I, _I, _VP, _SZ, _VP, _VP]
    lib.sdm_draft_chain.restype = _I
    lib.sdm_draft_chain.argtypes = [_VP, _I, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _F, SdmRng, _VP, _VP, _VP, _VP,
                                    _SZ, _VP, _VP]
    lib.sdm_draft_tree.restype = _I
    lib.sdm_draft_tree.argtypes = [_VP, _I, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I, _I, _VP, _VP, _VP, _VP, _VP,
                                   _VP, _VP, _SZ, _VP, _VP]
    lib.sdm_schedule_budget.restype = _I
    lib.sdm_schedule_budget.argtypes = [_VP, _I, _I, _VP, _VP, _VP, _VP, _VP, _VP, _SZ, _VP, _VP]
    lib.sdm_schedule_dynamic.restype = _I
    lib.sdm_schedule_dynamic.argtypes = [_VP, _VP, _I, _I, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP]
    lib.sdm_pack_ragged.restype = _I
    lib.sdm_pack_ragged.argtypes = [_VP, _VP, _VP, _I, _I, _VP, _I, _I, _VP, _VP, _VP, _VP, _I, _VP, _VP, _VP, _VP]
    lib.sdm_draft_chain_front.restype = _I
    lib.sdm_draft_chain_front.argtypes = [_VP, _I, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _VP, _VP, _I, _VP, _I, _I,
                                          _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _I, _VP, _VP, _VP, _SZ, _VP, _VP]
    lib.sdm_draft_chain_packed.restype = _I
    lib.sdm_draft_chain_packed.argtypes = [_VP, _I, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _VP, _VP, _I, _VP, _VP, _VP,
                                           _SZ, _VP, _VP]
    lib.sdm_check_timeout_path.restype = _I
    lib.sdm_check_timeout_path.argtypes = [_VP, _I, _VP, _VP, _VP, _I, _I, _I, _I, ctypes.c_ulonglong, _VP, _SZ, _VP,
                                           _VP]
    lib.sdm_status_of_device.restype = _I
    lib.sdm_status_of_device.argtypes = [ctypes.c_int32]
    lib.sdm_verify.restype = _I
    lib.sdm_verify.argtypes = [_I, _I, _F, SdmRng, _VP, _I, _I, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _I, _VP, _VP, _I,
                               _I, _I, _I, _VP, _VP, _VP, _VP, _VP, _SZ, _VP, _VP]
    lib.sdm_verify_greedy_static.restype = _I
    lib.sdm_verify_greedy_static.argtypes = [_I, _VP, _I, _I, _VP, _VP, _VP, _I, _I, _I, _VP, _VP, _VP, _VP, _VP, _VP]
    lib.sdm_draft_chain_rnn.restype = _I
    lib.sdm_draft_chain_rnn.argtypes = [_VP, _I, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _F, SdmRng, _VP, _VP, _VP,
                                        _VP, _VP, _SZ, _VP, _VP]
    lib.sdm_schedule_threshold.restype = _I
    lib.sdm_schedule_threshold.argtypes = [_VP, _I, _I, _F, _VP, _VP, _VP, _VP]
    lib.sdm_threshold_sweep.restype = _I
    lib.sdm_threshold_sweep.argtypes = [_VP, _VP, _I, _I, _VP, _I, _VP, _VP, _VP, _VP, _VP]
    lib.sdm_tv_label.restype = _I
    lib.sdm_tv_label.argtypes = [_F, _VP, _I, _I, _VP, _VP, _VP, _VP, _VP, _I, _VP, _VP, _I, _I, _I, _I, _VP, _VP,
                                 _SZ, _VP, _VP]
    lib.sdm_observe.restype = _I
    lib.sdm_observe.argtypes = [_VP, _VP, _VP, _VP, _I, _I, _I, _I, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP]
    lib.sdm_verify_tree.restype = _I
    lib.sdm_verify_tree.argtypes = [_VP, _I, _VP, _VP, _VP, _I, _I, _I, _I, _VP, _VP, _VP, _VP, _SZ, _VP, _VP]


def load(path: str = LIB_PATH):
    """Load libsdm.so (built by __graft_entry__.build / build.py); raises if absent."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(f"libsdm.so not built at {path}: run speculative_decoding_markov_gb300.build")
        lib = ctypes.CDLL(path)
        _declare(lib)
        _lib = lib
    return _lib


def lib():
    return load()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _check(st: int, what: str):
    if st != 0:
        raise RuntimeError(f"{what}: {lib().sdm_status_str(st).decode()} (status {st})")


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return FP32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _need_cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("inputs must be contiguous CUDA tensors")


def _need_cost(cost, R, gamma):
    """The step-cost table the schedulers index up to cost[R * (gamma + 1)]:
    fp64 with at least R * (gamma + 1) + 1 entries."""
    if cost.dtype != torch.float64 or cost.numel() < R * (gamma + 1) + 1:
        raise ValueError(f"cost must be fp64 with at least R*(gamma+1)+1 = {R * (gamma + 1) + 1} entries")


def _u16(t):
    """bf16 tensors are passed by pointer; this only checks the dtype."""
    if t.dtype != torch.bfloat16:
        raise TypeError("U and W must be bf16")
    return t


def workspace(op, R, B=0, V=0, r=0, P=0, k=0, N=0, device="cuda"):
    n = lib().sdm_workspace_size(op, R, B, V, r, P, k, N)
    return torch.empty(max(int(n), 256), dtype=torch.uint8, device=device)


def new_status(device="cuda"):
    return torch.zeros(1, dtype=torch.int32, device=device)


# ---------------------------------------------------------------------------
def markov_prepare(U, W, out=None, dev_status=None):
    """Prepared tables of the Markov head (W^T, per-token bounds of the Markov
    term) for greedy drafting."""
    _need_cuda(U, W)
    V, r = U.shape
    n = lib().sdm_markov_prepared_size(V, r)
    if out is None:
        out = torch.empty(int(n), dtype=torch.uint8, device=U.device)
    st = lib().sdm_markov_prepare(_ptr(_u16(U)), _ptr(_u16(W)), V, r, _ptr(out), out.numel(), _ptr(dev_status),
                                  _stream())
    _check(st, "sdm_markov_prepare")
    return out


def draft_chain(L, U, W, anchor, decode=GREEDY, temperature=1.0, seed=0, cycle=0, out=None, ws=None,
                dev_status=None, prepared=None):
    _need_cuda(L, U, W, anchor)
    R, B, V = L.shape
    r = U.shape[1]
    dev = L.device
    if out is None:
        out = dict(tokens=torch.empty((R, B), dtype=torch.int32, device=dev),
                   logq=torch.zeros((R, B), dtype=torch.float32, device=dev),
                   lse=torch.zeros((R, B), dtype=torch.float32, device=dev))
    ws = workspace(OP_DRAFT_CHAIN, R, B, V, r, device=dev) if ws is None else ws
    dev_status = new_status(dev) if dev_status is None else dev_status
    st = lib().sdm_draft_chain(_ptr(L), _dt(L), _ptr(_u16(U)), _ptr(_u16(W)), _ptr(prepared), _ptr(anchor), R, B, V,
                               r, decode,
                               float(temperature), SdmRng(seed, cycle), _ptr(out["tokens"]), _ptr(out["logq"]),
                               _ptr(out["lse"]), _ptr(ws), ws.numel(), _ptr(dev_status), _stream())
    _check(st, "sdm_draft_chain")
    out["dev_status"] = dev_status
    return out


def draft_chain_packed(L, U, W, anchor, prepared, cu_seqlens, packed_tok, tokens=None, layout_ready=None, ws=None,
                       dev_status=None):
    """Greedy chain draft (prepared tables) that also fills its drafts into a
    ragged layout made by pack_ragged(draft=None); layout_ready: a
    torch.cuda.Event recorded after that layout's producer (or None)."""
    _need_cuda(L, U, W, anchor, cu_seqlens, packed_tok)
    R, B, V = L.shape
    r = U.shape[1]
    dev = L.device
    tokens = torch.empty((R, B), dtype=torch.int32, device=dev) if tokens is None else tokens
    ws = workspace(OP_DRAFT_CHAIN, R, B, V, r, device=dev) if ws is None else ws
    dev_status = new_status(dev) if dev_status is None else dev_status
    ev = None if layout_ready is None else ctypes.c_void_p(layout_ready.cuda_event)
    st = lib().sdm_draft_chain_packed(_ptr(L), _dt(L), _ptr(_u16(U)), _ptr(_u16(W)), _ptr(prepared), _ptr(anchor), R,
                                      B, V, r, _ptr(cu_seqlens), _ptr(packed_tok), packed_tok.numel(), ev,
                                      _ptr(tokens), _ptr(ws), ws.numel(), _ptr(dev_status), _stream())
    _check(st, "sdm_draft_chain_packed")
    return dict(tokens=tokens, dev_status=dev_status)


def draft_chain_front(L, U, W, anchor, prepared, conf, cost, tiers, use_budget=True, strict=False, tokens=None,
                      sched=None, pk=None, capacity=None, ws=None, dev_status=None):
    """Greedy chain draft (prepared tables) with the budget scheduler and the
    ragged layout in the same launches: the outputs of schedule_budget,
    pack_ragged(draft=None) and draft_chain_packed.  sched / pk: output dicts
    as those calls return (made here when None)."""
    _need_cuda(L, U, W, anchor, conf, cost, tiers)
    R, B, V = L.shape
    _need_cost(cost, R, B)
    r = U.shape[1]
    dev = L.device
    tokens = torch.empty((R, B), dtype=torch.int32, device=dev) if tokens is None else tokens
    if sched is None:
        sched = dict(survival=torch.empty((R, B), dtype=torch.float32, device=dev),
                     budget=torch.empty((R,), dtype=torch.int32, device=dev),
                     expected=torch.empty((1,), dtype=torch.float64, device=dev),
                     total_tokens=torch.empty((1,), dtype=torch.int32, device=dev))
    if pk is None:
        cap = capacity if capacity else pack_capacity(R, B, tiers.tolist())
        pk = dict(cu_seqlens=torch.empty((R + 1,), dtype=torch.int32, device=dev),
                  packed_tok=torch.empty((cap,), dtype=torch.int32, device=dev),
                  packed_req=torch.empty((cap,), dtype=torch.int32, device=dev),
                  packed_pos=torch.empty((cap,), dtype=torch.int32, device=dev),
                  tier=torch.empty((1,), dtype=torch.int32, device=dev))
    ws = workspace(OP_DRAFT_CHAIN, R, B, V, r, device=dev) if ws is None else ws
    dev_status = new_status(dev) if dev_status is None else dev_status
    st = lib().sdm_draft_chain_front(
        _ptr(L), _dt(L), _ptr(_u16(U)), _ptr(_u16(W)), _ptr(prepared), _ptr(anchor), R, B, V, r, _ptr(conf),
        _ptr(cost), 1 if use_budget else 0, _ptr(tiers), tiers.numel(), 1 if strict else 0, _ptr(sched["survival"]),
        _ptr(sched["budget"]), _ptr(sched["expected"]), _ptr(sched["total_tokens"]), _ptr(pk["cu_seqlens"]),
        _ptr(pk["packed_tok"]), _ptr(pk["packed_req"]), _ptr(pk["packed_pos"]), pk["packed_tok"].numel(),
        _ptr(pk["tier"]), _ptr(tokens), _ptr(ws), ws.numel(), _ptr(dev_status), _stream())
    _check(st, "sdm_draft_chain_front")
    return dict(tokens=tokens, sched=sched, pk=pk, dev_status=dev_status)


def check_timeout_path(L, U, W, anchor, wait_ns, dev_status=None):
    """One Markov GEMM launch with its loads withheld and every wait limited
    to wait_ns: the kernel records DEV_TIMEOUT and winds down."""
    _need_cuda(L, U, W, anchor)
    R, B, V = L.shape
    r = U.shape[1]
    ws = workspace(OP_DRAFT_CHAIN, R, B, V, r, device=L.device)
    dev_status = new_status(L.device) if dev_status is None else dev_status
    st = lib().sdm_check_timeout_path(_ptr(L), _dt(L), _ptr(_u16(U)), _ptr(_u16(W)), _ptr(anchor), R, B, V, r,
                                      int(wait_ns), _ptr(ws), ws.numel(), _ptr(dev_status), _stream())
    _check(st, "sdm_check_timeout_path")
    return dev_status


def draft_chain_rnn(L, U, W, A, X, anchor, decode=GREEDY, temperature=1.0, seed=0, cycle=0, out=None, ws=None,
                    dev_status=None, memo=False):
    """Chain draft with the RNN head (memo m_d = tanh(A m_{d-1} + U[y_{d-1}]
    + x_d), logits L_d + bf16(m_d) W); memo=True also returns the memo."""
    _need_cuda(L, U, W, A, X, anchor)
    R, B, V = L.shape
    r = U.shape[1]
    dev = L.device
    if out is None:
        out = dict(tokens=torch.empty((R, B), dtype=torch.int32, device=dev),
                   logq=torch.zeros((R, B), dtype=torch.float32, device=dev),
                   lse=torch.zeros((R, B), dtype=torch.float32, device=dev))
        if memo:
            out["memo"] = torch.empty((R, B, r), dtype=torch.float32, device=dev)
    ws = workspace(OP_DRAFT_CHAIN_RNN, R, B, V, r, device=dev) if ws is None else ws
    dev_status = new_status(dev) if dev_status is None else dev_status
    st = lib().sdm_draft_chain_rnn(_ptr(L), _dt(L), _ptr(_u16(U)), _ptr(_u16(W)), _ptr(_u16(A)), _ptr(_u16(X)),
                                   _ptr(anchor), R, B, V, r, decode, float(temperature), SdmRng(seed, cycle),
                                   _ptr(out["tokens"]), _ptr(out.get("logq")), _ptr(out.get("lse")),
                                   _ptr(out.get("memo")), _ptr(ws), ws.numel(), _ptr(dev_status), _stream())
    _check(st, "sdm_draft_chain_rnn")
    out["dev_status"] = dev_status
    return out


def draft_tree(L, U, W, anchor, k, P, N, out=None, ws=None, dev_status=None, prepared=None):
    _need_cuda(L, U, W, anchor)
    R, B, V = L.shape
    r = U.shape[1]
    dev = L.device
    S = N + 1
    words = (S + 31) // 32
    if out is None:
        out = dict(tok=torch.empty((R, S), dtype=torch.int32, device=dev),
                   parent=torch.empty((R, S), dtype=torch.int32, device=dev),
                   depth=torch.empty((R, S), dtype=torch.int32, device=dev),
                   score=torch.empty((R, S), dtype=torch.float32, device=dev),
                   mask=torch.empty((R, S, words), dtype=torch.int32, device=dev),
                   n_nodes=torch.empty((R,), dtype=torch.int32, device=dev))
    ws = workspace(OP_DRAFT_TREE, R, B, V, r, P, k, N, device=dev) if ws is None else ws
    dev_status = new_status(dev) if dev_status is None else dev_status
    st = lib().sdm_draft_tree(_ptr(L), _dt(L), _ptr(_u16(U)), _ptr(_u16(W)), _ptr(prepared), _ptr(anchor), R, B, V, r,
                              k, P, N,
                              _ptr(out["tok"]), _ptr(out["parent"]), _ptr(out["depth"]), _ptr(out["score"]),
                              _ptr(out["mask"]), _ptr(out["n_nodes"]), _ptr(ws), ws.numel(), _ptr(dev_status),
                              _stream())
    _check(st, "sdm_draft_tree")
    out["dev_status"] = dev_status
    return out


def schedule_budget(conf, cost, out=None, dev_status=None):
    _need_cuda(conf, cost)
    R, g = conf.shape
    _need_cost(cost, R, g)
    dev = conf.device
    if out is None:
        out = dict(survival=torch.empty((R, g), dtype=torch.float32, device=dev),
                   budget=torch.empty((R,), dtype=torch.int32, device=dev),
                   expected=torch.empty((1,), dtype=torch.float64, device=dev),
                   total_tokens=torch.empty((1,), dtype=torch.int32, device=dev))
    dev_status = new_status(dev) if dev_status is None else dev_status
    st = lib().sdm_schedule_budget(_ptr(conf), R, g, _ptr(cost), _ptr(out["survival"]), _ptr(out["budget"]),
                                   _ptr(out["expected"]), _ptr(out["total_tokens"]), None, 0, _ptr(dev_status),
                                   _stream())
    _check(st, "sdm_schedule_budget")
    out["dev_status"] = dev_status
    return out


def schedule_dynamic(conf, conf_stale, cost, out=None, dev_status=None):
    """The production scheduler: capacity from conf_stale (the confidences of
    two steps before) by a global search over cost, then the top K of conf's
    survivals."""
    _need_cuda(conf, conf_stale, cost)
    R, g = conf.shape
    _need_cost(cost, R, g)
    assert tuple(conf_stale.shape) == (R, g)
    dev = conf.device
    if out is None:
        out = dict(survival=torch.empty((R, g), dtype=torch.float32, device=dev),
                   budget=torch.empty((R,), dtype=torch.int32, device=dev),
                   expected=torch.empty((1,), dtype=torch.float64, device=dev),
                   total_tokens=torch.empty((1,), dtype=torch.int32, device=dev),
                   capacity=torch.empty((1,), dtype=torch.int32, device=dev))
    dev_status = new_status(dev) if dev_status is None else dev_status
    st = lib().sdm_schedule_dynamic(_ptr(conf), _ptr(conf_stale), R, g, _ptr(cost), _ptr(out["survival"]),
                                    _ptr(out["budget"]), _ptr(out["expected"]), _ptr(out["total_tokens"]),
                                    _ptr(out["capacity"]), _ptr(dev_status), _stream())
    _check(st, "sdm_schedule_dynamic")
    out["dev_status"] = dev_status
    return out


def schedule_threshold(conf, tau, out=None, dev_status=None):
    """Fixed-threshold verify length: the longest prefix with every
    confidence >= tau."""
    _need_cuda(conf)
    R, g = conf.shape
    dev = conf.device
    if out is None:
        out = dict(budget=torch.empty((R,), dtype=torch.int32, device=dev),
                   total_tokens=torch.empty((1,), dtype=torch.int32, device=dev))
    dev_status = new_status(dev) if dev_status is None else dev_status
    st = lib().sdm_schedule_threshold(_ptr(conf), R, g, float(tau), _ptr(out["budget"]), _ptr(out["total_tokens"]),
                                      _ptr(dev_status), _stream())
    _check(st, "sdm_schedule_threshold")
    return out


def threshold_sweep(conf, taus, ceiling=None, out=None, dev_status=None):
    """Drafts verified, drafts accepted (given whole-block ceilings) and
    expected accepted drafts at every threshold in taus."""
    _need_cuda(conf, taus, ceiling)
    R, g = conf.shape
    K = taus.numel()
    dev = conf.device
    if out is None:
        out = dict(drafts=torch.empty((K,), dtype=torch.int32, device=dev),
                   accepted=torch.empty((K,), dtype=torch.int32, device=dev),
                   expected=torch.empty((K,), dtype=torch.float64, device=dev))
    dev_status = new_status(dev) if dev_status is None else dev_status
    st = lib().sdm_threshold_sweep(_ptr(conf), _ptr(ceiling), R, g, _ptr(taus), K, _ptr(out["drafts"]),
                                   _ptr(out["accepted"]), _ptr(out["expected"]), _ptr(dev_status), _stream())
    _check(st, "sdm_threshold_sweep")
    return out


def pack_capacity(R, gamma, tiers) -> int:
    return max(max(tiers) if len(tiers) else 0, R * (gamma + 1))


def pack_ragged(anchor, draft, budget, tiers, capacity=None, out=None, dev_status=None, tier_host=None,
                strict=False, gamma=None):
    """Ragged front-pack; draft=None (give gamma) lays out the windows alone,
    every draft row -1, for draft_chain_packed to fill."""
    _need_cuda(anchor, draft, budget, tiers)
    R = anchor.numel()
    g = draft.shape[1] if draft is not None else int(gamma)
    dev = anchor.device
    if out is None:
        cap = capacity if capacity else pack_capacity(R, g, tiers.tolist())
        out = dict(cu_seqlens=torch.empty((R + 1,), dtype=torch.int32, device=dev),
                   packed_tok=torch.empty((cap,), dtype=torch.int32, device=dev),
                   packed_req=torch.empty((cap,), dtype=torch.int32, device=dev),
                   packed_pos=torch.empty((cap,), dtype=torch.int32, device=dev),
                   tier=torch.empty((1,), dtype=torch.int32, device=dev))
    cap = out["packed_tok"].numel()
    dev_status = new_status(dev) if dev_status is None else dev_status
    st = lib().sdm_pack_ragged(_ptr(anchor), _ptr(draft), _ptr(budget), R, g, _ptr(tiers), tiers.numel(),
                               1 if strict else 0, _ptr(out["cu_seqlens"]), _ptr(out["packed_tok"]), _ptr(out["packed_req"]),
                               _ptr(out["packed_pos"]), cap, _ptr(out["tier"]), _ptr(tier_host), _ptr(dev_status),
                               _stream())
    _check(st, "sdm_pack_ragged")
    out["dev_status"] = dev_status
    return out


def verify(mode, decode, target, cu_seqlens, anchor, draft, budget=None, logq=None, lse_q=None, L=None, U=None,
           W=None, temperature=1.0, seed=0, cycle=0, out=None, ws=None, dev_status=None):
    _need_cuda(target, cu_seqlens, anchor, draft, budget, logq, lse_q, L, U, W)
    R, g = draft.shape
    V = target.shape[-1]
    rows = target.numel() // V
    dev = target.device
    r = 0 if U is None else U.shape[1]
    if out is None:
        out = dict(accept=torch.empty((R,), dtype=torch.int32, device=dev),
                   ceiling=torch.empty((R,), dtype=torch.int32, device=dev),
                   out_tok=torch.empty((R, g + 1), dtype=torch.int32, device=dev),
                   n_out=torch.empty((R,), dtype=torch.int32, device=dev))
    ws = workspace(OP_VERIFY, R, g, V, r, rows, device=dev) if ws is None else ws
    dev_status = new_status(dev) if dev_status is None else dev_status
    st = lib().sdm_verify(mode, decode, float(temperature), SdmRng(seed, cycle), _ptr(target), _dt(target), rows,
                          _ptr(cu_seqlens), _ptr(anchor), _ptr(draft), _ptr(budget), _ptr(logq), _ptr(lse_q),
                          _ptr(L), _dt(L) if L is not None else BF16, _ptr(U), _ptr(W), r, R, g, V,
                          _ptr(out["accept"]), _ptr(out["ceiling"]), _ptr(out["out_tok"]), _ptr(out["n_out"]),
                          _ptr(ws), ws.numel(), _ptr(dev_status), _stream())
    _check(st, "sdm_verify")
    out["dev_status"] = dev_status
    return out


def tv_label(target, cu_seqlens, anchor, draft, L, U, W, lse_q=None, temperature=1.0, out=None, ws=None,
             dev_status=None):
    """Soft label 1 - TV(q, p) [R, gamma] of every verified window row (-1
    past the window).  target holds the packed verify rows; lse_q (the
    sampling draft's log-sum-exp) may be None."""
    _need_cuda(target, cu_seqlens, anchor, draft, L, U, W, lse_q)
    R, g = draft.shape
    V = target.shape[-1]
    rows = target.numel() // V
    dev = target.device
    r = U.shape[1]
    if out is None:
        out = torch.empty((R, g), dtype=torch.float32, device=dev)
    ws = workspace(OP_TV_LABEL, R, g, V, r, rows, device=dev) if ws is None else ws
    dev_status = new_status(dev) if dev_status is None else dev_status
    st = lib().sdm_tv_label(float(temperature), _ptr(target), _dt(target), rows, _ptr(cu_seqlens), _ptr(anchor),
                            _ptr(draft), _ptr(lse_q), _ptr(L), _dt(L), _ptr(_u16(U)), _ptr(_u16(W)), r, R, g, V,
                            _ptr(out), _ptr(ws), ws.numel(), _ptr(dev_status), _stream())
    _check(st, "sdm_tv_label")
    return out


def observe(conf, cu_seqlens, ceiling, cls, n_class, n_bins, out=None, dev_status=None):
    """Verify-cycle statistics: ceiling histograms per class, per-position
    observed / accepted counts, calibration bins and their ECE."""
    _need_cuda(conf, cu_seqlens, ceiling, cls)
    R, g = conf.shape
    dev = conf.device
    i32 = dict(dtype=torch.int32, device=dev)
    if out is None:
        out = dict(hist=torch.empty((n_class, g + 1), **i32), reached=torch.empty((n_class, g), **i32),
                   hits=torch.empty((n_class, g), **i32), bin_n=torch.empty((n_bins,), **i32),
                   bin_hit=torch.empty((n_bins,), **i32),
                   bin_conf=torch.empty((n_bins,), dtype=torch.float64, device=dev),
                   ece=torch.empty((1,), dtype=torch.float64, device=dev))
    dev_status = new_status(dev) if dev_status is None else dev_status
    st = lib().sdm_observe(_ptr(conf), _ptr(cu_seqlens), _ptr(ceiling), _ptr(cls), R, g, n_class, n_bins,
                           _ptr(out["hist"]), _ptr(out["reached"]), _ptr(out["hits"]), _ptr(out["bin_n"]),
                           _ptr(out["bin_hit"]), _ptr(out["bin_conf"]), _ptr(out["ece"]), _ptr(dev_status),
                           _stream())
    _check(st, "sdm_observe")
    out["dev_status"] = dev_status
    return out


def verify_tree(target, tok, parent, n_nodes, B, out=None, ws=None, dev_status=None):
    _need_cuda(target, tok, parent, n_nodes)
    R, S, V = target.shape
    dev = target.device
    if out is None:
        out = dict(accept=torch.empty((R,), dtype=torch.int32, device=dev),
                   out_tok=torch.empty((R, B + 1), dtype=torch.int32, device=dev),
                   n_out=torch.empty((R,), dtype=torch.int32, device=dev))
    ws = workspace(OP_VERIFY_TREE, R, B, V, 0, 0, 0, S - 1, device=dev) if ws is None else ws
    dev_status = new_status(dev) if dev_status is None else dev_status
    st = lib().sdm_verify_tree(_ptr(target), _dt(target), _ptr(tok), _ptr(parent), _ptr(n_nodes), R, S - 1, B, V,
                               _ptr(out["accept"]), _ptr(out["out_tok"]), _ptr(out["n_out"]), _ptr(ws), ws.numel(),
                               _ptr(dev_status), _stream())
    _check(st, "sdm_verify_tree")
    out["dev_status"] = dev_status
    return out
