"""Seeded synthetic inputs for the hot path (shared by the CUDA path and the oracle).

Holds only input synthesis: random backbone logits, Markov tables, anchors,
target noise, confidences, cost tables, and the stand-in for the target LLM
forward pass.  None of the method's own steps (drafting, scheduling, packing,
verification) lives here.

The stand-in target model.  The drafter backbone and the target LLM are out
of scope; the pages' synthetic workloads describe the target as "draft logits
plus noise".  It is modelled as a function of the position d and the previous
token:

    T_d(prev) = (L_d + U[prev] W) + eta_d        (fp32, then the target dtype)

so along any drafted prefix the target row equals the drafter's logits plus
eta, and target-only greedy decoding is defined for any prefix.  The bonus
position B+1 uses an extra backbone row L_bonus drawn here for the target
only.  U and W sit on a 2^-8 grid (|value| < 1), so U[prev] W is exact in
fp32 whatever the summation order; every device and library computes the same
target rows bit for bit.
"""
from __future__ import annotations

import math

import torch

from .workloads import BF16, FP32, Workload

_TORCH_DTYPE = {BF16: torch.bfloat16, FP32: torch.float32}

# distinct generator streams per tensor (seed * 64 + stream)
_S_L, _S_LB, _S_U, _S_W, _S_ANCHOR, _S_ETA, _S_CONF, _S_CLASS, _S_STALE, _S_ARNN, _S_XRNN = range(16, 27)


def torch_dtype(code: int) -> torch.dtype:
    return _TORCH_DTYPE[code]


def _gen(seed: int, stream: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 64 + stream)
    return g


def grid_table(shape, r: int, seed: int, stream: int, device) -> torch.Tensor:
    """N(0, 1/r) entries rounded to the 2^-8 grid, clamped to +-255/256, bf16.

    Every entry is k/256 with |k| <= 255 (exactly representable in bf16) so
    each product U*W is a multiple of 2^-16 below 1 and every partial sum over
    r <= 256 terms stays below 2^8: the Markov product is exact in fp32.
    """
    g = torch.randn(shape, generator=_gen(seed, stream, device), device=device, dtype=torch.float32)
    q = torch.clamp(torch.round(g * (256.0 / math.sqrt(r))), -255.0, 255.0) / 256.0
    return q.to(torch.bfloat16)


def request_class(w: Workload, seed: int) -> torch.Tensor:
    """Traffic class of every request (int64 [R], CPU): its target-noise std
    is w.sigma[class]."""
    nc = len(w.sigma)
    if nc == 1:
        return torch.zeros(w.R, dtype=torch.int64)
    if w.class_mix == "alternate":
        return torch.arange(w.R) % nc
    # equal class shares (rounded up), shuffled, truncated to R
    per = -(-w.R // nc)
    pool = torch.arange(nc).repeat_interleave(per)
    perm = torch.randperm(pool.numel(), generator=_gen(seed, _S_CLASS, "cpu"))
    return pool[perm][: w.R]


def request_sigma(w: Workload, seed: int, device) -> torch.Tensor:
    """Per-request target-noise std (fp32 [R])."""
    s = torch.tensor(w.sigma, dtype=torch.float32)[request_class(w, seed)]
    return s.to(device)


def cost_table(w: Workload, R: int | None = None, B: int | None = None) -> torch.Tensor:
    """Additive step cost a + b N for N = 0 .. R (B + 1), fp64."""
    R = w.R if R is None else R
    B = w.B if B is None else B
    a, b = w.cost
    n = torch.arange(R * (B + 1) + 1, dtype=torch.float64)
    return a + b * n


def tiered_cost_table(w: Workload, R: int | None = None, B: int | None = None) -> torch.Tensor:
    """The stepped form of the additive table: a + b tier(N), tier(N) = the
    smallest captured tier >= N (N itself above every tier), the cost of the
    graph a packed total actually replays (fp64)."""
    R = w.R if R is None else R
    B = w.B if B is None else B
    a, b = w.cost
    tiers = sorted(w.tiers)
    n = torch.arange(R * (B + 1) + 1, dtype=torch.float64)
    t = torch.tensor([next((x for x in tiers if x >= k), k) for k in range(R * (B + 1) + 1)], dtype=torch.float64)
    return a + b * t if tiers else a + b * n


def stale_confidences(conf: torch.Tensor, seed: int) -> torch.Tensor:
    """Stand-in for the confidences of the same requests two steps before:
    this step's, moved in logit space by N(0, 0.5) (fp32 [R, B])."""
    x = torch.logit(conf.to(torch.float64).clamp(1e-6, 1 - 1e-6))
    noise = torch.randn(conf.shape, generator=_gen(seed, _S_STALE, conf.device), device=conf.device,
                        dtype=torch.float64) * 0.5
    return torch.sigmoid(x + noise).to(torch.float32)


def rnn_inputs(w: Workload, seed: int = 0, device="cpu", a_scale: float = 0.9, x_std: float = 0.5) -> dict:
    """Weights and inputs of the RNN head (bf16): the memo recurrence A
    [r, r] with entries N(0, a_scale^2 / r) (spectral radius near a_scale),
    and the backbone state projected to the memo's size, X [R, B, r] ~
    N(0, x_std^2)."""
    R, B, r = w.R, w.B, w.r
    A = torch.randn((r, r), generator=_gen(seed, _S_ARNN, device), device=device) * (a_scale / math.sqrt(r))
    X = torch.randn((R, B, r), generator=_gen(seed, _S_XRNN, device), device=device) * x_std
    return dict(A_rnn=A.to(torch.bfloat16), X_rnn=X.to(torch.bfloat16))


def generate(w: Workload, seed: int = 0, device="cpu") -> dict:
    """All inputs of one decode cycle of workload w, on `device`."""
    R, B, V, r = w.R, w.B, w.V, w.r
    ldt = _TORCH_DTYPE[w.l_dtype]
    L = (torch.randn((R, B, V), generator=_gen(seed, _S_L, device), device=device) * w.l_std).to(ldt)
    L_bonus = (torch.randn((R, V), generator=_gen(seed, _S_LB, device), device=device) * w.l_std).to(ldt)
    U = grid_table((V, r), r, seed, _S_U, device)
    W = grid_table((r, V), r, seed, _S_W, device)
    anchor = torch.randint(0, V, (R,), generator=_gen(seed, _S_ANCHOR, device), device=device,
                           dtype=torch.int64).to(torch.int32)
    sigma = request_sigma(w, seed, device)
    eta = torch.randn((R, B + 1, V), generator=_gen(seed, _S_ETA, device), device=device) * sigma.view(R, 1, 1)
    out = dict(L=L, L_bonus=L_bonus, U=U, W=W, anchor=anchor, sigma=sigma, eta=eta,
               cost=cost_table(w).to(device), tiers=torch.tensor(w.tiers, dtype=torch.int32, device=device))
    out["conf"] = confidences(w, out, seed, device)
    out["conf_stale"] = stale_confidences(out["conf"], seed)
    out["cost_tiered"] = tiered_cost_table(w).to(device)
    return out


def confidences(w: Workload, inp: dict, seed: int, device) -> torch.Tensor:
    """Post-sigmoid confidences c_{i,d} (fp32 [R, B]); the confidence head is out of scope."""
    R, B = w.R, w.B
    if w.conf == "sigmoid":
        x = torch.randn((R, B), generator=_gen(seed, _S_CONF, device), device=device, dtype=torch.float64) + 1.0
        return torch.sigmoid(x).to(torch.float32)
    # soft acceptance label 1 - TV(q, p) = sum_v min(q_v, p_v) between the
    # backbone distribution at position d and the noisy target there
    c = torch.empty((R, B), dtype=torch.float64, device=device)
    for d in range(B):
        ld = inp["L"][:, d, :].to(torch.float64)
        q = torch.softmax(ld, dim=-1)
        p = torch.softmax(ld + inp["eta"][:, d, :].to(torch.float64), dim=-1)
        c[:, d] = torch.minimum(q, p).sum(dim=-1)
    return c.to(torch.float32)


def target_rows(inp: dict, req: torch.Tensor, pos: torch.Tensor, prev: torch.Tensor,
                target_dtype: int, chunk: int = 1024) -> torch.Tensor:
    """Stand-in target logits for rows (request, window position, previous token).

    Row (i, p, prev) is T_{p+1}(prev) = (L[i, p] + U[prev] W) + eta[i, p], with
    L[i, B] meaning L_bonus[i].  Returns [n, V] in the target dtype.
    """
    L, Lb, U, W, eta = inp["L"], inp["L_bonus"], inp["U"], inp["W"], inp["eta"]
    B = L.shape[1]
    n = req.numel()
    V = L.shape[2]
    out = torch.empty((n, V), dtype=_TORCH_DTYPE[target_dtype], device=L.device)
    Wf = W.to(torch.float32)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        ri, pi, yi = req[s:e].long(), pos[s:e].long(), prev[s:e].long()
        lrow = torch.where((pi < B).view(-1, 1), L[ri, pi.clamp(max=B - 1)].to(torch.float32),
                           Lb[ri].to(torch.float32))
        m = U[yi].to(torch.float32) @ Wf
        z = lrow + m
        t = z + eta[ri, pi]
        out[s:e] = t.to(out.dtype)
    return out


def chain_target(inp: dict, tokens: torch.Tensor, target_dtype: int) -> torch.Tensor:
    """Target logits for every window row of a drafted chain: [R, B+1, V].

    Row p of request i is the target's prediction after y_p (y_0 = anchor).
    """
    R, B = tokens.shape
    dev = tokens.device
    prev = torch.cat([inp["anchor"].view(R, 1).to(dev), tokens.to(torch.int32)], dim=1)
    req = torch.arange(R, device=dev).repeat_interleave(B + 1)
    pos = torch.arange(B + 1, device=dev).repeat(R)
    return target_rows(inp, req, pos, prev.reshape(-1), target_dtype).view(R, B + 1, -1)


def tree_target(inp: dict, tok: torch.Tensor, depth: torch.Tensor, n_nodes: torch.Tensor,
                target_dtype: int) -> torch.Tensor:
    """Target logits for every tree slot: [R, N+1, V] (slot c predicts c's child).

    Unused slots (c >= n_nodes[i]) get the root's row.
    """
    R, S = tok.shape
    dev = tok.device
    valid = torch.arange(S, device=dev).view(1, S) < n_nodes.view(R, 1).to(dev)
    t = torch.where(valid, tok, tok[:, :1]).to(torch.int32)
    dp = torch.where(valid, depth, torch.zeros_like(depth))
    req = torch.arange(R, device=dev).repeat_interleave(S)
    return target_rows(inp, req, dp.reshape(-1), t.reshape(-1), target_dtype).view(R, S, -1)


def gather_packed(target: torch.Tensor, packed_req: torch.Tensor, packed_pos: torch.Tensor,
                  out: torch.Tensor | None = None) -> torch.Tensor:
    """Stand-in for the target forward over the packed verify buffer.

    Copies row (packed_req[j], packed_pos[j]) of target [R, B+1, V] into packed
    row j; padding rows (req = -1) receive row 0.  Indices are clamped into
    range, so a buffer with unwritten tail entries cannot index out of bounds.
    """
    R, S, V = target.shape
    idx = packed_req.long().clamp(0, R - 1) * S + packed_pos.long().clamp(0, S - 1)
    flat = target.view(R * S, V)
    if out is None:
        return flat.index_select(0, idx)
    torch.index_select(flat, 0, idx, out=out[: idx.numel()])
    return out
