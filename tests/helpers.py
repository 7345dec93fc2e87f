"""Shared test helpers: array conversion and the multi-cycle decode drivers."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from speculative_decoding_markov_gb300 import synthetic
from speculative_decoding_markov_gb300.workloads import BF16, FP32, Workload


def np_of(t: torch.Tensor) -> np.ndarray:
    """Tensor -> numpy on the host; bf16 becomes its uint16 bit pattern."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def small(R=3, B=4, V=48, r=16, l_dtype=FP32, target_dtype=FP32, sigma=(0.5,), **kw) -> Workload:
    return Workload(name="small", R=R, B=B, V=V, r=r, l_dtype=l_dtype, l_std=kw.pop("l_std", 1.0),
                    sigma=sigma, target_dtype=target_dtype, **kw)


# ---------------------------------------------------------------------------
# absolute-position inputs for multi-cycle decoding
# ---------------------------------------------------------------------------
def absolute_inputs(w: Workload, positions: int, seed: int = 0) -> dict:
    """Backbone rows and target noise for absolute positions 1..positions.

    L_abs[i, q] predicts the token at absolute position q+1; eta_abs[i, q] is
    the target noise there.  Generated as one long 'block' of the workload.
    """
    big = Workload(**{**w.__dict__, "B": positions})
    inp = synthetic.generate(big, seed=seed)
    return dict(L_abs=inp["L"], eta_abs=inp["eta"][:, :positions], U=inp["U"], W=inp["W"],
                anchor=inp["anchor"], conf_abs=inp["conf"], cost=synthetic.cost_table(w))


def cycle_inputs(ab: dict, pos: np.ndarray, B: int) -> dict:
    """The per-cycle input dict seen by a cycle whose anchors sit at `pos`."""
    R = pos.shape[0]
    idx = torch.as_tensor(pos, dtype=torch.long).view(R, 1) + torch.arange(B).view(1, B)
    ar = torch.arange(R).view(R, 1)
    L = ab["L_abs"][ar, idx]
    eidx = torch.as_tensor(pos, dtype=torch.long).view(R, 1) + torch.arange(B + 1).view(1, B + 1)
    eta = ab["eta_abs"][ar, eidx]
    Lb = ab["L_abs"][torch.arange(R), torch.as_tensor(pos, dtype=torch.long) + B]
    conf = ab["conf_abs"][ar, idx]
    return dict(L=L, L_bonus=Lb, U=ab["U"], W=ab["W"], eta=eta, conf=conf)


def target_only_greedy(ab: dict, n_tokens: int, target_dtype: int) -> np.ndarray:
    """t_0 = anchor, t_{q+1} = argmax_v T_{q+1}(t_q) (lowest id on ties)."""
    R = ab["anchor"].shape[0]
    seq = np.zeros((R, n_tokens + 1), np.int64)
    seq[:, 0] = ab["anchor"].numpy()
    inp = dict(L=ab["L_abs"], L_bonus=ab["L_abs"][:, -1], U=ab["U"], W=ab["W"], eta=ab["eta_abs"])
    for q in range(n_tokens):
        rows = synthetic.target_rows(inp, torch.arange(R), torch.full((R,), q), torch.as_tensor(seq[:, q]),
                                     target_dtype)
        seq[:, q + 1] = torch.argmax(rows.float(), dim=1).numpy()   # first maximal index
    return seq


def oracle_greedy_decode(w: Workload, ab: dict, cycles: int, mode: str = "compact", gamma=None):
    """Runs `cycles` speculative cycles through the oracle (greedy decode).

    Returns the committed sequences (anchor first) and per-cycle records.
    """
    B = w.B if gamma is None else gamma
    R = ab["anchor"].shape[0]
    pos = np.zeros(R, np.int64)
    anchor = ab["anchor"].numpy().astype(np.int32)
    seqs = [[int(a)] for a in anchor]
    records = []
    U, W = np_of(ab["U"]), np_of(ab["W"])
    for _ in range(cycles):
        ci = cycle_inputs(ab, pos, B)
        dr = oracle.draft_chain(np_of(ci["L"]), U, W, anchor)
        sc = oracle.schedule_budget(np_of(ci["conf"]), synthetic.cost_table(w, R=R, B=B).numpy())
        budget = None if mode == "static" else sc["budget"]
        pk = oracle.pack_ragged(anchor, dr["tokens"], budget, np.array(w.tiers, np.int32))
        tgt = synthetic.chain_target(ci | {"anchor": torch.as_tensor(anchor)}, torch.as_tensor(dr["tokens"]),
                                     w.target_dtype)
        packed = synthetic.gather_packed(tgt, torch.as_tensor(pk["packed_req"]), torch.as_tensor(pk["packed_pos"]))
        omode = {"static": oracle.STATIC, "compact": oracle.COMPACT}[mode]
        vr = oracle.verify(omode, oracle.GREEDY, np_of(packed), pk["cu_seqlens"], anchor, dr["tokens"])
        for i in range(R):
            seqs[i].extend(int(t) for t in vr["out_tok"][i, : vr["n_out"][i]])
        pos = pos + vr["n_out"]
        anchor = np.array([s[-1] for s in seqs], np.int32)
        records.append(dict(draft=dr, sched=sc, pack=pk, verify=vr))
    return seqs, records


# ---------------------------------------------------------------------------
# tie-zone events, localised to the first decision that differs
# ---------------------------------------------------------------------------
def verify_first_decision(ref: dict, j: int, accept: int, ceiling: int, out_tok: np.ndarray):
    """For request j of an oracle verify result, the (position, margin) of
    the first decision on which a GPU result (accept, ceiling, out_tok)
    differs, or None when it agrees.  The accept tests run left to right, so
    two ceilings first part at the test of row min(ceilings); equal ceilings
    with a different final token part at the final draw (margin column
    gamma)."""
    g = ref["margin"].shape[1] - 1
    if ceiling != ref["ceiling"][j]:
        p = int(min(ceiling, ref["ceiling"][j]))
        return p, float(ref["margin"][j, p])
    if accept != ref["accept"][j] or not np.array_equal(out_tok, ref["out_tok"][j]):
        return g, float(ref["margin"][j, g])
    return None


def tree_paths(tok: np.ndarray, parent: np.ndarray, depth: np.ndarray, n: int) -> dict:
    """depth -> set of the token paths (root excluded) of the tree's nodes."""
    out = {}
    for c in range(1, n):
        path, a = [], c
        while a > 0:
            path.append(int(tok[a]))
            a = int(parent[a])
        out.setdefault(int(depth[c]), set()).add(tuple(reversed(path)))
    return out


def tree_first_decision(ref: dict, j: int, tok, parent, depth, n_nodes: int, B: int):
    """For request j of an oracle tree, the (kind, margin) of the first
    decision on which a GPU tree differs, or None when it agrees: the first
    depth whose set of nodes differs (its level's prune boundary, or the
    top-N boundary, whichever is closer), else the order of the output
    ranking."""
    same = all(np.array_equal(a, ref[k][j]) for a, k in ((tok, "tok"), (parent, "parent"), (depth, "depth")))
    if same and n_nodes == ref["n_nodes"][j]:
        return None
    gp = tree_paths(tok, parent, depth, n_nodes)
    rp = tree_paths(ref["tok"][j], ref["parent"][j], ref["depth"][j], int(ref["n_nodes"][j]))
    for d in range(1, B + 1):
        if gp.get(d, set()) != rp.get(d, set()):
            return f"level {d}", float(min(ref["margin"][j, d - 1], ref["margin"][j, B]))
    return "ranking", float(ref["margin"][j, B + 1])


def oracle_threads() -> int:
    """Host cores this process may run on (the oracle's calls release the GIL)."""
    import os

    return max(1, len(os.sched_getaffinity(0)))


def oracle_map(fn, items):
    """fn over items on a thread pool: each call is one single-threaded
    oracle call (ctypes releases the GIL), results in order."""
    from concurrent.futures import ThreadPoolExecutor

    items = list(items)
    if len(items) <= 1:
        return [fn(x) for x in items]
    with ThreadPoolExecutor(max_workers=min(len(items), oracle_threads())) as ex:
        return list(ex.map(fn, items))
