"""The five synthetic workloads of the DSpark / PCTree hot path, as data.

Each entry fixes the shapes and the value distributions of one workload.
Sources: the DSpark study notes (LayerX, 2026-06-30) for the chain drafter,
the scheduler and verification; the Qiita PCTree article for the tree
workload; "DSpark in SGLang" (winzheng.jp) for the mixed-traffic workload,
its additive step-cost table, ragged tiers and verify modes.

Readings fixed here (the pages leave them open):
  * "N(mu, x)" gives the standard deviation x, except the Markov tables
    U, W ~ N(0, 1/r), read as variance 1/r (std r^-1/2, fan-in scaling).
  * Confidences of the chain workloads are sigmoid(N(1, 1)); the mixed-traffic
    workload uses the soft acceptance label 1 - TV(q, p) of the notes'
    confidence-head section, computed between the backbone distribution and
    the noisy target at that position.
  * The target LLM is replaced by T_d(prev) = L_d + U[prev] W + eta_d, i.e.
    "draft logits plus noise" along any drafted prefix.
  * Seed 0 everywhere; the additive table 2.0 + 0.004 N (ms) and the tiers
    {64, ..., 2048} are reused where a workload names none (the two batches
    of 256 requests add 4096 and 8192, so that their totals fall in a tier).
"""
from __future__ import annotations

from dataclasses import dataclass, field

BF16 = 0
FP32 = 1

TIERS = (64, 128, 256, 512, 1024, 2048)
# batches of 256 requests verify up to 256 (gamma + 1) rows: two more tiers
TIERS_LARGE = TIERS + (4096, 8192)


@dataclass(frozen=True)
class Workload:
    name: str
    R: int                      # requests in the batch
    B: int                      # draft block length (gamma)
    V: int                      # vocabulary size
    r: int                      # Markov rank
    l_dtype: int                # dtype of the backbone logits L
    l_std: float                # std of L
    sigma: tuple                # per-class target-noise std
    target_dtype: int           # dtype of the target logits
    decode: str = "greedy"      # "greedy" | "sample" | "tree"
    modes: tuple = ("compact",)
    temperature: float = 1.0
    conf: str = "sigmoid"       # "sigmoid" | "one_minus_tv"
    cost: tuple = (2.0, 0.004)  # additive step cost a + b N (ms)
    tiers: tuple = TIERS
    P: int = 0                  # PCTree frontier width
    k: int = 0                  # PCTree local top-k
    N: int = 0                  # PCTree node budget (root excluded)
    class_mix: str = "alternate"  # how sigma classes are assigned to requests
    extra: dict = field(default_factory=dict)


WORKLOADS = {
    "tiny_chain": Workload(
        name="tiny_chain", R=4, B=7, V=1024, r=64, l_dtype=FP32, l_std=1.0,
        sigma=(0.5,), target_dtype=FP32, decode="greedy", modes=("compact",),
        conf="sigmoid", cost=(1.0, 0.05)),
    "qwen3_8b_chain": Workload(
        name="qwen3_8b_chain", R=64, B=7, V=151936, r=256, l_dtype=BF16, l_std=2.0,
        sigma=(0.3, 1.0), target_dtype=BF16, decode="greedy", modes=("compact",),
        conf="sigmoid", cost=(2.0, 0.004)),
    "rejection_sampling": Workload(
        name="rejection_sampling", R=256, B=16, V=151936, r=256, l_dtype=BF16, l_std=2.0,
        sigma=(0.7,), target_dtype=FP32, decode="sample", modes=("static",),
        temperature=1.0, conf="sigmoid", tiers=TIERS_LARGE),
    "pctree": Workload(
        name="pctree", R=32, B=16, V=151936, r=256, l_dtype=BF16, l_std=2.0,
        sigma=(0.5,), target_dtype=BF16, decode="tree", modes=("tree",),
        P=8, k=4, N=64),
    "mixed_traffic": Workload(
        name="mixed_traffic", R=256, B=8, V=129280, r=256, l_dtype=BF16, l_std=2.0,
        sigma=(0.2, 0.8, 1.5), target_dtype=BF16, decode="greedy",
        modes=("static", "compact", "cap_accept"), conf="one_minus_tv",
        cost=(2.0, 0.004), class_mix="shuffle", tiers=TIERS_LARGE),
}

# the order the workloads are listed in (the second is the headline one)
ORDER = ("tiny_chain", "qwen3_8b_chain", "rejection_sampling", "pctree", "mixed_traffic")


def scaled(w: Workload, **changes) -> Workload:
    """A copy of workload w with some fields replaced (smaller test shapes)."""
    d = dict(w.__dict__)
    d.update(changes)
    return Workload(**d)
