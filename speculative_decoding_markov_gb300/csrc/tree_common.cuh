// tree_common.cuh - the per-level prune of PCTree ([PCTree] tree drafting:
// every frontier parent's top-k children get the path score s(c) = s(p) +
// log pi(v | p); the P best children of the level are kept), shared by the
// record-based and the bound-pruned level kernels.
#pragma once
#include "device.cuh"
#include "internal.h"

namespace sdm {

struct Cand {
    float s;
    int slot, rank, tok;
};

// (s desc, slot asc, rank asc), with s compared through its order-preserving
// bits: a strict total order even when a score is NaN, so that parallel ranks
// form a permutation.
__device__ __forceinline__ bool cand_before(const Cand& a, const Cand& b) {
    const uint32_t oa = ordered_bits(a.s), ob = ordered_bits(b.s);
    if (oa != ob) return oa > ob;
    if (a.slot != b.slot) return a.slot < b.slot;
    return a.rank < b.rank;
}

// Request i's nc children in cand[] (shared memory; every thread of the CTA
// calls this): ranked in parallel into sorted[], the best P become level d's
// pool nodes and the next frontier.  parent_node[f] = the pool node of
// frontier slot f; np = the pool's size before the level.
__device__ __forceinline__ void tree_keep_children(int i, int P, int B, int d, int nc, const Cand* cand, Cand* sorted,
                                                   const int* parent_node, int np, int32_t* front_tok,
                                                   int32_t* front_node, float* front_score, int32_t* n_front,
                                                   int32_t* pool_tok, int32_t* pool_parent, int32_t* pool_depth,
                                                   float* pool_score, int32_t* pool_n) {
    // a child's rank = the children before it, four threads per child each
    // counting a quarter (blockDim is a multiple of 32: every lane of a warp
    // runs each round)
    for (int t0 = 0; t0 < 4 * nc; t0 += blockDim.x) {
        const int t = t0 + static_cast<int>(threadIdx.x);
        const int c = t >> 2;
        int rk = 0;
        Cand me{};
        if (c < nc) {
            me = cand[c];
            for (int u = t & 3; u < nc; u += 4) rk += cand_before(cand[u], me) ? 1 : 0;
        }
        rk += __shfl_xor_sync(0xffffffffu, rk, 1);
        rk += __shfl_xor_sync(0xffffffffu, rk, 2);
        if (c < nc && (t & 3) == 0) sorted[rk] = me;
    }
    __syncthreads();
    const int keep = nc < P ? nc : P;
    const int pool_cap = 1 + P * B;
    const size_t pb = static_cast<size_t>(i) * pool_cap;
    for (int c = threadIdx.x; c < P; c += blockDim.x) {
        const size_t fo = static_cast<size_t>(i) * P + c;
        if (c < keep) {
            const Cand cd = sorted[c];
            pool_tok[pb + np + c] = cd.tok;
            pool_parent[pb + np + c] = parent_node[cd.slot];
            pool_depth[pb + np + c] = d;
            pool_score[pb + np + c] = cd.s;
            front_tok[fo] = cd.tok;
            front_node[fo] = np + c;
            front_score[fo] = cd.s;
        } else {
            front_tok[fo] = -1;
            front_node[fo] = -1;
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        n_front[i] = keep;
        pool_n[i] = np + keep;
    }
}

}  // namespace sdm
