// tree_pruned.cu - a PCTree level without vocabulary-wide records.
//
// A level expands every frontier parent p (token y) of request i: its
// children are the top-k ids of z(y) = fp32(L_d) + U[y] . W by (z desc, id
// asc), scored s = s(p) + z - lse(y) ([PCTree] tree drafting: one Markov call
// for all frontier parents, local top-k, path log-probabilities, the P best
// kept).  Two quantities need the whole vocabulary, and they are split:
//   * lse(y): the Markov GEMM's MODE_TREE_LSE epilogue leaves one online
//     (max, sum) partial per frontier row, CTA and column group;
//   * the top-k: with |U[y] . W[:, v]| <= c(y) for every v (the prepared
//     tables), an id in the top k of z(y) has L_v >= L_(k) - 2 c(y), L_(k) the
//     k-th largest backbone logit of the row.  The scan of the cycle's start
//     (chain_pruned.cu, k-th mode) lists, per 32 KB chunk of each row, every id
//     with L >= theta - 2 c_max, theta a lower bound on the chunk's k-th
//     largest value, so the lists hold every chunk's top k (hence the row's top
//     k and L_(k)) and every id any parent can need.
// tree_level_kernel, one CTA per request:
//   1. (before the GEMM has finished) gathers the row's lists, finds L_(k),
//      keeps the ids with L >= L_(k) - 2 c_max and copies their W^T rows into
//      shared memory;
//   2. (after) the parents' U rows and log-sum-exps, then z for every (parent,
//      kept id) with L >= L_(k) - 2 c(y), exactly (fp32 products summed in
//      fp32: exact on the grid tables), the top k of each parent, the children's
//      scores and the per-level prune.
// A row whose lists overflowed, or whose kept ids do not fit, takes every
// parent's top k over the whole vocabulary from global memory instead
// (exhaustive; slow, but exact).
#include "device.cuh"
#include "internal.h"
#include "tree_common.cuh"

namespace sdm {
namespace {

constexpr int kLvThreads = 256;
constexpr int kLvWarps = kLvThreads / 32;
constexpr int kGather = 2048;    // listed entries of a row held in shared memory
constexpr int kStageCap = 192;   // kept ids (W^T rows staged)

struct LevelLayout {
    uint32_t w, u, g, z, cand, sorted, total;
    int rs;   // staged row stride (elements): r + 8 (16 bytes apart in the banks)
};

// Dynamic shared memory: staged W^T rows [kStageCap][rs] bf16, parents' U
// rows [P][rs] bf16, then the gathered list entries [kGather] (id, L bits),
// which the logits [P][kStageCap] fp32 reuse once the ids are staged, then the
// children [P k] and their rank order.
__host__ __device__ inline LevelLayout level_layout(int P, int k, int r) {
    LevelLayout l;
    l.rs = r + 8;
    const uint32_t row = 2u * static_cast<uint32_t>(l.rs);
    l.w = 0;
    l.u = l.w + static_cast<uint32_t>(kStageCap) * row;
    l.g = l.u + static_cast<uint32_t>(P) * row;
    const uint32_t gz = static_cast<uint32_t>(kGather) * 8u;
    const uint32_t zz = static_cast<uint32_t>(P) * kStageCap * 4u;
    l.z = l.g;
    l.cand = l.g + ((gz > zz ? gz : zz) + 15u) / 16u * 16u;
    l.sorted = l.cand + static_cast<uint32_t>(P * k) * 16u;
    l.total = l.sorted + static_cast<uint32_t>(P * k) * 16u;
    return l;
}

// Segment holding entry t of the row's concatenated lists.
__device__ __forceinline__ int list_of(const int* pref, int nc, int t) {
    int lo = 0, hi = nc - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (pref[mid] <= t)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

__device__ __forceinline__ float elem(const void* base, int fp32, size_t idx) {
    if (fp32) return static_cast<const float*>(base)[idx];
    return bf16_bits_to_float(static_cast<const uint16_t*>(base)[idx]);
}

// sum_j a[j] b[j] over r bf16 elements of two rows (shared or global memory,
// 16-byte aligned), fp32.
__device__ __forceinline__ float dot_rows(const uint16_t* a, const uint16_t* b, int r) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int q = 0; q < r; q += 8) {
        const uint4 x = *reinterpret_cast<const uint4*>(a + q);
        const uint4 y = *reinterpret_cast<const uint4*>(b + q);
        const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            acc[e] = fmaf(__uint_as_float(xs[e] << 16), __uint_as_float(ys[e] << 16), acc[e]);
            acc[e] = fmaf(__uint_as_float(xs[e] & 0xffff0000u), __uint_as_float(ys[e] & 0xffff0000u), acc[e]);
        }
    }
    return (acc[0] + acc[1]) + (acc[2] + acc[3]);
}

__device__ __forceinline__ unsigned long long block_max_u64(unsigned long long v, unsigned long long* red) {
    v = warp_max_u64(v);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    unsigned long long m = red[0];
#pragma unroll
    for (int w = 1; w < kLvWarps; ++w) m = umax64(m, red[w]);
    return m;
}

__global__ void __launch_bounds__(kLvThreads, 1) tree_level_kernel(const TreeLevelParams p) {
    extern __shared__ __align__(16) uint8_t s_dyn[];
    const LevelLayout lay = level_layout(p.P, p.k, p.r);
    const int RS = lay.rs;
    uint16_t* s_w = reinterpret_cast<uint16_t*>(s_dyn + lay.w);     // [kStageCap][RS]
    uint16_t* s_u = reinterpret_cast<uint16_t*>(s_dyn + lay.u);     // [P][RS]
    uint2* s_g = reinterpret_cast<uint2*>(s_dyn + lay.g);           // [kGather] (id, L bits)
    float* s_z = reinterpret_cast<float*>(s_dyn + lay.z);           // [P][kStageCap] (after staging)
    Cand* s_cand = reinterpret_cast<Cand*>(s_dyn + lay.cand);       // [P k]
    Cand* s_sorted = reinterpret_cast<Cand*>(s_dyn + lay.sorted);   // [P k]
    __shared__ int s_pref[kMaxPickChunks + 1];
    __shared__ uint2 s_keep[kStageCap];    // kept (id, L bits), in (L desc, id asc) order
    __shared__ int s_nkeep, s_exhaust, s_over;
    __shared__ float s_lk;                 // L_(k) of the row
    __shared__ int s_tok[kMaxTreeSlots], s_node[kMaxTreeSlots], s_cnt[kMaxTreeSlots];
    __shared__ float s_score[kMaxTreeSlots], s_lse[kMaxTreeSlots], s_thr[kMaxTreeSlots];
    __shared__ float2 s_top[kMaxTreeSlots][kMaxTopK];   // per parent: (z, id bits) in rank order
    __shared__ unsigned long long s_red[kLvWarps];
    const int i = blockIdx.x;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nc = p.n_chunks, P = p.P, K = p.k, r = p.r;
    const int seg0 = (i * p.B + (p.d - 1)) * nc;
    const float cmax = __ldcg(p.c_max);

    // 1. the row's lists (written by the scan at the cycle's start, not by the
    //    kernel this launch follows)
    if (warp == 0) {
        int run = 0, over = 0;
        for (int c0 = 0; c0 < nc; c0 += 32) {
            const int c = c0 + lane;
            int n = 0;
            if (c < nc) {
                const int cn = __ldcg(p.cand_n + seg0 + c);
                over |= cn > kSegCap;
                n = min(cn, kSegCap);
            }
            int x = n;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            if (c < nc) s_pref[c] = run + x - n;
            run += __shfl_sync(0xffffffffu, x, 31);
        }
        over = __any_sync(0xffffffffu, over);
        if (lane == 0) {
            s_pref[nc] = run;
            s_over = over;
            s_exhaust = over || run > kGather;
            s_nkeep = 0;
            s_lk = -INFINITY;
        }
    }
    __syncthreads();
    const int total = s_pref[nc];
    if (!s_exhaust) {
        for (int t = tid; t < total; t += kLvThreads) {
            const int c = list_of(s_pref, nc, t);
            s_g[t] = __ldcg(p.cand + static_cast<size_t>(seg0 + c) * kSegCap + (t - s_pref[c]));
        }
        __syncthreads();
        // L_(k): the entry with fewer than k entries above it and at least k
        // at or above it (the lists hold every chunk's top k, so the row's
        // top k are among them)
        for (int t = tid; t < total; t += kLvThreads) {
            const float x = __uint_as_float(s_g[t].y);
            int gt = 0, ge = 0;
            for (int u = 0; u < total; ++u) {
                const float y = __uint_as_float(s_g[u].y);
                gt += y > x ? 1 : 0;
                ge += y >= x ? 1 : 0;
            }
            if (gt < K && ge >= K) s_lk = x;   // one value, whoever writes it
        }
        __syncthreads();
        const float lk = s_lk;
        if (lk == -INFINITY) {
            if (tid == 0) s_exhaust = 1;       // fewer than k listed values
        } else {
            // the ids any parent can need: L >= L_(k) - 2 c_max
            const float tu = markov_cut(lk, cmax);
            for (int t = tid; t < total; t += kLvThreads) {
                const uint2 e = s_g[t];
                if (e.x < static_cast<uint32_t>(p.V) && __uint_as_float(e.y) >= tu) {
                    const int slot = atomicAdd(&s_nkeep, 1);
                    if (slot < kStageCap) s_keep[slot] = e;
                }
            }
        }
        __syncthreads();
        if (s_nkeep > kStageCap && tid == 0) s_exhaust = 1;
        __syncthreads();
        if (!s_exhaust) {
            // order the kept ids by (L desc, id asc): a parent's ids are then a prefix
            const int nk = s_nkeep;
            uint2 mine = make_uint2(0u, 0u);
            int rk = -1;
            if (tid < nk) {   // nk <= kStageCap < kLvThreads: one id per thread
                mine = s_keep[tid];
                const float x = __uint_as_float(mine.y);
                rk = 0;
                for (int u = 0; u < nk; ++u) {
                    const uint2 o = s_keep[u];
                    const float y = __uint_as_float(o.y);
                    rk += (y > x || (y == x && o.x < mine.x)) ? 1 : 0;
                }
            }
            __syncthreads();
            if (rk >= 0) s_keep[rk] = mine;
            __syncthreads();
            // their W^T rows into shared memory (16 bytes per lane)
            for (int j = warp; j < nk; j += kLvWarps) {
                const uint16_t* src = p.Wt + static_cast<size_t>(s_keep[j].x) * r;
                for (int q = lane * 8; q < r; q += 256) cp_async_16(s_w + static_cast<size_t>(j) * RS + q, src + q, 16u);
            }
        }
    }

    // 2. the parents, once the GEMM (and the level before it) has finished
    pdl_wait();
    pdl_trigger();
    const int nf = min(p.n_front[i], P);
    for (int f = tid; f < P; f += kLvThreads) {
        const size_t fr = static_cast<size_t>(i) * P + f;
        int t = f < nf ? p.front_tok[fr] : -1;
        if (t >= p.V) {
            set_status(p.dev_status, SDM_DEV_BAD_TOKEN);
            t = -1;
        }
        s_tok[f] = t;
        s_node[f] = p.front_node[fr];
        s_score[f] = p.front_score[fr];
        s_thr[f] = t >= 0 ? markov_cut(s_lk, p.c_bound[t]) : INFINITY;
    }
    __syncthreads();
    for (int f = warp; f < nf; f += kLvWarps) {
        const int t = s_tok[f];
        if (t >= 0)
            for (int q = lane * 8; q < r; q += 256)
                cp_async_16(s_u + static_cast<size_t>(f) * RS + q, p.U + static_cast<size_t>(t) * r + q, 16u);
        // lse of the parent's logits from the GEMM's partials: the largest
        // maximum, then every partial's sum rescaled to it (fp32 exponential,
        // fp64 sum)
        const float2* pr = p.part + (static_cast<size_t>(i) * P + f) * p.n_part;
        float m = -INFINITY;
        for (int q = lane; q < p.n_part; q += 32) {
            const float2 x = pr[q];
            if (x.y > 0.f) m = fmaxf(m, x.x);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        double sum = 0.0;
        for (int q = lane; q < p.n_part; q += 32) {
            const float2 x = pr[q];
            if (x.y > 0.f) sum += static_cast<double>(x.y * expf(x.x - m));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        if (lane == 0) s_lse[f] = static_cast<float>(static_cast<double>(m) + log(sum));
    }
    cp_async_wait_all();
    __syncthreads();

    if (!s_exhaust) {
        const int nk = s_nkeep;
        // each parent's ids: the kept prefix with L >= L_(k) - 2 c(y)
        for (int f = warp; f < nf; f += kLvWarps) {
            int n = 0;
            for (int j0 = 0; j0 < nk; j0 += 32) {
                const int j = j0 + lane;
                const bool in = j < nk && __uint_as_float(s_keep[j].y) >= s_thr[f];
                n += __popc(__ballot_sync(0xffffffffu, in));
            }
            if (lane == 0) s_cnt[f] = s_tok[f] >= 0 ? n : 0;
        }
        __syncthreads();
        // z for every (parent, id) pair: fp32(L) + U[y] . W^T[v]
        for (int t = tid; t < nf * nk; t += kLvThreads) {
            const int f = t / nk, j = t - f * nk;
            if (j < s_cnt[f])
                s_z[f * kStageCap + j] = __uint_as_float(s_keep[j].y) +
                                         dot_rows(s_u + static_cast<size_t>(f) * RS, s_w + static_cast<size_t>(j) * RS, r);
        }
        __syncthreads();
        // each parent's top k by (z desc, id asc)
        for (int t = tid; t < nf * nk; t += kLvThreads) {
            const int f = t / nk, j = t - f * nk;
            const int n = s_cnt[f];
            if (j >= n) continue;
            const unsigned long long me = argmax_key(s_z[f * kStageCap + j], s_keep[j].x);
            int rk = 0;
            for (int u = 0; u < n && rk < K; ++u)
                rk += argmax_key(s_z[f * kStageCap + u], s_keep[u].x) > me ? 1 : 0;
            if (rk < K) s_top[f][rk] = make_float2(s_z[f * kStageCap + j], __int_as_float(static_cast<int>(s_keep[j].x)));
        }
    } else {
        // every id of the vocabulary for every parent, W^T rows from global
        // memory; per thread a sorted list of its k best keys, then k rounds
        // of the block maximum
        const size_t lrow = (static_cast<size_t>(i) * p.B + (p.d - 1)) * p.V;
        for (int f = 0; f < nf; ++f) {
            if (s_tok[f] < 0) continue;
            unsigned long long best[kMaxTopK];
#pragma unroll
            for (int q = 0; q < kMaxTopK; ++q) best[q] = 0ull;
            const uint16_t* urow = s_u + static_cast<size_t>(f) * RS;
            for (int v = tid; v < p.V; v += kLvThreads) {
                const float z = elem(p.L, p.l_fp32, lrow + v) + dot_rows(urow, p.Wt + static_cast<size_t>(v) * r, r);
                unsigned long long key = argmax_key(z, static_cast<uint32_t>(v));
#pragma unroll
                for (int q = 0; q < kMaxTopK; ++q) {   // insert, keeping the list sorted
                    if (q < K && key > best[q]) {
                        const unsigned long long t2 = best[q];
                        best[q] = key;
                        key = t2;
                    }
                }
            }
            int head = 0;
            for (int q = 0; q < K; ++q) {
                unsigned long long mine = 0ull;
#pragma unroll
                for (int e = 0; e < kMaxTopK; ++e)
                    if (e == head) mine = best[e];
                const unsigned long long m = block_max_u64(mine, s_red);
                if (mine == m && m != 0ull) ++head;   // keys are distinct (ids differ)
                if (tid == 0) s_top[f][q] = make_float2(key_value(m), __int_as_float(static_cast<int>(key_token(m))));
            }
        }
    }
    __syncthreads();
    // children s = s(p) + (z - lse(p)), the P best kept
    const int ncand = nf * K;
    for (int t = tid; t < ncand; t += kLvThreads) {
        const int f = t / K, q = t - f * K;
        const float2 e = s_top[f][q];
        s_cand[t] = s_tok[f] >= 0 ? Cand{s_score[f] + (e.x - s_lse[f]), f, q, __float_as_int(e.y)}
                                  : Cand{-INFINITY, f, q, -1};
    }
    __syncthreads();
    tree_keep_children(i, P, p.B, p.d, ncand, s_cand, s_sorted, s_node, p.pool_n[i], p.front_tok, p.front_node,
                       p.front_score, p.n_front, p.pool_tok, p.pool_parent, p.pool_depth, p.pool_score, p.pool_n);
}

}  // namespace

size_t tree_level_smem(int P, int k, int r) { return level_layout(P, k, r).total; }

cudaError_t launch_tree_level(const TreeLevelParams& p, cudaStream_t s) {
    if (p.P > kMaxTreeSlots || p.k > kMaxTopK || p.n_chunks > kMaxPickChunks) return cudaErrorInvalidValue;
    const size_t smem = tree_level_smem(p.P, p.k, p.r);
    static size_t configured = 0;   // the dynamic shared memory allowed so far
    if (smem > configured) {
        const cudaError_t e =
            cudaFuncSetAttribute(tree_level_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        configured = smem;
    }
    return launch_pdl(tree_level_kernel, dim3(p.R), dim3(kLvThreads), smem, s, p);
}

}  // namespace sdm
