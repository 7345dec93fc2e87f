// small.cu - the latency-bound kernels of the cycle: greedy chain finalisation,
// the prefix scheduler, the ragged pack, the per-request verification scans,
// and PCTree's per-level merge/prune and final top-N selection.
#include "device.cuh"
#include "internal.h"
#include "schedule_pack.cuh"
#include "tree_common.cuh"
#include "verify_greedy.cuh"

namespace sdm {
namespace {

__device__ __forceinline__ float load_elem(const void* base, int fp32, size_t idx) {
    if (fp32) return static_cast<const float*>(base)[idx];
    return bf16_bits_to_float(static_cast<const uint16_t*>(base)[idx]);
}

// ---------------------------------------------------------------------------
__global__ void fill_u64_kernel(unsigned long long* p, size_t n, unsigned long long v) {
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<size_t>(gridDim.x) * blockDim.x)
        p[i] = v;
}

// ---------------------------------------------------------------------------
// greedy chain finalize: tokens [R, B] from the argmax keys [B][R]
// ---------------------------------------------------------------------------
__global__ void chain_finalize_kernel(const unsigned long long* keys, int R, int B, int V, int32_t* tokens,
                                      int32_t* dev_status) {
    const int idx = blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= R * B) return;
    const int i = idx / B, d = idx % B + 1;
    int y = static_cast<int>(key_token(keys[static_cast<size_t>(d - 1) * R + i]));
    if (y < 0 || y >= V) {
        set_status(dev_status, SDM_DEV_BAD_TOKEN);
        y = 0;
    }
    tokens[idx] = y;
}

// ---------------------------------------------------------------------------
// scheduler: one CTA
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kSchedThreads) schedule_kernel(const float* conf, int R, int gamma,
                                                                 const double* cost, float* survival,
                                                                 int32_t* budget, double* expected,
                                                                 int32_t* total_tokens, int n_pad) {
    extern __shared__ unsigned long long sk[];
    pdl_wait();
    pdl_trigger();
    schedule_block(conf, R, gamma, cost, survival, budget, expected, total_tokens, n_pad, sk, kSchedThreads);
}

// ---------------------------------------------------------------------------
// production scheduler ([DSpark notes] sec. 9.2): capacity K from the
// confidences of two steps before by a global search over the cost table,
// then the top K of this step's survivals.  One CTA, the same survival keys,
// floor and bitonic sort as schedule_kernel.
// ---------------------------------------------------------------------------
// Survivals of conf (fp32 products, left to right) as descending sort keys
// (S bits, then ~(i * gamma + k): request asc, position asc), those below the
// floor as 0; writes the survivals to surv_out when not NULL.  Returns the
// number of keys above the floor (all threads).
__device__ int ranked_keys(const float* conf, int R, int gamma, float* s_surv, unsigned long long* sk, int n_pad,
                           float* surv_out, int* s_count) {
    const int tid = threadIdx.x, nt = blockDim.x;
    const int n = R * gamma;
    const float floor_s = 1.0f / 262144.0f;
    for (int t = tid; t < n; t += nt) s_surv[t] = conf[t];
    for (int t = n + tid; t < n_pad; t += nt) sk[t] = 0ull;
    if (tid == 0) *s_count = 0;
    __syncthreads();
    for (int i = tid; i < R; i += nt) {
        float s = 1.0f;
        for (int k = 0; k < gamma; ++k) {
            const int t = i * gamma + k;
            s = __fmul_rn(s, s_surv[t]);
            s_surv[t] = s;
            sk[t] = (s >= floor_s) ? ((static_cast<unsigned long long>(__float_as_uint(s)) << 32) | ~static_cast<uint32_t>(t))
                                   : 0ull;
        }
    }
    __syncthreads();
    if (surv_out)
        for (int t = tid; t < n; t += nt) surv_out[t] = s_surv[t];
    for (int size = 2; size <= n_pad; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int t = tid; t < n_pad; t += nt) {
                const int u = t ^ stride;
                if (u > t) {
                    const bool desc = (t & size) == 0;
                    const unsigned long long a = sk[t], b = sk[u];
                    if (desc ? (a < b) : (a > b)) {
                        sk[t] = b;
                        sk[u] = a;
                    }
                }
            }
            __syncthreads();
        }
    }
    for (int t = tid; t < n_pad; t += nt)
        if (sk[t] != 0ull && (t + 1 == n_pad || sk[t + 1] == 0ull)) *s_count = t + 1;
    __syncthreads();
    return *s_count;
}

// A ranked survival as an exact integer (every survival >= 2^-18 is a
// multiple of 2^-41).
__device__ __forceinline__ unsigned long long surv_units(unsigned long long key) {
    return static_cast<unsigned long long>(ldexpf(__uint_as_float(static_cast<uint32_t>(key >> 32)), 41));
}

__global__ void __launch_bounds__(kSchedThreads) schedule_dynamic_kernel(const float* conf, const float* conf_stale,
                                                                         int R, int gamma, const double* cost,
                                                                         float* survival, int32_t* budget,
                                                                         double* expected, int32_t* total_tokens,
                                                                         int32_t* capacity, int n_pad) {
    extern __shared__ unsigned long long sk[];              // n_pad sort keys
    unsigned long long* part = sk + n_pad;                   // kSchedThreads exclusive prefixes
    int* cnt = reinterpret_cast<int*>(part + kSchedThreads);  // R counters
    float* s_surv = reinterpret_cast<float*>(cnt + R);       // R * gamma confidences, then survivals
    __shared__ int s_count;
    __shared__ unsigned long long best_bits;
    __shared__ int best_m;
    __shared__ unsigned long long sum_units;
    pdl_wait();
    pdl_trigger();
    const int tid = threadIdx.x, nt = blockDim.x;
    const int per = (n_pad + 1 + nt - 1) / nt;   // m = 0 .. n_pad
    // 1. capacity from the stale confidences: f(m) = E'(m) / cost[R + m] for
    //    every m (E' exact in units of 2^-41, one IEEE fp64 division each, as
    //    in the oracle), the largest f, the smallest m among equals
    const int Ms = ranked_keys(conf_stale, R, gamma, s_surv, sk, n_pad, nullptr, &s_count);
    unsigned long long local = 0;
    for (int q = 0; q < per; ++q) {
        const int t = tid * per + q;
        if (t < Ms) local += surv_units(sk[t]);
    }
    {   // exclusive block scan of the thread partials (integer: exact in any order)
        const int lane = tid & 31, warp = tid >> 5;
        unsigned long long x = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) part[warp] = x;
        if (tid == 0) {
            best_bits = 0ull;
            best_m = 0x7fffffff;
            sum_units = 0ull;
        }
        __syncthreads();
        if (warp == 0) {
            unsigned long long wv = lane < (nt >> 5) ? part[lane] : 0ull;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned long long y = __shfl_up_sync(0xffffffffu, wv, o);
                if (lane >= o) wv += y;
            }
            part[lane] = wv;
        }
        __syncthreads();
        const unsigned long long before = (warp > 0 ? part[warp - 1] : 0ull) + x - local;
        __syncthreads();
        part[tid] = before;
    }
    __syncthreads();
    const double two_m41 = 4.547473508864641e-13;   // 2^-41
    const unsigned long long base = static_cast<unsigned long long>(R) << 41;
    double fbest = -1.0;
    int mbest = 0x7fffffff;
    {
        unsigned long long run = part[tid];
        for (int q = 0; q < per; ++q) {
            const int m = tid * per + q;   // E'(m) uses the first m survivals
            if (m > Ms) break;
            const double f = __ddiv_rn(static_cast<double>(base + run) * two_m41, cost[R + m]);
            if (f > fbest) {               // m rises: the first of equal values stays
                fbest = f;
                mbest = m;
            }
            if (m < Ms) run += surv_units(sk[m]);
        }
    }
    if (mbest != 0x7fffffff) atomicMax(&best_bits, static_cast<unsigned long long>(__double_as_longlong(fbest)));
    __syncthreads();   // (f > 0: the bits of positive doubles order like their values)
    if (mbest != 0x7fffffff && static_cast<unsigned long long>(__double_as_longlong(fbest)) == best_bits)
        atomicMin(&best_m, mbest);
    __syncthreads();
    const int K = best_m == 0x7fffffff ? 0 : best_m;
    // 2. this step's survivals, ranked; the top min(K, available) are verified
    const int Mn = ranked_keys(conf, R, gamma, s_surv, sk, n_pad, survival, &s_count);
    const int take = K < Mn ? K : Mn;
    for (int i = tid; i < R; i += nt) cnt[i] = 0;
    __syncthreads();
    unsigned long long mine = 0;
    for (int t = tid; t < take; t += nt) {
        const uint32_t id = ~static_cast<uint32_t>(sk[t] & 0xffffffffull);
        atomicAdd(&cnt[id / gamma], 1);
        mine += surv_units(sk[t]);
    }
    atomicAdd(&sum_units, mine);
    __syncthreads();
    for (int i = tid; i < R; i += nt) budget[i] = cnt[i];
    if (tid == 0) {
        *expected = static_cast<double>(base + sum_units) * two_m41;
        *total_tokens = R + take;
        *capacity = K;
    }
}

// ---------------------------------------------------------------------------
// ragged pack: one CTA
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kPackThreads) pack_kernel(const int32_t* anchor, const int32_t* draft,
                                                            const int32_t* budget, int R, int gamma,
                                                            const int32_t* tiers, int n_tiers, int strict, int32_t* cu,
                                                            int32_t* ptok, int32_t* preq, int32_t* ppos,
                                                            int capacity, int32_t* tier, int32_t* dev_status) {
    pdl_wait();
    pdl_trigger();
    pack_block(anchor, draft, budget, R, gamma, tiers, n_tiers, strict, cu, ptok, preq, ppos, capacity, tier,
               dev_status);
}

// ---------------------------------------------------------------------------
// greedy verification: first mismatch per request
// ---------------------------------------------------------------------------
__global__ void verify_greedy_finalize_kernel(int mode, const int32_t* cu, const int32_t* draft,
                                              const int32_t* budget, const unsigned long long* row_keys, int n_chunks,
                                              int R, int gamma, int V, int rows_avail, int32_t* accept,
                                              int32_t* ceiling, int32_t* out_tok, int32_t* n_out,
                                              int32_t* dev_status) {
    // one warp per request: lane p resolves window rows p, p + 32, ...
    pdl_wait();
    pdl_trigger();
    const int i = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (i >= R) return;
    greedy_resolve(i, lane, mode, cu, draft, budget, row_keys, n_chunks, gamma, V, rows_avail, cu[R], accept, ceiling,
                   out_tok, n_out, dev_status);
}

// ---------------------------------------------------------------------------
// rejection sampling: accept scan per request
// ---------------------------------------------------------------------------
__global__ void verify_sample_scan_kernel(int mode, const int32_t* cu, const int32_t* anchor, const int32_t* draft,
                                          const int32_t* budget, const float* logq, const void* target, int t_fp32,
                                          int V, const float2* lse_part, int n_chunks, float inv_t, uint32_t k0,
                                          uint32_t k1, uint32_t cycle, int R, int gamma, int32_t* accept,
                                          int32_t* ceiling, int32_t* res_tok, int32_t* res_pos, int32_t* res_trow,
                                          float* res_lse_p, int32_t* bonus_row, int32_t* bonus_pos,
                                          int rows_avail, int32_t* dev_status) {
    // one warp per request; lane p runs the accept test of window row p (all
    // rows at once, each from its own partials), the first failure wins
    pdl_wait();
    pdl_trigger();
    const int i = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (i >= R) return;
    const RngKey rk{k0, k1, cycle};
    const int row0 = cu[i];
    const int row1 = cu[i + 1];
    // the log-sum-exp stream wrote partials for rows below min(cu[R],
    // rows_avail) only
    if (row1 <= row0 || row0 < 0 || row1 > rows_avail || row1 > cu[R]) {
        // no rows, rows past the packed buffer or past cu[R]: flagged, and
        // neither a residual nor a bonus draw (the resample kernel commits
        // token 0)
        if (lane == 0) {
            set_status(dev_status, row1 > rows_avail ? SDM_DEV_CAPACITY : SDM_DEV_BAD_WINDOW);
            accept[i] = 0;
            if (ceiling) ceiling[i] = 0;
            res_tok[i] = -1;
            res_pos[i] = 0;
            res_trow[i] = 0;
            res_lse_p[i] = 0.f;
            bonus_row[i] = -1;
            bonus_pos[i] = 0;
        }
        return;
    }
    int w = row1 - row0 - 1;
    if (w > gamma) {
        if (lane == 0) set_status(dev_status, SDM_DEV_BAD_WINDOW);
        w = gamma;
    }
    int cap = w;
    if (mode == SDM_CAP_ACCEPT) {
        cap = budget[i];
        if (cap < 0 || cap > w) {
            if (lane == 0) set_status(dev_status, SDM_DEV_BAD_WINDOW);
            cap = cap < 0 ? 0 : w;
        }
    }
    const int32_t* y = draft + static_cast<size_t>(i) * gamma;
    auto row_lse = [&](int p) {
        Lse acc{-INFINITY, 0.f};
        const float2* pp = lse_part + static_cast<size_t>(row0 + p) * n_chunks;
        for (int c = 0; c < n_chunks; ++c) acc = lse_merge(acc, Lse{pp[c].x, pp[c].y});
        return acc.m + logf(acc.s);
    };
    int A = w;
    for (int p0 = 0; p0 < w && A == w; p0 += 32) {
        const int p = p0 + lane;
        bool reject = false;
        if (p < w) {
            int yp = y[p];
            if (yp < 0 || yp >= V) {
                set_status(dev_status, SDM_DEV_BAD_TOKEN);
                yp = 0;
            }
            const float lp = load_elem(target, t_fp32, static_cast<size_t>(row0 + p) * V + yp) * inv_t - row_lse(p);
            const float lq = logq[static_cast<size_t>(i) * gamma + p];
            const float u = uniform_at(rk, 1u, static_cast<uint32_t>(i), static_cast<uint32_t>(p), 0u);
            reject = !(logf(u) < lp - lq);   // accept iff u < p(y) / q(y)
        }
        const unsigned bal = __ballot_sync(0xffffffffu, reject);
        if (bal) A = p0 + __ffs(bal) - 1;
    }
    if (lane != 0) return;
    const int a = A < cap ? A : cap;
    accept[i] = a;
    if (ceiling) ceiling[i] = A;
    if (A < cap) {   // rejected at row a: residual from max(0, p - q)
        res_tok[i] = (a == 0) ? anchor[i] : y[a - 1];
        res_pos[i] = a;
        res_trow[i] = row0 + a;
        res_lse_p[i] = row_lse(a);
        bonus_row[i] = -1;
        bonus_pos[i] = 0;
    } else {         // every committed draft passed: bonus from p at row a
        res_tok[i] = -1;
        res_pos[i] = 0;
        res_trow[i] = 0;
        res_lse_p[i] = 0.f;
        bonus_row[i] = row0 + a;
        bonus_pos[i] = a;
    }
}

// ---------------------------------------------------------------------------
// PCTree
// ---------------------------------------------------------------------------
__global__ void tree_init_kernel(const int32_t* anchor, int R, int P, int B, int32_t* front_tok, int32_t* front_node,
                                 float* front_score, int32_t* n_front, int32_t* pool_tok, int32_t* pool_parent,
                                 int32_t* pool_depth, float* pool_score, int32_t* pool_n, int32_t* dev_status) {
    pdl_wait();
    pdl_trigger();
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= R) return;
    const int pool_cap = 1 + P * B;
    const size_t pb = static_cast<size_t>(i) * pool_cap;
    pool_tok[pb] = anchor[i];
    pool_parent[pb] = -1;
    pool_depth[pb] = 0;
    pool_score[pb] = 0.f;
    pool_n[i] = 1;
    for (int s = 0; s < P; ++s) {
        front_tok[static_cast<size_t>(i) * P + s] = (s == 0) ? anchor[i] : -1;
        front_node[static_cast<size_t>(i) * P + s] = (s == 0) ? 0 : -1;
        front_score[static_cast<size_t>(i) * P + s] = 0.f;
    }
    n_front[i] = 1;
}

// One CTA per request: the children of every frontier slot (its top-k by z,
// from the level's select kernel) get s(c) = s(p) + z - lse; they are ranked
// in parallel and the best P kept.
__global__ void tree_merge_kernel(const float2* row_top, const float* row_lse, int R, int P, int k, int B, int d,
                                  int32_t* front_tok, int32_t* front_node, float* front_score, int32_t* n_front,
                                  int32_t* pool_tok, int32_t* pool_parent, int32_t* pool_depth, float* pool_score,
                                  int32_t* pool_n) {
    extern __shared__ float tm_smem[];
    Cand* cand = reinterpret_cast<Cand*>(tm_smem);                   // [P * k] children
    Cand* sorted = cand + P * k;                                     // [P * k] in rank order
    int* parent_node = reinterpret_cast<int*>(sorted + P * k);       // [P]
    pdl_wait();
    pdl_trigger();
    const int i = blockIdx.x;
    const int nf = n_front[i];
    for (int f = threadIdx.x; f < P; f += blockDim.x) parent_node[f] = front_node[static_cast<size_t>(i) * P + f];
    for (int t = threadIdx.x; t < nf * k; t += blockDim.x) {
        const int f = t / k, q = t % k;
        const size_t grow = static_cast<size_t>(i) * P + f;
        const float2 e = row_top[grow * kMaxTopK + q];
        // s(c) = s(p) + log pi(v | p)
        cand[t] = Cand{front_score[grow] + (e.x - row_lse[grow]), f, q, __float_as_int(e.y)};
    }
    __syncthreads();
    tree_keep_children(i, P, B, d, nf * k, cand, sorted, parent_node, pool_n[i], front_tok, front_node, front_score,
                       n_front, pool_tok, pool_parent, pool_depth, pool_score, pool_n);
}

// One CTA per request: rank the pool by (score desc, depth asc, creation asc),
// keep the top N, emit root + nodes in rank order and the tree-causal mask.
// The pool is staged in shared memory first.
__global__ void tree_finalize_kernel(int R, int P, int B, int N, const int32_t* pool_tok, const int32_t* pool_parent,
                                     const int32_t* pool_depth, const float* pool_score, const int32_t* pool_n,
                                     int32_t* tok, int32_t* parent, int32_t* depth, float* score, uint32_t* mask,
                                     int32_t* n_nodes) {
    extern __shared__ unsigned long long tf_smem[];
    const int pool_cap = 1 + P * B;
    unsigned long long* s_key = tf_smem;   // pool rank keys: larger = earlier in the output order
    int* slot_of = reinterpret_cast<int*>(s_key + pool_cap);   // pool index -> output slot (-1: not selected)
    int* node_at = slot_of + pool_cap;    // output slot -> pool index
    int* s_par = node_at + (N + 1);       // pool parents
    pdl_wait();
    pdl_trigger();
    const int i = blockIdx.x;
    const size_t pb = static_cast<size_t>(i) * pool_cap;
    const int np = pool_n[i];
    const int S = N + 1;
    const int take = (np - 1) < N ? (np - 1) : N;
    for (int j = threadIdx.x; j < pool_cap; j += blockDim.x) {
        slot_of[j] = -1;
        if (j < np) {
            s_par[j] = pool_parent[pb + j];
            // (score desc, depth asc, creation asc) as one key; scores through
            // their order-preserving bits, a strict total order even for NaN
            // (depth <= B < 2^15, creation < 2^16); depth and score are read
            // back from the key
            s_key[j] = (static_cast<unsigned long long>(ordered_bits(pool_score[pb + j])) << 32) |
                       (static_cast<unsigned long long>(0x7fffu - static_cast<uint32_t>(pool_depth[pb + j])) << 16) |
                       static_cast<unsigned long long>(0xffffu - static_cast<uint32_t>(j));
        }
    }
    __syncthreads();
    // the rank of pool node j >= 1: the nodes before it, four threads per node
    // each counting a quarter (blockDim is a multiple of 32: every lane of a
    // warp runs each round)
    for (int t0 = 0; t0 < 4 * (np - 1); t0 += blockDim.x) {
        const int t = t0 + static_cast<int>(threadIdx.x);
        const int j = 1 + (t >> 2);
        int rank = 0;
        if (j < np) {
            const unsigned long long kj = s_key[j];
            for (int q = 1 + (t & 3); q < np; q += 4) rank += s_key[q] > kj ? 1 : 0;
        }
        rank += __shfl_xor_sync(0xffffffffu, rank, 1);
        rank += __shfl_xor_sync(0xffffffffu, rank, 2);
        if (j < np && (t & 3) == 0 && rank < take) {
            slot_of[j] = rank + 1;
            node_at[rank + 1] = j;
        }
    }
    if (threadIdx.x == 0) {
        slot_of[0] = 0;
        node_at[0] = 0;
    }
    __syncthreads();
    const size_t ob = static_cast<size_t>(i) * S;
    const int words = (S + 31) / 32;
    for (int c = threadIdx.x; c < S; c += blockDim.x) {
        uint32_t* mrow = mask + (ob + c) * words;
        if (c <= take) {
            const int j = node_at[c];
            tok[ob + c] = pool_tok[pb + j];
            parent[ob + c] = (c == 0) ? -1 : slot_of[s_par[j]];
            depth[ob + c] = 0x7fff - static_cast<int>((s_key[j] >> 16) & 0xffffu);
            score[ob + c] = (c == 0) ? 0.f : key_value(s_key[j]);
            for (int w = 0; w < words; ++w) {   // bit sa of the row: ancestors (and the node) in word w
                uint32_t bits = 0u;
                for (int a = j; a >= 0; a = (a == 0 ? -1 : s_par[a])) {
                    const int sa = slot_of[a];
                    if (sa >= 0 && (sa >> 5) == w) bits |= 1u << (sa & 31);
                }
                mrow[w] = bits;
            }
        } else {
            tok[ob + c] = -1;
            parent[ob + c] = -1;
            depth[ob + c] = -1;
            score[ob + c] = 0.f;
            for (int w = 0; w < words; ++w) mrow[w] = 0u;
        }
    }
    if (threadIdx.x == 0) n_nodes[i] = take + 1;
}

// One warp per request: the tree (parents, tokens) and the target argmax of
// every slot are staged in shared memory, then the walk follows, from the
// root, the child whose token is the target's choice (lowest slot first).
__global__ void tree_verify_walk_kernel(const unsigned long long* row_keys, int n_chunks, const int32_t* tok,
                                        const int32_t* parent, const int32_t* n_nodes, int R, int N, int B, int V,
                                        int32_t* accept, int32_t* out_tok, int32_t* n_out, int32_t* dev_status) {
    extern __shared__ int tw_smem[];
    pdl_wait();
    pdl_trigger();
    const int S = N + 1;
    int* s_par = tw_smem;
    int* s_tok = s_par + S;
    int* s_rt = s_tok + S;
    const int i = blockIdx.x;
    const int lane = threadIdx.x;
    const size_t base = static_cast<size_t>(i) * S;
    int32_t* o = out_tok + static_cast<size_t>(i) * (B + 1);
    int nn = n_nodes[i];
    if (nn < 1 || nn > S) {
        if (lane == 0) set_status(dev_status, SDM_DEV_BAD_WINDOW);
        nn = nn < 1 ? 1 : S;
    }
    for (int c = lane; c < nn; c += 32) {
        s_par[c] = parent[base + c];
        s_tok[c] = tok[base + c];
        int t = row_token(row_keys, base + c, n_chunks);
        if (t < 0 || t >= V) {
            set_status(dev_status, SDM_DEV_BAD_TOKEN);
            t = 0;
        }
        s_rt[c] = t;
    }
    __syncwarp();
    int cur = 0, a = 0;
    for (;;) {
        const int t = s_rt[cur];
        int next = -1;
        for (int c0 = 1; c0 < nn; c0 += 32) {
            const int c = c0 + lane;
            const bool hit = c < nn && s_par[c] == cur && s_tok[c] == t;
            const unsigned bal = __ballot_sync(0xffffffffu, hit);
            if (bal) {
                next = c0 + __ffs(bal) - 1;
                break;
            }
        }
        if (lane == 0) o[a] = t;
        if (next < 0 || a >= B) break;
        ++a;
        cur = next;
    }
    for (int p = a + 1 + lane; p <= B; p += 32) o[p] = -1;
    if (lane == 0) {
        accept[i] = a;
        n_out[i] = a + 1;
    }
}

inline int blocks_for(long long n, int t) { return static_cast<int>((n + t - 1) / t); }

}  // namespace

cudaError_t launch_fill_u64(unsigned long long* p, size_t n, unsigned long long v, cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    const int grid = static_cast<int>(n / 256 + 1 < 1024 ? n / 256 + 1 : 1024);
    fill_u64_kernel<<<grid, 256, 0, s>>>(p, n, v);
    return cudaGetLastError();
}

cudaError_t launch_chain_finalize(const unsigned long long* keys, int R, int B, int V, int32_t* tokens,
                                  int32_t* dev_status, cudaStream_t s) {
    chain_finalize_kernel<<<blocks_for(static_cast<long long>(R) * B, 128), 128, 0, s>>>(keys, R, B, V, tokens,
                                                                                         dev_status);
    return cudaGetLastError();
}

cudaError_t launch_schedule(const float* conf, int R, int gamma, const double* cost, float* survival,
                            int32_t* budget, double* expected, int32_t* total_tokens, unsigned long long*,
                            int32_t* dev_status, cudaStream_t s) {
    (void)dev_status;
    int n_pad = 1;
    while (n_pad < R * gamma) n_pad <<= 1;
    const size_t smem = schedule_smem_bytes(R, gamma, n_pad, kSchedThreads);
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(schedule_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    const int nt = n_pad < 64 ? 64 : (n_pad > kSchedThreads ? kSchedThreads : n_pad);
    return launch_pdl(schedule_kernel, dim3(1), dim3(nt), smem, s, conf, R, gamma, cost, survival, budget,
                      expected, total_tokens, n_pad);
}

cudaError_t launch_schedule_dynamic(const float* conf, const float* conf_stale, int R, int gamma, const double* cost,
                                    float* survival, int32_t* budget, double* expected, int32_t* total_tokens,
                                    int32_t* capacity, cudaStream_t s) {
    int n_pad = 1;
    while (n_pad < R * gamma) n_pad <<= 1;
    const size_t smem = static_cast<size_t>(n_pad) * 8 + kSchedThreads * 8 + static_cast<size_t>(R) * 4 +
                        static_cast<size_t>(R) * gamma * 4;
    static bool configured = false;
    if (!configured) {
        cudaError_t e =
            cudaFuncSetAttribute(schedule_dynamic_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    const int nt = n_pad < 64 ? 64 : (n_pad > kSchedThreads ? kSchedThreads : n_pad);
    return launch_pdl(schedule_dynamic_kernel, dim3(1), dim3(nt), smem, s, conf, conf_stale, R, gamma, cost, survival,
                      budget, expected, total_tokens, capacity, n_pad);
}

cudaError_t launch_pack(const int32_t* anchor, const int32_t* draft, const int32_t* budget, int R, int gamma,
                        const int32_t* tiers, int n_tiers, int strict, int32_t* cu, int32_t* ptok, int32_t* preq,
                        int32_t* ppos, int capacity, int32_t* tier, int32_t* dev_status, cudaStream_t s) {
    return launch_pdl(pack_kernel, dim3(1), dim3(kPackThreads), 0, s, anchor, draft, budget, R, gamma, tiers, n_tiers,
                      strict, cu, ptok, preq, ppos, capacity, tier, dev_status);
}

cudaError_t launch_verify_greedy_finalize(int mode, const int32_t* cu, const int32_t* draft, const int32_t* budget,
                                          const unsigned long long* row_keys, int n_chunks, int R, int gamma, int V,
                                          int rows_avail, int32_t* accept, int32_t* ceiling, int32_t* out_tok,
                                          int32_t* n_out, int32_t* dev_status, cudaStream_t s) {
    return launch_pdl(verify_greedy_finalize_kernel, dim3(blocks_for(static_cast<long long>(R) * 32, 128)), dim3(128),
                      0, s, mode, cu, draft, budget, row_keys, n_chunks, R, gamma, V, rows_avail, accept, ceiling,
                      out_tok, n_out, dev_status);
}

cudaError_t launch_verify_sample_scan(int mode, const int32_t* cu, const int32_t* anchor, const int32_t* draft,
                                      const int32_t* budget, const float* logq, const void* target, int t_fp32,
                                      int V, const float2* lse_part, int n_chunks, float inv_t, uint32_t k0,
                                      uint32_t k1, uint32_t cycle, int R, int gamma, int32_t* accept,
                                      int32_t* ceiling, int32_t* res_tok, int32_t* res_pos, int32_t* res_trow,
                                      float* res_lse_p, int32_t* bonus_row, int32_t* bonus_pos, int rows_avail,
                                      int32_t* dev_status, cudaStream_t s) {
    return launch_pdl(verify_sample_scan_kernel, dim3(blocks_for(static_cast<long long>(R) * 32, 128)), dim3(128), 0,
                      s, mode, cu, anchor, draft, budget, logq, target, t_fp32, V, lse_part, n_chunks, inv_t, k0, k1,
                      cycle, R, gamma, accept, ceiling, res_tok, res_pos, res_trow, res_lse_p, bonus_row, bonus_pos,
                      rows_avail, dev_status);
}

cudaError_t launch_tree_init(const int32_t* anchor, int R, int P, int B, int32_t* front_tok, int32_t* front_node,
                             float* front_score, int32_t* n_front, int32_t* pool_tok, int32_t* pool_parent,
                             int32_t* pool_depth, float* pool_score, int32_t* pool_n, int32_t* dev_status,
                             cudaStream_t s) {
    return launch_pdl(tree_init_kernel, dim3(blocks_for(R, 128)), dim3(128), 0, s, anchor, R, P, B, front_tok,
                      front_node, front_score, n_front, pool_tok, pool_parent, pool_depth, pool_score, pool_n,
                      dev_status);
}

cudaError_t launch_tree_merge(const float2* row_top, const float* row_lse, int R, int P, int k, int B, int d,
                              int32_t* front_tok, int32_t* front_node, float* front_score, int32_t* n_front,
                              int32_t* pool_tok, int32_t* pool_parent, int32_t* pool_depth, float* pool_score,
                              int32_t* pool_n, cudaStream_t s) {
    const size_t smem = 2 * static_cast<size_t>(P) * k * sizeof(Cand) + static_cast<size_t>(P) * 4;
    return launch_pdl(tree_merge_kernel, dim3(R), dim3(128), smem, s, row_top, row_lse, R, P, k, B, d, front_tok,
                      front_node, front_score, n_front, pool_tok, pool_parent, pool_depth, pool_score, pool_n);
}

cudaError_t launch_tree_finalize(int R, int P, int B, int N, const int32_t* pool_tok, const int32_t* pool_parent,
                                 const int32_t* pool_depth, const float* pool_score, const int32_t* pool_n,
                                 int32_t* tok, int32_t* parent, int32_t* depth, float* score, uint32_t* mask,
                                 int32_t* n_nodes, cudaStream_t s) {
    const int pool_cap = 1 + P * B;
    const size_t smem = static_cast<size_t>(pool_cap) * 16 + static_cast<size_t>(N + 1) * 4;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(tree_finalize_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             200 * 1024);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    return launch_pdl(tree_finalize_kernel, dim3(R), dim3(256), smem, s, R, P, B, N, pool_tok, pool_parent, pool_depth,
                      pool_score, pool_n, tok, parent, depth, score, mask, n_nodes);
}

cudaError_t launch_tree_verify_walk(const unsigned long long* row_keys, int n_chunks, const int32_t* tok, const int32_t* parent,
                                    const int32_t* n_nodes, int R, int N, int B, int V, int32_t* accept,
                                    int32_t* out_tok, int32_t* n_out, int32_t* dev_status, cudaStream_t s) {
    const size_t smem = static_cast<size_t>(N + 1) * 12;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(tree_verify_walk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             200 * 1024);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    return launch_pdl(tree_verify_walk_kernel, dim3(R), dim3(32), smem, s, row_keys, n_chunks, tok, parent, n_nodes, R,
                      N, B, V, accept, out_tok, n_out, dev_status);
}

int num_sms() {
    static int n = 0;
    if (n == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0) n = 148;
    }
    return n;
}

}  // namespace sdm
