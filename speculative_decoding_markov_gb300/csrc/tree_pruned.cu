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
// tree_rows_kernel (once per cycle, one CTA per (request, level) row): the
//   row's lists, L_(k), and the ids with L >= L_(k) - 2 c_max in (L desc, id
//   asc) order; a row whose lists overflowed or whose ids do not fit is
//   marked for the exhaustive path.
// tree_level_kernel (per level, one CTA per request): the parents' U rows and
//   log-sum-exps, the row's ids' W^T rows, z for every (parent, id) with
//   L >= L_(k) - 2 c(y), exactly (fp32 products summed in fp32: exact on the
//   grid tables), each parent's top k, the children's scores and the
//   per-level prune.  A marked row takes every parent's top k over the whole
//   vocabulary from global memory instead (slow, but exact).
#include "device.cuh"
#include "internal.h"
#include "tree_common.cuh"

namespace sdm {
namespace {

constexpr int kLvThreads = 256;
constexpr int kLvWarps = kLvThreads / 32;
constexpr int kGather = 2048;   // listed entries of a row held in shared memory
constexpr int kMaxPartLane = 8;    // GEMM partials per lane a warp loads at once (n_part <= 256 CTA columns)

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

// Warp-wide tensor-core step for the level's dots: D[16 x 8] += A[16 x 16] B,
// A = 16 W^T rows (ids x K, K contiguous), B = 8 U rows (parents x K, K
// contiguous): bf16 in, fp32 accumulate.  Fragments by ldmatrix from rows
// 16-byte aligned; lane l addresses A row (l % 16), K offset 8 (l / 16), and
// B row (l % 8), K offset 8 ((l / 8) % 2).
__device__ __forceinline__ void ldsm_x4(uint32_t (&a)[4], const uint16_t* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3])
                 : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x2(uint32_t (&b)[2], const uint16_t* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];" : "=r"(b[0]), "=r"(b[1]) : "r"(smem_u32(p)));
}
__device__ __forceinline__ void mma_16816_bf16(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
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

// The warp's largest value among every lane's v[] (-inf when all are -inf),
// one occurrence of it removed (from the lowest lane holding it); every lane
// gets the value.
template <int N>
__device__ __forceinline__ float warp_take_max(float (&v)[N]) {
    const int lane = threadIdx.x & 31;
    float m = v[0];
#pragma unroll
    for (int e = 1; e < N; ++e) m = fmaxf(m, v[e]);
    float wm = m;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) wm = fmaxf(wm, __shfl_xor_sync(0xffffffffu, wm, o));
    const unsigned holders = __ballot_sync(0xffffffffu, m == wm && wm > -INFINITY);
    if (holders && lane == __ffs(holders) - 1) {
        bool done = false;
#pragma unroll
        for (int e = 0; e < N; ++e)
            if (!done && v[e] == wm) {
                v[e] = -INFINITY;
                done = true;
            }
    }
    return wm;
}

// ---------------------------------------------------------------------------
// Once per cycle: the ids each (request, level) row can need
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kLvThreads) tree_rows_kernel(const TreeRowsParams p) {
    __shared__ int s_pref[kMaxPickChunks + 1];
    __shared__ uint2 s_g[kGather];
    __shared__ uint2 s_keep[kTreeKeep];
    __shared__ int s_nkeep, s_bad;
    __shared__ float s_lk;
    __shared__ float s_wtop[kLvWarps][kMaxTopK];   // each warp's k largest listed values, in order
    pdl_wait();
    pdl_trigger();
    const int row = blockIdx.x;   // request * B + (level - 1)
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nc = p.n_chunks, K = p.k;
    const int seg0 = row * nc;
    if (warp == 0) {
        int run = 0, over = 0;
        for (int c0 = 0; c0 < nc; c0 += 32) {
            const int c = c0 + lane;
            int n = 0;
            if (c < nc) {
                const int cn = p.cand_n[seg0 + c];
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
        float lm = -INFINITY;   // the row's largest logit: the largest chunk maximum
        for (int c = lane; c < nc; c += 32) lm = fmaxf(lm, p.cmax[seg0 + c]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) lm = fmaxf(lm, __shfl_xor_sync(0xffffffffu, lm, o));
        if (lane == 0) {
            p.lmax[row] = lm;
            s_pref[nc] = run;
            s_bad = over || run > kGather;
            s_nkeep = 0;
            s_lk = -INFINITY;
        }
    }
    __syncthreads();
    const int total = s_pref[nc];
    if (!s_bad) {
        for (int t = tid; t < total; t += kLvThreads) {
            const int c = list_of(s_pref, nc, t);
            s_g[t] = p.cand[static_cast<size_t>(seg0 + c) * kSegCap + (t - s_pref[c])];
        }
        __syncthreads();
        // L_(k), the k-th largest listed value counted with multiplicity (the
        // lists hold every chunk's top k, so the row's top k are among
        // them): k rounds per warp of taking its largest remaining value
        // (one occurrence), then the same over the warps' k values
        constexpr int kPer = kGather / kLvThreads;
        float v[kPer];
#pragma unroll
        for (int e = 0; e < kPer; ++e) {
            const int t = tid + e * kLvThreads;
            v[e] = t < total ? __uint_as_float(s_g[t].y) : -INFINITY;
        }
        for (int q = 0; q < K; ++q) {
            const float top = warp_take_max<kPer>(v);
            if (lane == 0) s_wtop[warp][q] = top;
        }
        __syncthreads();
        if (warp == 0) {
            float w2[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int t = lane + 32 * e;   // (warp t / k, rank t % k) of the warps' lists
                w2[e] = t < kLvWarps * K ? s_wtop[t / K][t % K] : -INFINITY;
            }
            float top = -INFINITY;
            for (int q = 0; q < K; ++q) top = warp_take_max<2>(w2);
            if (lane == 0) s_lk = top;   // -inf when fewer than k values are listed
        }
        __syncthreads();
        const float lk = s_lk;
        if (lk == -INFINITY) {
            if (tid == 0) s_bad = 1;           // fewer than k listed values
        } else {
            const float tu = markov_cut(lk, *p.c_max);   // the ids any parent can need
            for (int t = tid; t < total; t += kLvThreads) {
                const uint2 e = s_g[t];
                if (e.x < static_cast<uint32_t>(p.V) && __uint_as_float(e.y) >= tu) {
                    const int slot = atomicAdd(&s_nkeep, 1);
                    if (slot < kTreeKeep) s_keep[slot] = e;
                }
            }
        }
        __syncthreads();
        if (s_nkeep > kTreeKeep && tid == 0) s_bad = 1;
        __syncthreads();
    }
    uint2* out = p.keep + static_cast<size_t>(row) * kTreeKeep;
    if (s_bad) {
        if (tid == 0) {
            p.n_keep[row] = -1;
            p.lk[row] = -INFINITY;
        }
        return;
    }
    // (L desc, id asc): a parent's ids are then a prefix
    const int nk = s_nkeep;
    if (tid < nk) {   // nk <= kTreeKeep <= kLvThreads: one id per thread
        const uint2 mine = s_keep[tid];
        const float x = __uint_as_float(mine.y);
        int rk = 0;
        for (int u = 0; u < nk; ++u) {
            const uint2 o = s_keep[u];
            const float y = __uint_as_float(o.y);
            rk += (y > x || (y == x && o.x < mine.x)) ? 1 : 0;
        }
        out[rk] = mine;
    }
    if (tid == 0) {
        p.n_keep[row] = nk;
        p.lk[row] = s_lk;
    }
}

// ---------------------------------------------------------------------------
// Per level: every parent's top k, the children's scores, the prune
// ---------------------------------------------------------------------------
struct LevelLayout {
    uint32_t w, u, z, total;
    int rs;   // staged row stride (elements): r + 8 (16 bytes apart in the banks)
};

// Dynamic shared memory: the row's ids' W^T rows [kTreeKeep][rs] bf16, the
// parents' U rows [P][rs] bf16, the logits [P][kTreeKeep] fp32.
__host__ __device__ inline LevelLayout level_layout(int P, int r) {
    LevelLayout l;
    l.rs = r + 8;
    const uint32_t row = 2u * static_cast<uint32_t>(l.rs);
    l.w = 0;
    l.u = l.w + static_cast<uint32_t>(kTreeKeep) * row;
    l.z = l.u + static_cast<uint32_t>(P) * row;
    l.total = l.z + static_cast<uint32_t>(P) * kTreeKeep * 4u;
    return l;
}

__global__ void __launch_bounds__(kLvThreads, 1) tree_level_kernel(const TreeLevelParams p) {
    extern __shared__ __align__(16) uint8_t s_dyn[];
    const LevelLayout lay = level_layout(p.P, p.r);
    const int RS = lay.rs;
    uint16_t* s_w = reinterpret_cast<uint16_t*>(s_dyn + lay.w);     // [kTreeKeep][RS]
    uint16_t* s_u = reinterpret_cast<uint16_t*>(s_dyn + lay.u);     // [P][RS]
    float* s_z = reinterpret_cast<float*>(s_dyn + lay.z);           // [P][kTreeKeep]
    __shared__ uint2 s_keep[kTreeKeep];    // the row's ids (id, L bits), (L desc, id asc)
    __shared__ int s_nk;
    __shared__ float s_lk;
    __shared__ int s_tok[kMaxTreeSlots], s_node[kMaxTreeSlots], s_cnt[kMaxTreeSlots];
    __shared__ float s_score[kMaxTreeSlots], s_lse[kMaxTreeSlots];
    __shared__ float2 s_top[kMaxTreeSlots][kMaxTopK];   // per parent: (z, id bits) in rank order
    __shared__ Cand s_cand[kMaxTreeSlots], s_sorted[kMaxTreeSlots];   // P k <= 64 children
    __shared__ unsigned long long s_red[kLvWarps];
    __shared__ int s_nf, s_np;
    const int i = blockIdx.x;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int P = p.P, K = p.k, r = p.r;
    const int row = i * p.B + (p.d - 1);
    // 0. before the wait on the level's GEMM, everything but its partials:
    //    the row's ids (made once per cycle, before the first level) and the
    //    copies of their W^T rows; the frontier and the pool's size, written
    //    by the previous level's kernel (complete before the GEMM passed its
    //    own wait, and this launch begins only after every GEMM CTA did), the
    //    parents' U rows, bounds and id counts.  Loads through L2.
    if (tid == 0) {
        s_nk = __ldcg(p.n_keep + row);
        s_lk = __ldcg(p.lk + row);
        s_nf = min(max(__ldcg(p.n_front + i), 0), P);
        s_np = __ldcg(p.pool_n + i);
    }
    for (int t = tid; t < kTreeKeep; t += kLvThreads) s_keep[t] = __ldcg(p.keep + static_cast<size_t>(row) * kTreeKeep + t);
    for (int f = tid; f < P; f += kLvThreads) {
        const size_t fr = static_cast<size_t>(i) * P + f;
        s_tok[f] = __ldcg(p.front_tok + fr);
        s_node[f] = __ldcg(p.front_node + fr);
        s_score[f] = __ldcg(p.front_score + fr);
    }
    __syncthreads();
    const int nk = s_nk, nf = s_nf;
    const bool exhaust = nk < 0;
    if (!exhaust)
        for (int j = warp; j < nk; j += kLvWarps) {
            const uint16_t* src = p.Wt + static_cast<size_t>(s_keep[j].x) * r;
            for (int q = lane * 8; q < r; q += 256) cp_async_16(s_w + static_cast<size_t>(j) * RS + q, src + q, 16u);
        }
    for (int f = warp; f < nf; f += kLvWarps) {
        const int t = s_tok[f];
        if (t >= 0 && t < p.V)
            for (int q = lane * 8; q < r; q += 256)
                cp_async_16(s_u + static_cast<size_t>(f) * RS + q, p.U + static_cast<size_t>(t) * r + q, 16u);
    }
    // each parent's ids: the prefix of the row's list with L >= L_(k) - 2 c(y)
    for (int f = warp; f < nf; f += kLvWarps) {
        int t = s_tok[f];
        if (t >= p.V) {
            if (lane == 0) set_status(p.dev_status, SDM_DEV_BAD_TOKEN);
            t = -1;
        }
        int n = 0;
        if (t >= 0 && !exhaust) {
            const float thr = markov_cut(s_lk, p.c_bound[t]);
            for (int j0 = 0; j0 < nk; j0 += 32) {
                const int j = j0 + lane;
                n += __popc(__ballot_sync(0xffffffffu, j < nk && __uint_as_float(s_keep[j].y) >= thr));
            }
        }
        __syncwarp();
        if (lane == 0) {
            s_cnt[f] = n;
            if (t < 0) s_tok[f] = -1;
        }
    }
    pdl_wait();
    pdl_trigger();
    // 1. the log-sum-exp of each parent's logits from the GEMM's partials:
    //    the largest maximum, then every partial's sum rescaled to it, summed
    //    in fp32 (a lane's terms, then the butterfly)
    for (int f = warp; f < nf; f += kLvWarps) {
        const float2* pr = p.part + (static_cast<size_t>(i) * P + f) * p.n_part;
        float2 x[kMaxPartLane];
#pragma unroll
        for (int e = 0; e < kMaxPartLane; ++e) {
            const int q = lane + e * 32;
            x[e] = q < p.n_part ? pr[q] : make_float2(-INFINITY, 0.f);
        }
        float m = -INFINITY;
#pragma unroll
        for (int e = 0; e < kMaxPartLane; ++e)
            if (x[e].y > 0.f) m = fmaxf(m, x[e].x);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float sum = 0.f;
#pragma unroll
        for (int e = 0; e < kMaxPartLane; ++e)
            if (x[e].y > 0.f) sum += x[e].y * expf(x[e].x - m);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        if (lane == 0) s_lse[f] = m + logf(sum);
    }
    cp_async_wait_all();
    __syncthreads();

    if (!exhaust) {
        // 2. z for every (parent, id) pair: fp32(L) + U[y] . W^T[v], one warp
        //    per 16 ids x 8 parents on the tensor cores (m16n8k16); rows past
        //    the staged ids or parents give values nobody reads
        int nmax = 0;
        for (int f = 0; f < nf; ++f) nmax = max(nmax, s_cnt[f]);
        const int nb16 = (nmax + 15) >> 4, nb8 = (nf + 7) >> 3;
        for (int tb = warp; tb < nb16 * nb8; tb += kLvWarps) {
            const int jb = (tb % nb16) * 16, fb = (tb / nb16) * 8;
            const uint16_t* arow = s_w + static_cast<size_t>(jb + (lane & 15)) * RS + ((lane >> 4) << 3);
            const uint16_t* brow = s_u + static_cast<size_t>(min(fb + (lane & 7), P - 1)) * RS + (((lane >> 3) & 1) << 3);
            // two accumulators over alternate K steps (r / 16 is even): half
            // the dependent chain
            float d[4] = {0.f, 0.f, 0.f, 0.f}, d2[4] = {0.f, 0.f, 0.f, 0.f};
            for (int k0 = 0; k0 < r; k0 += 32) {
                uint32_t a[4], b[2], a2[4], b2[2];
                ldsm_x4(a, arow + k0);
                ldsm_x2(b, brow + k0);
                ldsm_x4(a2, arow + k0 + 16);
                ldsm_x2(b2, brow + k0 + 16);
                mma_16816_bf16(d, a, b);
                mma_16816_bf16(d2, a2, b2);
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) d[e] += d2[e];
            // lane (g, t) = (lane / 4, lane % 4) holds ids jb + g, jb + g + 8
            // and parents fb + 2 t, fb + 2 t + 1
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int j = jb + (lane >> 2) + (e >> 1) * 8, f = fb + 2 * (lane & 3) + (e & 1);
                if (f < nf && j < s_cnt[f]) s_z[f * kTreeKeep + j] = __uint_as_float(s_keep[j].y) + d[e];
            }
        }
        __syncthreads();
        // each parent's top k by (z desc, id asc): one warp per parent, k
        // rounds of the warp's largest remaining key (keys are distinct: the
        // ids differ)
        for (int f = warp; f < nf; f += kLvWarps) {
            const int n = s_cnt[f];
            unsigned long long key[kTreeKeep / 32];
#pragma unroll
            for (int e = 0; e < kTreeKeep / 32; ++e) {
                const int j = lane + 32 * e;
                key[e] = j < n ? argmax_key(s_z[f * kTreeKeep + j], s_keep[j].x) : 0ull;
            }
            for (int q = 0; q < K; ++q) {
                unsigned long long best = 0ull;
#pragma unroll
                for (int e = 0; e < kTreeKeep / 32; ++e) best = umax64(best, key[e]);
                // the warp's largest key: its high word, then the low word
                // among the lanes that hold that high word
                const uint32_t hi = __reduce_max_sync(0xffffffffu, static_cast<uint32_t>(best >> 32));
                const uint32_t lo = __reduce_max_sync(
                    0xffffffffu, static_cast<uint32_t>(best >> 32) == hi ? static_cast<uint32_t>(best) : 0u);
                const unsigned long long m = (static_cast<unsigned long long>(hi) << 32) | lo;
#pragma unroll
                for (int e = 0; e < kTreeKeep / 32; ++e)
                    if (key[e] == m) key[e] = 0ull;
                if (lane == 0)
                    s_top[f][q] = m ? make_float2(key_value(m), __int_as_float(static_cast<int>(key_token(m))))
                                    : make_float2(-INFINITY, __int_as_float(-1));
            }
        }
    } else {
        // every id of the vocabulary for every parent, W^T rows from global
        // memory; per thread a sorted list of its k best keys, then k rounds
        // of the block maximum
        const size_t lrow = static_cast<size_t>(row) * p.V;
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
    // 3. children s = s(p) + (z - lse(p)), the P best kept; every child's U
    //    row is asked into L2 for the next level's GEMM, which gathers the
    //    kept ones
    const int ncand = nf * K;
    for (int t = tid; t < ncand; t += kLvThreads) {
        const int f = t / K, q = t - f * K;
        const float2 e = s_top[f][q];
        const int ct = __float_as_int(e.y);
        if (s_tok[f] >= 0 && ct >= 0 && ct < p.V)
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p.U + static_cast<size_t>(ct) * r),
                         "r"(r * 2)
                         : "memory");
        s_cand[t] = s_tok[f] >= 0 ? Cand{s_score[f] + (e.x - s_lse[f]), f, q, __float_as_int(e.y)}
                                  : Cand{-INFINITY, f, q, -1};
    }
    __syncthreads();
    tree_keep_children(i, P, p.B, p.d, ncand, s_cand, s_sorted, s_node, s_np, p.front_tok, p.front_node,
                       p.front_score, p.n_front, p.pool_tok, p.pool_parent, p.pool_depth, p.pool_score, p.pool_n);
}

}  // namespace

size_t tree_level_smem(int P, int r) { return level_layout(P, r).total; }

cudaError_t launch_tree_rows(const TreeRowsParams& p, cudaStream_t s) {
    if (p.k > kMaxTopK || p.n_chunks > kMaxPickChunks) return cudaErrorInvalidValue;
    return launch_pdl(tree_rows_kernel, dim3(p.rows), dim3(kLvThreads), 0, s, p);
}

cudaError_t launch_tree_level(const TreeLevelParams& p, cudaStream_t s) {
    if (p.P > kMaxTreeSlots || p.k > kMaxTopK || p.n_part > 32 * kMaxPartLane) return cudaErrorInvalidValue;
    const size_t smem = tree_level_smem(p.P, p.r);
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
