// chain_pruned.cu - the greedy Markov-head chain without the dense projection.
//
// Greedy drafting needs y_d = argmax_v z_d[v], z_d = fp32(L_d) + U[y_{d-1}] W.
// The Markov term is bounded: |U[y] . W[:, v]| <= |U[y]|_2 |W[:, v]|_2 <= C(y)
// with C(y) = u_norm[y] * n_max from the prepared tables (Cauchy-Schwarz), so
// no id with L_d[v] < max_v L_d[v] - 2 C(y) can be the argmax.  Only the
// threshold depends on the previous token, and C(y) <= C_max = u_max * n_max,
// which splits the chain into two launches:
//
//   chain_scan_kernel  (every (request, step) row in parallel, HBM-bound)
//     a cluster of CTAs per row copies the row L_d into shared memory (bulk
//     TMA), reduces its maximum over the cluster through distributed shared
//     memory and lists every id with L_d[v] >= max - 2 C_max.  L is read from
//     HBM exactly once.
//   chain_pick_kernel  (one CTA per request, the B dependent steps)
//     step d keeps the listed ids with L_d[v] >= max - 2 C(y_{d-1}) and scores
//     them exactly, z = L + U[y_{d-1}] . W^T[v] (fp32, from the prepared W^T,
//     whose rows were prefetched into L2), then takes the (z desc, id asc)
//     winner.  A row whose list overflowed is rescanned in full.
//
// The result equals the dense argmax bit for bit: the kept set contains every
// id that can reach the maximum and the kept ids are scored exactly.
#include <cooperative_groups.h>
#include <cuda_bf16.h>

#include "device.cuh"
#include "internal.h"

namespace cg = cooperative_groups;

namespace sdm {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

template <int FP32>
__device__ __forceinline__ void unpack(const uint4& x, float (&v)[FP32 ? 4 : 8]) {
    if (FP32) {
        v[0] = __uint_as_float(x.x);
        v[1] = __uint_as_float(x.y);
        v[2] = __uint_as_float(x.z);
        v[3] = __uint_as_float(x.w);
    } else {
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            v[2 * q] = __uint_as_float(w[q] << 16);
            v[2 * q + 1] = __uint_as_float(w[q] & 0xffff0000u);
        }
    }
}

// Maximum of the elements of a 16-byte vector folded into a running maximum.
template <int FP32>
__device__ __forceinline__ void fold_max(const uint4& x, uint4& acc) {
    if (FP32) {
        acc.x = __float_as_uint(fmaxf(__uint_as_float(acc.x), __uint_as_float(x.x)));
        acc.y = __float_as_uint(fmaxf(__uint_as_float(acc.y), __uint_as_float(x.y)));
        acc.z = __float_as_uint(fmaxf(__uint_as_float(acc.z), __uint_as_float(x.z)));
        acc.w = __float_as_uint(fmaxf(__uint_as_float(acc.w), __uint_as_float(x.w)));
    } else {   // packed bf16x2 maxima: one instruction per pair of elements
        __nv_bfloat162 a[4], b[4];
        memcpy(a, &acc, 16);
        memcpy(b, &x, 16);
#pragma unroll
        for (int q = 0; q < 4; ++q) a[q] = __hmax2(a[q], b[q]);
        memcpy(&acc, a, 16);
    }
}

template <int FP32>
__device__ __forceinline__ float vec_max(const uint4& x) {
    float v[FP32 ? 4 : 8];
    unpack<FP32>(x, v);
    float m = v[0];
#pragma unroll
    for (int q = 1; q < (FP32 ? 4 : 8); ++q) m = fmaxf(m, v[q]);
    return m;
}

// Maximum of one 16-byte vector: a packed bf16x2 tree, two conversions at the end.
template <int FP32>
__device__ __forceinline__ float vec_max_packed(const uint4& x) {
    if (FP32)
        return fmaxf(fmaxf(__uint_as_float(x.x), __uint_as_float(x.y)), fmaxf(__uint_as_float(x.z), __uint_as_float(x.w)));
    __nv_bfloat162 w[4];
    memcpy(w, &x, 16);
    const __nv_bfloat162 m = __hmax2(__hmax2(w[0], w[1]), __hmax2(w[2], w[3]));
    uint32_t b;
    memcpy(&b, &m, 4);
    return fmaxf(__uint_as_float(b << 16), __uint_as_float(b & 0xffff0000u));
}

__device__ __forceinline__ const uint8_t* row_ptr(const PrunedParams& p, int row, int d, int v) {
    const size_t esz = p.l_fp32 ? 4 : 2;
    return static_cast<const uint8_t*>(p.L) + ((static_cast<size_t>(row) * p.B + (d - 1)) * p.V + v) * esz;
}

// Bulk (non-tensor) TMA copy global -> shared, completing on an mbarrier.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// The bound C on |Markov(prev)| with slack for the fp32 rounding of the
// product, and the candidate threshold below a row maximum m.
__device__ __forceinline__ float bound_c(float norm_u, float n_max) {
    return norm_u * n_max * 1.0009765625f + 9.5367431640625e-7f;
}
__device__ __forceinline__ float threshold(float m, float c) {
    return m - 2.0f * c - fabsf(m) * 9.765625e-4f - 9.5367431640625e-7f;
}

// ---------------------------------------------------------------------------
// A: candidate lists of every (request, step, chunk)
// ---------------------------------------------------------------------------
// Work item = kChunkIds consecutive ids of one row L_d (32 KB); a persistent
// grid walks the items.  Each thread holds 8 16-byte vectors of the chunk in
// registers, the chunk maximum m_c is reduced over the CTA, and every id with
// L >= m_c - 2 C_max is listed.  m_c <= max_v L_d[v] and C(y) <= C_max, so the
// list holds every id the exact step can need.
template <int FP32>
__global__ void __launch_bounds__(kThreads) chain_scan_kernel(const PrunedParams p) {
    constexpr int VEC = FP32 ? 4 : 8;
    constexpr int VPT = kChunkBytes / 16 / kThreads;        // vectors per thread
    __shared__ float s_wmax[kWarps];
    __shared__ int s_cnt;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int chunk_ids = kChunkBytes / (FP32 ? 4 : 2);
    const long long items = static_cast<long long>(p.R) * p.B * p.n_chunks;
    const float cmax = bound_c(*p.u_max, *p.n_max);
    for (long long it = blockIdx.x; it < items; it += gridDim.x) {
        const int rs = static_cast<int>(it / p.n_chunks);
        const int c = static_cast<int>(it % p.n_chunks);
        const int row = rs / p.B, d = rs % p.B + 1;
        const int v0 = c * chunk_ids;
        const int n_vec = (min(p.V, v0 + chunk_ids) - v0) / VEC;
        const uint4* src = reinterpret_cast<const uint4*>(row_ptr(p, row, d, v0));
        {   // this CTA's next item starts moving from HBM into L2 now
            const long long nx = it + gridDim.x;
            if (nx < items) {
                const int nrs = static_cast<int>(nx / p.n_chunks), nc = static_cast<int>(nx % p.n_chunks);
                const int nv0 = nc * chunk_ids;
                const int nbytes = (min(p.V, nv0 + chunk_ids) - nv0) * (FP32 ? 4 : 2);
                const char* nsrc = reinterpret_cast<const char*>(row_ptr(p, nrs / p.B, nrs % p.B + 1, nv0));
                for (int off = threadIdx.x * 128; off < nbytes; off += kThreads * 128)
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(nsrc + off));
            }
        }
        uint4 x[VPT];
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int i = threadIdx.x + k * kThreads;
            x[k] = i < n_vec ? __ldcs(src + i) : (FP32 ? make_uint4(0xff800000u, 0xff800000u, 0xff800000u, 0xff800000u)
                                                       : make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u));
        }
        uint4 acc = x[0];
#pragma unroll
        for (int k = 1; k < VPT; ++k) fold_max<FP32>(x[k], acc);
        const float tmax = vec_max<FP32>(acc);
        float m = tmax;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) s_wmax[warp] = m;
        if (threadIdx.x == 0) s_cnt = 0;
        __syncthreads();
        float mc = s_wmax[0];
#pragma unroll
        for (int w = 1; w < kWarps; ++w) mc = fmaxf(mc, s_wmax[w]);
        const float T = threshold(mc, cmax);
        const size_t seg = static_cast<size_t>(rs) * p.n_chunks + c;
        uint2* out = p.cand + seg * kSegCap;
        if (tmax >= T) {
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                if (vec_max_packed<FP32>(x[k]) < T) continue;
                float v[VEC];
                unpack<FP32>(x[k], v);
                const int i = threadIdx.x + k * kThreads;
#pragma unroll
                for (int q = 0; q < VEC; ++q) {
                    if (v[q] >= T) {
                        const int slot = atomicAdd(&s_cnt, 1);
                        if (slot < kSegCap)
                            out[slot] = make_uint2(static_cast<uint32_t>(v0 + i * VEC + q), __float_as_uint(v[q]));
                    }
                }
            }
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            p.cand_n[seg] = s_cnt;        // the true count: above kSegCap the list is incomplete
            p.cmax[seg] = mc;
        }
    }
}

// ---------------------------------------------------------------------------
// B: the B dependent steps of each request
// ---------------------------------------------------------------------------
constexpr int kGroup = 8;       // candidates a warp scores per round
constexpr int kPickCap = 1024;  // ids staged per step (more: the full-row path)
constexpr int kStageEntries = 16384;   // listed ids of one request held in shared memory

// Warp-cooperative exact scores of the staged ids: lanes hold 8 of r; a warp
// scores kGroup ids per round with all their W^T row loads in flight.
__device__ __forceinline__ unsigned long long score_staged(const PrunedParams& p, const uint2* ids, int n,
                                                           const float (&ub)[8], int warp, int lane) {
    unsigned long long best = 0ull;
    for (int c0 = warp * kGroup; c0 < n; c0 += kWarps * kGroup) {
        uint2 cd[kGroup];
        uint4 wv[kGroup];
#pragma unroll
        for (int j = 0; j < kGroup; ++j) {
            cd[j] = (c0 + j < n) ? ids[c0 + j] : make_uint2(0xffffffffu, 0u);
            const bool ok = cd[j].x < static_cast<uint32_t>(p.V) && lane * 8 < p.r;
            wv[j] = ok ? __ldg(reinterpret_cast<const uint4*>(p.Wt + static_cast<size_t>(cd[j].x) * p.r) + lane)
                       : make_uint4(0, 0, 0, 0);
        }
        float acc[kGroup];
#pragma unroll
        for (int j = 0; j < kGroup; ++j) {
            float a[8];
            unpack<0>(wv[j], a);
            acc[j] = 0.f;
#pragma unroll
            for (int q = 0; q < 8; ++q) acc[j] = fmaf(a[q], ub[q], acc[j]);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
#pragma unroll
            for (int j = 0; j < kGroup; ++j) acc[j] += __shfl_xor_sync(0xffffffffu, acc[j], o);
#pragma unroll
        for (int j = 0; j < kGroup; ++j)
            if (cd[j].x < static_cast<uint32_t>(p.V))
                best = umax64(best, argmax_key(__uint_as_float(cd[j].y) + acc[j], cd[j].x));   // fp32(L) + Markov
    }
    return best;
}

__device__ __forceinline__ void prefetch_row_l2(const uint16_t* base, uint32_t v, int r) {
    const char* a = reinterpret_cast<const char*>(base + static_cast<size_t>(v) * r);
    for (int off = 0; off < r * 2; off += 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(a + off));
}

template <int FP32>
__global__ void __launch_bounds__(kThreads, 1) chain_pick_kernel(const PrunedParams p) {
    constexpr int VEC = FP32 ? 4 : 8;
    const int row = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    extern __shared__ __align__(16) uint8_t s_dyn[];
    const int nc = p.n_chunks;
    const int nseg = p.B * nc;
    uint2* s_list = reinterpret_cast<uint2*>(s_dyn);               // [kStageEntries] all lists, packed
    float* s_cm = reinterpret_cast<float*>(s_list + kStageEntries); // [B][nc] chunk maxima
    int* s_cn = reinterpret_cast<int*>(s_cm + nseg);               // [B][nc] list lengths
    int* s_soff = s_cn + nseg;                                     // [B * nc + 1] packed offsets
    __shared__ __align__(8) uint64_t s_bar;
    __shared__ int s_staged;
    __shared__ uint4 s_u[32];
    __shared__ uint2 s_cand[kPickCap];       // this step's ids with L >= max - 2C
    __shared__ uint2 s_ids[kPickCap];        // the ids of one scoring round
    __shared__ float s_lmax[kMaxPickSteps];
    __shared__ int s_off[kMaxPickChunks + 1];
    __shared__ int s_n, s_m, s_over, s_prev;
    __shared__ unsigned long long s_best;
    const float n_max = *p.n_max;
    const float cmax = bound_c(*p.u_max, n_max);
    const size_t seg0 = static_cast<size_t>(row) * nseg;

    // chunk maxima and list lengths of every step, once
    if (threadIdx.x == 0) {
        mbar_init(&s_bar, 1);
        fence_mbar_init();
    }
    for (int i = threadIdx.x; i < nseg; i += kThreads) {
        s_cm[i] = p.cmax[seg0 + i];
        s_cn[i] = p.cand_n[seg0 + i];
    }
    __syncthreads();
    // every list of this request into shared memory by bulk copies (each
    // list padded to an even length so that copies are 16-byte multiples)
    if (threadIdx.x == 0) {
        int run = 0;
        for (int i = 0; i < nseg; ++i) {
            s_soff[i] = run;
            run += (min(s_cn[i], kSegCap) + 1) & ~1;
        }
        s_soff[nseg] = run;
        s_staged = run <= kStageEntries;
        if (s_staged && run > 0) {
            mbar_arrive_expect_tx(&s_bar, static_cast<uint32_t>(run) * 8u);
            for (int i = 0; i < nseg; ++i) {
                const uint32_t n = static_cast<uint32_t>(s_soff[i + 1] - s_soff[i]) * 8u;
                if (n) bulk_load(s_list + s_soff[i], p.cand + (seg0 + i) * kSegCap, n, &s_bar);
            }
        }
    }
    __syncthreads();
    if (s_staged && s_soff[nseg] > 0) {
        const bool ok = mbar_wait(&s_bar, 0);
        if (!__syncthreads_and(ok) && threadIdx.x == 0) set_status(p.dev_status, SDM_DEV_TIMEOUT);
        for (int i = threadIdx.x; i < nseg; i += kThreads) {   // the padding slot is not an id
            const int n = min(s_cn[i], kSegCap);
            if (s_soff[i] + n < s_soff[i + 1]) s_list[s_soff[i] + n] = make_uint2(0xffffffffu, 0u);
        }
        __syncthreads();
    }
    for (int d = warp; d < p.B; d += kWarps) {
        float m = -INFINITY;
        for (int c = lane; c < nc; c += 32) m = fmaxf(m, s_cm[d * nc + c]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) s_lmax[d] = m;
    }
    __syncthreads();
    // the likely winners of every step (L >= max - C_max): their W^T rows, and
    // their U rows for the next step, into L2
    if (s_staged) {
        for (int d = 0; d < p.B; ++d) {
            const float cut = s_lmax[d] - cmax;
            for (int t = s_soff[d * nc] + threadIdx.x; t < s_soff[(d + 1) * nc]; t += kThreads) {
                const uint2 en = s_list[t];
                if (en.x >= static_cast<uint32_t>(p.V) || __uint_as_float(en.y) < cut) continue;
                prefetch_row_l2(p.Wt, en.x, p.r);
                if (d + 1 < p.B) prefetch_row_l2(p.U, en.x, p.r);
            }
        }
    }
    int prev = p.anchor[row];
    if (prev < 0 || prev >= p.V) {
        if (threadIdx.x == 0) set_status(p.dev_status, SDM_DEV_BAD_TOKEN);
        prev = 0;
    }
    for (int d = 1; d <= p.B; ++d) {
        const int ds = (d - 1) * nc;
        if (warp == 0 && lane * 8 < p.r)
            s_u[lane] = __ldg(reinterpret_cast<const uint4*>(p.U + static_cast<size_t>(prev) * p.r) + lane);
        if (warp == 1) {   // list offsets of this step (exclusive scan over the chunks)
            int over = 0, run = 0;
            for (int c0 = 0; c0 < nc; c0 += 32) {
                const int c = c0 + lane;
                const int n = c < nc ? s_cn[ds + c] : 0;
                over |= __any_sync(0xffffffffu, n > kSegCap);
                int x = n;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int y = __shfl_up_sync(0xffffffffu, x, o);
                    if (lane >= o) x += y;
                }
                if (c < nc) s_off[c] = run + x - n;
                run += __shfl_sync(0xffffffffu, x, 31);
            }
            if (lane == 0) {
                s_off[nc] = run;
                s_over = over;
                s_n = 0;
                s_best = 0ull;
            }
        }
        __syncthreads();
        const float C = bound_c(p.u_norm[prev], n_max);
        const float lmax = s_lmax[d - 1];
        const float tall = threshold(lmax, C);   // every id that can win has L >= tall
        // stage this step's ids with L >= tall (from the lists, or from the row)
        int m = 0;
        if (!s_over) {
            if (s_staged) {
                for (int t = s_soff[ds] + threadIdx.x; t < s_soff[ds + nc]; t += kThreads) {
                    const uint2 en = s_list[t];
                    if (en.x < static_cast<uint32_t>(p.V) && __uint_as_float(en.y) >= tall) {
                        const int slot = atomicAdd(&s_n, 1);
                        if (slot < kPickCap) s_cand[slot] = en;
                    }
                }
            } else {
                const int total = s_off[nc];
                for (int t = threadIdx.x; t < total; t += kThreads) {
                    int c = 0;
                    while (s_off[c + 1] <= t) ++c;
                    const uint2 en = p.cand[(seg0 + ds + c) * kSegCap + (t - s_off[c])];
                    if (__uint_as_float(en.y) >= tall) {
                        const int slot = atomicAdd(&s_n, 1);
                        if (slot < kPickCap) s_cand[slot] = en;
                    }
                }
            }
            __syncthreads();
            m = s_n;
            if (m > kPickCap) {
                if (threadIdx.x == 0) s_over = 1;
                __syncthreads();
            }
        }
        float ub[8];
        unpack<0>(lane * 8 < p.r ? s_u[lane] : make_uint4(0, 0, 0, 0), ub);
        if (!s_over) {
            // Any id that can reach the maximum z* has L >= z* - C.  Round 1
            // scores the staged ids with L >= max - C (z* >= their best z1);
            // round 2 those with z1 - C <= L < max - C.
            float lo = threshold(lmax, 0.5f * C), hi = INFINITY;
            for (int round = 0; round < 2; ++round) {
                if (threadIdx.x == 0) s_m = 0;
                __syncthreads();
                for (int t = threadIdx.x; t < m; t += kThreads) {
                    const float lv = __uint_as_float(s_cand[t].y);
                    if (lv >= lo && lv < hi) s_ids[atomicAdd(&s_m, 1)] = s_cand[t];
                }
                __syncthreads();
                unsigned long long b = score_staged(p, s_ids, s_m, ub, warp, lane);
                b = warp_max_u64(b);
                if (lane == 0 && b) atomicMax(&s_best, b);
                __syncthreads();
                const unsigned long long k = s_best;
                hi = lo;
                lo = threshold(k ? key_value(k) : -INFINITY, 0.5f * C);
                if (!(lo < hi)) break;
            }
        } else {
            // a list overflowed: scan the whole row in batches (exact for any input)
            const uint4* src = reinterpret_cast<const uint4*>(row_ptr(p, row, d, 0));
            const int nv = p.V / VEC;
            for (int c0 = 0; c0 < nv; c0 += kPickCap / VEC) {
                if (threadIdx.x == 0) s_m = 0;
                __syncthreads();
                for (int i = c0 + threadIdx.x; i < min(nv, c0 + kPickCap / VEC); i += kThreads) {
                    float v[VEC];
                    unpack<FP32>(__ldg(src + i), v);
#pragma unroll
                    for (int q = 0; q < VEC; ++q)
                        if (v[q] >= tall)
                            s_ids[atomicAdd(&s_m, 1)] = make_uint2(static_cast<uint32_t>(i * VEC + q), __float_as_uint(v[q]));
                }
                __syncthreads();
                unsigned long long b = score_staged(p, s_ids, s_m, ub, warp, lane);
                b = warp_max_u64(b);
                if (lane == 0 && b) atomicMax(&s_best, b);
                __syncthreads();
            }
        }
        if (threadIdx.x == 0) {
            int y = static_cast<int>(key_token(s_best));
            if (y < 0 || y >= p.V) {
                set_status(p.dev_status, SDM_DEV_BAD_TOKEN);
                y = 0;
            }
            p.tokens[static_cast<size_t>(row) * p.B + (d - 1)] = y;
            s_prev = y;
        }
        __syncthreads();
        prev = s_prev;
    }
}

// --- prepared tables ---------------------------------------------------------

// W^T [V, r] from W [r, V] through 32 x 32 shared tiles.
__global__ void transpose_kernel(const uint16_t* W, int r, int V, uint16_t* Wt) {
    __shared__ uint16_t tile[32][33];
    const int v0 = blockIdx.x * 32, j0 = blockIdx.y * 32;
    for (int y = threadIdx.y; y < 32; y += blockDim.y) {
        const int j = j0 + y, v = v0 + threadIdx.x;
        if (j < r && v < V) tile[y][threadIdx.x] = W[static_cast<size_t>(j) * V + v];
    }
    __syncthreads();
    for (int y = threadIdx.y; y < 32; y += blockDim.y) {
        const int v = v0 + y, j = j0 + threadIdx.x;
        if (j < r && v < V) Wt[static_cast<size_t>(v) * r + j] = tile[threadIdx.x][y];
    }
}

// Euclidean norms of the rows of a [V, r] bf16 table, rounded up to fp32
// (accumulated in fp64, so the stored value bounds the exact norm).  With
// max_out, the maximum over rows is also formed (atomic max on the bits of a
// non-negative float orders like the value).
__global__ void row_norm_kernel(const uint16_t* T, int V, int r, float* out, unsigned int* max_out) {
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (warp >= V) return;
    double s = 0.0;
    for (int j = lane; j < r; j += 32) {
        const double x = static_cast<double>(bf16_bits_to_float(T[static_cast<size_t>(warp) * r + j]));
        s += x * x;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) {
        const float n = __double2float_ru(__dsqrt_ru(s));
        if (out) out[warp] = n;
        if (max_out) atomicMax(max_out, __float_as_uint(n));
    }
}

}  // namespace

int pruned_chunks(int V, int l_fp32) {
    const int per = kChunkBytes / (l_fp32 ? 4 : 2);
    return (V + per - 1) / per;
}

cudaError_t launch_chain_pruned(const PrunedParams& p, cudaStream_t s) {
    const long long items = static_cast<long long>(p.R) * p.B * p.n_chunks;
    const int grid = static_cast<int>(items < 8LL * num_sms() ? items : 8LL * num_sms());
    if (p.l_fp32)
        chain_scan_kernel<1><<<grid, kThreads, 0, s>>>(p);
    else
        chain_scan_kernel<0><<<grid, kThreads, 0, s>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const size_t smem = static_cast<size_t>(kStageEntries) * 8 + static_cast<size_t>(p.B) * p.n_chunks * 12 + 16;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(chain_pick_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             200 * 1024);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(chain_pick_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    if (p.l_fp32)
        chain_pick_kernel<1><<<p.R, kThreads, smem, s>>>(p);
    else
        chain_pick_kernel<0><<<p.R, kThreads, smem, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_markov_prepare(const uint16_t* U, const uint16_t* W, int V, int r, uint16_t* Wt, float* u_norm,
                                  float* n_max, float* u_max, cudaStream_t s) {
    transpose_kernel<<<dim3((V + 31) / 32, (r + 31) / 32), dim3(32, 8), 0, s>>>(W, r, V, Wt);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = cudaMemsetAsync(n_max, 0, sizeof(float), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(u_max, 0, sizeof(float), s);
    if (e != cudaSuccess) return e;
    const int blocks = (V * 32 + 255) / 256;
    row_norm_kernel<<<blocks, 256, 0, s>>>(U, V, r, u_norm, reinterpret_cast<unsigned int*>(u_max));
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    row_norm_kernel<<<blocks, 256, 0, s>>>(Wt, V, r, nullptr, reinterpret_cast<unsigned int*>(n_max));
    return cudaGetLastError();
}

}  // namespace sdm
