// schedule_pack.cuh - the budget scheduler and the ragged pack as one-block
// device functions: run by their own one-CTA kernels, or by an extra CTA of
// the greedy chain's scan, which then needs no SM of its own for them (the
// scan fills every SM; a separate kernel could only start as it drains).
#pragma once
#include "device.cuh"
#include "internal.h"

namespace sdm {

constexpr int kSchedThreads = 1024;   // most threads a scheduler block runs with
constexpr int kPackThreads = 256;     // the pack block's threads

// Dynamic shared memory of schedule_block: n_pad sort keys, part_n partial
// sums, R counters, R * gamma survivals, n_pad + 1 screens.
__host__ __device__ inline size_t schedule_smem_bytes(int R, int gamma, int n_pad, int part_n) {
    return static_cast<size_t>(n_pad) * 8 + static_cast<size_t>(part_n) * 8 + static_cast<size_t>(R) * 4 +
           static_cast<size_t>(R) * gamma * 4 + (static_cast<size_t>(n_pad) + 1) * 4;
}

// The budget scheduler of one CTA ([DSpark notes] sec. 5.2: survival
// products, the survivals ranked (S desc, request asc, position asc), the
// greedy prefix while E(m) / cost strictly improves): the whole block takes
// part, blockDim.x threads (any count, at most part_n).  sk: dynamic shared
// memory of schedule_smem_bytes(R, gamma, n_pad, part_n) bytes.
__device__ __forceinline__ void schedule_block(const float* conf, int R, int gamma, const double* cost,
                                               float* survival, int32_t* budget, double* expected,
                                               int32_t* total_tokens, int n_pad, unsigned long long* sk,
                                               int part_n) {
    unsigned long long* part = sk + n_pad;                   // part_n partial sums
    int* cnt = reinterpret_cast<int*>(part + part_n);         // R counters
    float* s_surv = reinterpret_cast<float*>(cnt + R);       // R * gamma confidences, then survivals
    float* fq = s_surv + R * gamma;                          // n_pad + 1 fp32 screens of f(m)
    __shared__ int m_star;
    __shared__ int n_cand;
    const int tid = threadIdx.x, nt = blockDim.x;
    const int n = R * gamma;
    const float floor_s = 1.0f / 262144.0f;                 // 2^-18

    // all confidences in one coalesced pass (no dependent global loads below)
    for (int t = tid; t < n; t += nt) s_surv[t] = conf[t];
    for (int i = tid; i < R; i += nt) cnt[i] = 0;
    for (int t = n + tid; t < n_pad; t += nt) sk[t] = 0ull;
    if (tid == 0) {
        m_star = 0x7fffffff;
        n_cand = 0;
    }
    __syncthreads();
    // survival S_{i,k} = S_{i,k-1} c_{i,k}, fp32, left to right
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
    for (int t = tid; t < n; t += nt) survival[t] = s_surv[t];
    // bitonic sort, descending (S desc, then request asc, position asc)
    if (n_pad <= nt) {
        // one key per thread: partners closer than a warp swap by shuffle
        unsigned long long key = tid < n_pad ? sk[tid] : 0ull;
        for (int size = 2; size <= n_pad; size <<= 1) {
            for (int stride = size >> 1; stride > 0; stride >>= 1) {
                unsigned long long other;
                if (stride >= 32) {
                    if (tid < n_pad) sk[tid] = key;
                    __syncthreads();
                    other = tid < n_pad ? sk[tid ^ stride] : 0ull;
                    __syncthreads();
                } else {
                    other = __shfl_xor_sync(0xffffffffu, key, stride);
                }
                const bool desc = (tid & size) == 0, lower = (tid & stride) == 0;
                key = (desc == lower) ? umax64(key, other) : (key < other ? key : other);
            }
        }
        if (tid < n_pad) sk[tid] = key;
        __syncthreads();
    } else {
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
    }
    // number of ranked survivals
    for (int t = tid; t < n_pad; t += nt)
        if (sk[t] != 0ull && (t + 1 == n_pad || sk[t + 1] == 0ull)) n_cand = t + 1;
    __syncthreads();
    const int M = n_cand;
    // exact prefix sums: a survival >= 2^-18 is an integer multiple of 2^-41
    const int per = (n_pad + nt - 1) / nt;
    unsigned long long local = 0;
    for (int q = 0; q < per; ++q) {
        const int t = tid * per + q;
        if (t < M) local += static_cast<unsigned long long>(ldexpf(__uint_as_float(static_cast<uint32_t>(sk[t] >> 32)), 41));
    }
    // exclusive block scan of the thread partials (warp shuffles, then the
    // 32 warp totals by warp 0); integer adds are exact in any order
    {
        const int lane = tid & 31, warp = tid >> 5;
        unsigned long long x = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) part[warp] = x;
        __syncthreads();
        if (warp == 0) {   // lanes past the last warp hold 0
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
    // f(m) = E(m) / cost[R + m]; the greedy stops at the first m whose next
    // survival does not raise f strictly (compared as fp64 quotients).  Each
    // f(m) is first formed in fp32 (relative error < 2^-22); when two
    // neighbours differ by more than 2^-20 relative, the fp64 quotients
    // order the same way, and only closer pairs are divided in fp64 (fp64
    // throughput is low on this part).
    const double two_m41 = 4.547473508864641e-13;   // 2^-41
    const unsigned long long base = static_cast<unsigned long long>(R) << 41;
    auto f32_of = [&](unsigned long long e_int, int m) {
        return __fdiv_rn(__ull2float_rn(e_int) * 4.547473508864641e-13f, __double2float_rn(cost[R + m]));
    };
    {
        unsigned long long run = part[tid];
        for (int q = 0; q < per; ++q) {
            const int m = tid * per + q;              // E(m) uses the first m survivals
            if (m >= M) break;
            fq[m] = f32_of(base + run, m);
            run += static_cast<unsigned long long>(ldexpf(__uint_as_float(static_cast<uint32_t>(sk[m] >> 32)), 41));
            if (m == M - 1) fq[M] = f32_of(base + run, M);
        }
    }
    __syncthreads();
    {
        unsigned long long run = part[tid];
        for (int q = 0; q < per; ++q) {
            const int m = tid * per + q;
            if (m >= M) break;
            const unsigned long long s_int =
                static_cast<unsigned long long>(ldexpf(__uint_as_float(static_cast<uint32_t>(sk[m] >> 32)), 41));
            const float g0 = fq[m], g1 = fq[m + 1];
            bool up;
            if (g1 > g0 * 1.00000095367431640625f) {
                up = true;
            } else if (g1 < g0 * 0.99999904632568359375f) {
                up = false;
            } else {
                const double f0 = __ddiv_rn(static_cast<double>(base + run) * two_m41, cost[R + m]);
                const double f1 = __ddiv_rn(static_cast<double>(base + run + s_int) * two_m41, cost[R + m + 1]);
                up = f1 > f0;
            }
            if (!up) atomicMin(&m_star, m);
            run += s_int;
        }
    }
    __syncthreads();
    const int ms = (m_star == 0x7fffffff) ? M : m_star;
    for (int t = tid; t < ms; t += nt) {
        const uint32_t id = ~static_cast<uint32_t>(sk[t] & 0xffffffffull);
        atomicAdd(&cnt[id / gamma], 1);
    }
    __syncthreads();
    for (int i = tid; i < R; i += nt) budget[i] = cnt[i];
    if (tid == 0) {
        // prefix at m*: the owning thread's exclusive prefix plus its first entries
        const int owner = ms / per < nt ? ms / per : nt - 1;
        unsigned long long sum = part[owner];
        for (int t = owner * per; t < ms; ++t)
            sum += static_cast<unsigned long long>(ldexpf(__uint_as_float(static_cast<uint32_t>(sk[t] >> 32)), 41));
        *expected = static_cast<double>((static_cast<unsigned long long>(R) << 41) + sum) * 4.547473508864641e-13;
        *total_tokens = R + ms;
    }
}

// The ragged front-pack of one CTA of kPackThreads threads ([SGLang] "ragged
// verify"): window i = the anchor and budget[i] (or gamma) drafts, offsets by
// a block scan, the packed total rounded up to the smallest tier that holds
// it; draft may be NULL (the layout alone, draft rows -1).
__device__ __forceinline__ void pack_block(const int32_t* anchor, const int32_t* draft, const int32_t* budget, int R,
                                           int gamma, const int32_t* tiers, int n_tiers, int strict, int32_t* cu,
                                           int32_t* ptok, int32_t* preq, int32_t* ppos, int capacity, int32_t* tier,
                                           int32_t* dev_status) {
    __shared__ int warp_sum[32];
    __shared__ int s_total, s_tier;
    __shared__ int s_start[kPackThreads], s_n[kPackThreads];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int carry = 0;
    // exclusive scan of (n_i + 1), kPackThreads requests per pass
    for (int base = 0; base < R; base += kPackThreads) {
        const int i = base + tid;
        int n = 0;
        if (i < R) {
            n = budget ? budget[i] : gamma;
            if (n < 0 || n > gamma) {
                set_status(dev_status, SDM_DEV_BAD_WINDOW);
                n = n < 0 ? 0 : gamma;
            }
        }
        const int len = (i < R) ? n + 1 : 0;
        int x = len;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_sum[warp] = x;
        __syncthreads();
        if (warp == 0) {   // lanes past the last warp hold 0
            int w = lane < kPackThreads / 32 ? warp_sum[lane] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += y;
            }
            warp_sum[lane] = w;
        }
        __syncthreads();
        const int incl = x + (warp > 0 ? warp_sum[warp - 1] : 0) + carry;
        const int start = incl - len;
        if (i < R) cu[i] = start;
        s_start[tid] = start;
        s_n[tid] = (i < R) ? n : -1;
        __syncthreads();
        // one (request, position) pair per thread: the loads are independent
        const int per = gamma + 1;
        const int chunk_r = min(kPackThreads, R - base);
        for (int idx = tid; idx < chunk_r * per; idx += kPackThreads) {
            const int il = idx / per, p = idx - il * per;
            if (p > s_n[il]) continue;
            const int row = s_start[il] + p;
            if (row < 0 || row >= capacity) {
                set_status(dev_status, SDM_DEV_CAPACITY);
                continue;
            }
            const int ig = base + il;
            // without drafts (a layout for sdm_draft_chain_packed to fill) the draft rows hold -1
            ptok[row] = (p == 0) ? anchor[ig] : (draft ? draft[static_cast<size_t>(ig) * gamma + p - 1] : -1);
            preq[row] = ig;
            ppos[row] = p;
        }
        const int chunk_total = warp_sum[kPackThreads / 32 - 1];
        __syncthreads();
        carry += chunk_total;
    }
    // the smallest tier that holds the total (the tiers are read in parallel)
    if (tid == 0) s_tier = 0x7fffffff;
    __syncthreads();
    for (int q = tid; q < n_tiers; q += kPackThreads) {
        const int tq = tiers[q];
        if (tq >= carry) atomicMin(&s_tier, tq);
    }
    __syncthreads();
    if (tid == 0) {
        cu[R] = carry;
        int t = s_tier;
        if (t == 0x7fffffff) {   // above every tier: run uncaptured, or an error in strict mode
            t = carry;
            set_status(dev_status, strict ? SDM_DEV_TIER_OVERFLOW : SDM_DEV_TIER_UNCAPTURED);
        }
        s_total = carry;
        s_tier = t;
        *tier = t;
    }
    __syncthreads();
    // every row past the packed total (the tier padding and the rest of the
    // buffer) holds -1, so a consumer may read the whole buffer safely
    for (int row = s_total + tid; row < capacity; row += kPackThreads) {
        ptok[row] = -1;
        preq[row] = -1;
        ppos[row] = -1;
    }
}

}  // namespace sdm
