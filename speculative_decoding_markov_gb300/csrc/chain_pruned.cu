// chain_pruned.cu - the greedy Markov-head chain without the dense projection.
//
// Greedy drafting needs y_d = argmax_v z_d[v], z_d = fp32(L_d) + U[y_{d-1}] W.
// The Markov term of a previous token y is bounded over the whole vocabulary:
// |U[y] . W[:, v]| <= c(y) for every v, with c(y) from the prepared tables
// (the exact maximum max_v |U[y] . W[:, v]|, formed once on the tensor cores,
// plus slack for rounding).  So no id with L_d[v] < max_v L_d[v] - 2 c(y) can
// be the argmax.  Only that threshold depends on the previous token, and
// c(y) <= c_max = max_y c(y), which splits the chain into two launches:
//
//   chain_scan_kernel  (every (request, step) row in parallel, HBM-bound)
//     a persistent grid walks 32 KB chunks of the rows of L; each CTA holds
//     its chunk in registers, reduces the chunk maximum m_c and lists every
//     id with L >= m_c - 2 c_max.  L is read from HBM exactly once.
//   chain_pick_kernel  (one CTA per request, the B dependent steps)
//     one warp per step keeps the listed ids with L >= max_v L_d - 2 c_max
//     (the ids any previous token can need) and copies their W^T rows and U
//     rows into shared memory; then the CTA walks the steps: step d scores
//     the ids with L >= max - 2 c(y_{d-1}) exactly,
//     z = L + U[y_{d-1}] . W^T[v] (fp32), and takes the (z desc, id asc)
//     winner; one warp walks these steps with no block barrier.  Steps whose
//     lists overflowed, or whose ids do not fit in shared memory, score from
//     global memory with every warp (a full-row scan when a list overflowed).
//
// The result equals the dense argmax bit for bit: the kept set contains every
// id that can reach the maximum and the kept ids are scored exactly.
#include <cuda_bf16.h>

#include "device.cuh"
#include "internal.h"
#include "schedule_pack.cuh"

namespace sdm {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
static_assert(kMaxTopK <= kWarps, "the scan's k-th threshold ranks the warps' maxima");
static_assert(kThreads == kPackThreads, "the scan's front CTA runs the pack block");
constexpr int kListHead = 32;   // list entries the pick kernel loads with the list length

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

// Maximum of one 16-byte vector: a packed bf16x2 tree, two conversions at the end.
template <int FP32>
__device__ __forceinline__ float vec_max(const uint4& x) {
    if (FP32)
        return fmaxf(fmaxf(__uint_as_float(x.x), __uint_as_float(x.y)), fmaxf(__uint_as_float(x.z), __uint_as_float(x.w)));
    __nv_bfloat162 w[4];
    memcpy(w, &x, 16);
    const __nv_bfloat162 m = __hmax2(__hmax2(w[0], w[1]), __hmax2(w[2], w[3]));
    uint32_t b;
    memcpy(&b, &m, 4);
    return fmaxf(__uint_as_float(b << 16), __uint_as_float(b & 0xffff0000u));
}

// Start of row (request `row`, step d) of L at id v.
__device__ __forceinline__ const uint8_t* row_ptr(const PrunedParams& p, int row, int d, int v) {
    const size_t esz = p.l_fp32 ? 4 : 2;
    return static_cast<const uint8_t*>(p.L) + ((static_cast<size_t>(row) * p.B + (d - 1)) * p.V + v) * esz;
}

// The candidate threshold below a row maximum m for a Markov bound c.
__device__ __forceinline__ float threshold(float m, float c) { return markov_cut(m, c); }

// ---------------------------------------------------------------------------
// A: candidate lists of every (request, step, chunk)
// ---------------------------------------------------------------------------
// Work item = kChunkBytes of one row L_d; row-major items, a persistent grid
// strides over them.  Each thread holds 8 16-byte vectors of the chunk in
// registers (all eight loads in flight at once; an explicit L2 prefetch of the
// next item measured slower on this part), the chunk maximum m_c is reduced
// over the CTA, and every id with L >= m_c - 2 c_max is listed.
// m_c <= max_v L_d[v] and c(y) <= c_max, so the list holds every id an exact
// step can need.
template <int FP32>
__global__ void __launch_bounds__(kThreads, 4) chain_scan_kernel(const PrunedParams p) {
    constexpr int VEC = FP32 ? 4 : 8;
    constexpr int ESZ = FP32 ? 4 : 2;
    constexpr int VPT = kChunkBytes / 16 / kThreads;        // vectors per thread
    constexpr int CHUNK_IDS = kChunkBytes / ESZ;
    __shared__ float s_wmax[kWarps];
    __shared__ int s_cnt[2];   // by item parity: a slot is reset two items after its last read
    extern __shared__ unsigned long long s_front[];   // the scheduler's arrays (the front CTA's only)
    pdl_wait();
    pdl_trigger();
    if (p.fr.on && blockIdx.x == 0) {
        // the front CTA (dispatched first): budgets, then the windows' layout
        // from them (the block barrier orders the budgets' global writes
        // before the pack reads them)
        schedule_block(p.fr.conf, p.R, p.B, p.fr.cost, p.fr.survival, p.fr.budget, p.fr.expected,
                       p.fr.total_tokens, p.fr.n_pad, s_front, kThreads);
        __syncthreads();
        pack_block(p.anchor, nullptr, p.fr.use_budget ? p.fr.budget : nullptr, p.R, p.B, p.fr.tiers, p.fr.n_tiers,
                   p.fr.strict, p.fr.cu, p.fr.ptok, p.fr.preq, p.fr.ppos, p.fr.capacity, p.fr.tier, p.dev_status);
        return;
    }
    const int g0 = p.fr.on ? 1 : 0;
    const int G = static_cast<int>(gridDim.x) - g0;   // the scanning CTAs
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nc = p.n_chunks;
    const int items = p.R * p.B * nc;       // <= 2^30 (checked by the host)
    const float cmax = *p.c_max;
    // item it = rs * nc + c, rs = request * B + (d - 1): walk (rs, c) by the
    // grid stride without dividing per item
    int it = static_cast<int>(blockIdx.x) - g0;
    int rs = it / nc, c = it - rs * nc;
    const int srs = G / nc, sc = G - srs * nc;
    const uint8_t* L = static_cast<const uint8_t*>(p.L);
    for (int par = 0; it < items; par ^= 1) {
        int nrs = rs + srs, ncc = c + sc;
        if (ncc >= nc) {
            ncc -= nc;
            ++nrs;
        }
        const int v0 = c * CHUNK_IDS;
        const int n_vec = (min(p.V, v0 + CHUNK_IDS) - v0) / VEC;
        const uint4* src = reinterpret_cast<const uint4*>(L + (static_cast<size_t>(rs) * p.V + v0) * ESZ);
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
        if (threadIdx.x == 0) s_cnt[par] = 0;
        __syncthreads();
        float mc = s_wmax[0];
#pragma unroll
        for (int w = 1; w < kWarps; ++w) mc = fmaxf(mc, s_wmax[w]);
        // the value the list is cut below: the chunk maximum for the argmax;
        // for a top-k the k-th largest of the warps' maxima (k <= kWarps: the
        // k warps with the largest maxima hold k distinct values at or above
        // it, so it is a lower bound on the chunk's k-th largest value; -inf
        // when fewer than k warps hold a value)
        float theta = mc;
        if (p.kth > 1) {   // lane w < kWarps ranks warp w's maximum
            const float x0 = s_wmax[lane & (kWarps - 1)];
            int gt = 0, ge = 0;
#pragma unroll
            for (int u = 0; u < kWarps; ++u) {
                gt += s_wmax[u] > x0 ? 1 : 0;
                ge += s_wmax[u] >= x0 ? 1 : 0;
            }
            const unsigned at = __ballot_sync(0xffffffffu, lane < kWarps && gt < p.kth && ge >= p.kth);
            theta = at ? __shfl_sync(0xffffffffu, x0, __ffs(at) - 1) : -INFINITY;
        }
        const float T = threshold(theta, cmax);
        const int seg = rs * nc + c;
        uint2* out = p.cand + static_cast<size_t>(seg) * kSegCap;
        if (tmax >= T) {   // only threads holding a candidate
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int i = threadIdx.x + k * kThreads;
                if (i >= n_vec || vec_max<FP32>(x[k]) < T) continue;   // (a padded vector is never listed)
                float v[VEC];
                unpack<FP32>(x[k], v);
#pragma unroll
                for (int q = 0; q < VEC; ++q) {
                    if (v[q] >= T) {
                        const int slot = atomicAdd(&s_cnt[par], 1);
                        if (slot < kSegCap)
                            out[slot] = make_uint2(static_cast<uint32_t>(v0 + i * VEC + q), __float_as_uint(v[q]));
                    }
                }
            }
        }
        __syncthreads();
        const int cnt = s_cnt[par];
        if (threadIdx.x == 0) {
            p.cand_n[seg] = cnt;          // the true count: above kSegCap the list is incomplete
            p.cmax[seg] = mc;
        }
        // the head of the list (kListHead entries) is always written, so that
        // the pick kernel's speculative head loads hit L2
        if (threadIdx.x >= cnt && threadIdx.x < kListHead) out[threadIdx.x] = make_uint2(0xffffffffu, 0u);
        it += G;
        rs = nrs;
        c = ncc;
    }
}

// ---------------------------------------------------------------------------
// B: the B dependent steps of each request
// ---------------------------------------------------------------------------
constexpr int kGroup = 8;              // candidates a warp scores per round (global path)
constexpr int kPickCap = 1024;         // ids per scoring batch of the global path
constexpr int kRowCapMax = 192;        // staged candidates (W^T row + U row each); < 256
constexpr int kPickSmem = 200 * 1024;  // dynamic shared memory of the pick kernel

struct PickLayout {
    uint32_t st_key, st_c, st_w, st_u, total;
    int cap, rs;   // staged candidates, row stride (elements)
};

__host__ __device__ inline uint32_t al16(uint32_t x) { return (x + 15u) & ~15u; }

// Dynamic shared memory: list prefix sums [B][nc + 1]; a pool of cap staged
// candidates shared by the steps: (id, L) keys, bounds c(id), W^T rows and U
// rows (plus U[anchor] as row cap), rows padded by 16 bytes so that the
// tensor-core fragment loads of eight rows fall in distinct banks.
__host__ __device__ inline PickLayout pick_layout(int B, int nc, int r) {
    PickLayout l;
    l.rs = r + 8;
    const uint32_t fixed = al16(static_cast<uint32_t>(B) * static_cast<uint32_t>(nc + 1) * 4u);
    const uint32_t row = 2u * static_cast<uint32_t>(l.rs);
    const uint32_t per = 8u + 4u + 2u * row;
    int cap = static_cast<int>((kPickSmem - fixed - row - 64u) / per);
    cap = cap < kRowCapMax ? cap : kRowCapMax;
    l.cap = cap;
    l.st_key = fixed;
    l.st_c = al16(l.st_key + static_cast<uint32_t>(cap) * 8u);
    l.st_w = al16(l.st_c + static_cast<uint32_t>(cap) * 4u);
    l.st_u = l.st_w + static_cast<uint32_t>(cap) * row;
    l.total = l.st_u + static_cast<uint32_t>(cap + 1) * row;
    return l;
}

// U row slice of a lane: elements [8 lane, 8 lane + 8) of a row that may sit
// in shared or global memory (generic address); zero past r.
__device__ __forceinline__ void load_ub(const uint16_t* urow, int lane, int r, float (&ub)[8]) {
    const uint4 u = lane * 8 < r ? *reinterpret_cast<const uint4*>(urow + lane * 8) : make_uint4(0, 0, 0, 0);
    unpack<0>(u, ub);
}

// U[y] . w for the lane slices, summed over the warp (every lane gets the sum).
__device__ __forceinline__ float warp_dot(const uint4& w, const float (&ub)[8]) {
    float a[8];
    unpack<0>(w, a);
    float acc = 0.f;
#pragma unroll
    for (int q = 0; q < 8; ++q) acc = fmaf(a[q], ub[q], acc);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    return acc;
}

// Global path: warp-cooperative exact scores of staged ids; a warp scores
// kGroup ids per round with all their W^T row loads in flight.
__device__ __forceinline__ unsigned long long score_global(const PrunedParams& p, const uint2* ids, int n,
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
#pragma unroll
        for (int j = 0; j < kGroup; ++j) {
            const float dot = warp_dot(wv[j], ub);
            if (cd[j].x < static_cast<uint32_t>(p.V))
                best = umax64(best, argmax_key(__uint_as_float(cd[j].y) + dot, cd[j].x));   // fp32(L) + Markov
        }
    }
    return best;
}

// Segment holding entry t of a step's concatenated lists: the largest c with
// pref[c] <= t (pref[0] = 0 <= t < pref[nc]).
__device__ __forceinline__ int segment_of(const int* pref, int nc, int t) {
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

// Four (x4) or two (x2) 8 x 8 bf16 matrices from shared memory, one 16-byte
// row address per lane (lanes 8m..8m+7 address matrix m); thread t receives
// row t / 4, elements 2 (t % 4) and 2 (t % 4) + 1 of each matrix.
__device__ __forceinline__ void ldmatrix_x4(const uint16_t* p, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldmatrix_x2(const uint16_t* p, uint32_t& r0, uint32_t& r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(smem_u32(p)));
}

// D += A B for one m16n8k16 tile: bf16 inputs, fp32 accumulation (the
// register layouts of A, B and D are those the PTX ISA gives for this shape).
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Draft token y of position d0 + 1 (0-based d0) of request `row`: the
// tokens array and, when a ragged layout is given, its row cu[row] + 1 + d0
// if the request's window holds it (pk0 = cu[row], pkn = its window).
__device__ __forceinline__ void emit_token(const PrunedParams& p, int row, int d0, int y, int pk0, int pkn) {
    p.tokens[static_cast<size_t>(row) * p.B + d0] = y;
    if (p.pack_tok && d0 < pkn) {
        const int prow = pk0 + 1 + d0;
        if (prow >= 0 && prow < p.pack_cap)
            p.pack_tok[prow] = y;
        else
            set_status(p.dev_status, SDM_DEV_CAPACITY);
    }
}

template <int FP32>
__global__ void __launch_bounds__(kThreads, 1) chain_pick_kernel(const PrunedParams p) {
    constexpr int VEC = FP32 ? 4 : 8;
    constexpr int kBatch = 4;   // list entries a lane loads at once (second round)
    constexpr int kHead = kListHead;
    const int row = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nc = p.n_chunks, B = p.B, r = p.r;
    const PickLayout lay = pick_layout(B, nc, r);
    const int RS = lay.rs;
    extern __shared__ __align__(16) uint8_t s_dyn[];
    int* s_pref = reinterpret_cast<int*>(s_dyn);                   // [B][nc + 1] list prefix sums
    uint2* st_key = reinterpret_cast<uint2*>(s_dyn + lay.st_key);  // [cap] staged (id, L bits)
    float* st_c = reinterpret_cast<float*>(s_dyn + lay.st_c);      // c(id)
    uint16_t* st_w = reinterpret_cast<uint16_t*>(s_dyn + lay.st_w);   // [cap][RS] W^T rows
    uint16_t* st_u = reinterpret_cast<uint16_t*>(s_dyn + lay.st_u);   // [cap + 1][RS] U rows, U[anchor] last
    uint16_t* u_anchor = st_u + static_cast<size_t>(lay.cap) * RS;
    __shared__ float s_lmax[kMaxPickSteps];
    __shared__ int s_scnt[kMaxPickSteps];                          // staged ids of each step
    __shared__ int s_sbeg[kMaxPickSteps];                          // their first pool slot
    __shared__ int s_staged[kMaxPickSteps];                        // the step's ids sit in the pool
    __shared__ int s_over[kMaxPickSteps];                          // a list of the step overflowed
    __shared__ int s_paired[kMaxPickSteps];                        // the step has pair scores
    __shared__ int s_toff[kMaxPickSteps + 1];                      // first tensor tile of each step
    __shared__ int s_aoff[kMaxPickSteps + 1];                      // first winner-table row of each step
    __shared__ unsigned long long s_rowkey[kRowCapMax + 1];        // winner key of every pair-score row
    __shared__ int s_alloc;                                        // pool slots handed out
    __shared__ float s_cprev0;
    __shared__ const uint16_t* s_urow;
    __shared__ float s_cprev;
    __shared__ uint2 s_ids[kPickCap];
    __shared__ int s_m;
    __shared__ unsigned long long s_best[2];
    __shared__ int s_pk0, s_pkn;                                    // the request's ragged window, if any
    // Before the wait, only what the scan does not write (the anchor and the
    // prepared tables), so that its latency hides under the scan's tail:
    // c_max, and U[anchor] and c(anchor) into shared memory (last warp).
    const float cmax = *p.c_max;
    bool bad_anchor = false;
    if (warp == kWarps - 1) {
        int a = p.anchor[row];
        bad_anchor = a < 0 || a >= p.V;
        if (bad_anchor) a = 0;
        if (lane * 8 < r) cp_async_16(u_anchor + lane * 8, p.U + static_cast<size_t>(a) * r + lane * 8, 16u);
        if (lane == 0) s_cprev0 = p.c_bound[a];
    }
    pdl_wait();
    pdl_trigger();
    if (bad_anchor && lane == 0) set_status(p.dev_status, SDM_DEV_BAD_TOKEN);
    const int seg0 = row * B * nc;
    // the request's ragged window (if the drafts go into one): loaded now,
    // used only when the tokens are written, so its latency hides under the
    // staging below
    int pk_c0 = 0, pk_c1 = -1;
    if (threadIdx.x == 0) {
        s_alloc = 0;
        if (p.pack_tok) {
            pk_c0 = p.pack_cu[row];
            pk_c1 = p.pack_cu[row + 1];
        }
    }
    for (int t = threadIdx.x; t <= kRowCapMax; t += kThreads) s_rowkey[t] = 0ull;
    __syncthreads();

    // One warp per step (lane = chunk): the chunk maxima, the list lengths
    // and, in the same round of loads, the head of every list; the listed
    // ids with L >= max - 2 c_max (those any previous token can need) are
    // compacted, then their W^T rows, U rows and bounds copied into shared
    // memory.  Lists longer than their loaded head take a second round.
    for (int d = warp; d < B; d += kWarps) {
        const int sg = seg0 + d * nc;
        int* pref = s_pref + d * (nc + 1);
        float m = -INFINITY;
        int over = 0, spill = 0, run = 0;
        uint2 head[kHead];
        int cn0 = 0;
        for (int c0 = 0; c0 < nc; c0 += 32) {
            const int c = c0 + lane;
            int n = 0;
            if (c < nc) {
                m = fmaxf(m, p.cmax[sg + c]);
                const int cn = p.cand_n[sg + c];
                if (c0 == 0) {
                    cn0 = cn;
                    const uint4* h = reinterpret_cast<const uint4*>(p.cand + static_cast<size_t>(sg + c) * kSegCap);
#pragma unroll
                    for (int q = 0; q < kHead / 2; ++q) {
                        const uint4 v = h[q];
                        head[2 * q] = make_uint2(v.x, v.y);
                        head[2 * q + 1] = make_uint2(v.z, v.w);
                    }
                }
                over |= cn > kSegCap;
                spill |= cn > kHead;
                n = min(cn, kSegCap);
            }
            int x = n;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            if (c < nc) pref[c] = run + x - n;
            run += __shfl_sync(0xffffffffu, x, 31);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        over = __any_sync(0xffffffffu, over);
        spill = __any_sync(0xffffffffu, spill) || nc > 32;
        __syncwarp();
        if (lane == 0) pref[nc] = run;
        const float t_all = threshold(m, cmax);
        // count, take a range of the pool, then write (a step whose ids do not
        // fit scores from global memory)
        int kept = 0, off = 0;
        bool fits = !over;
        if (fits && !spill) {
            // every list fits in its head: a keep mask per lane, a warp prefix
            // sum of the counts, then each lane writes its own entries
            uint32_t mask = 0u;
#pragma unroll
            for (int e = 0; e < kHead; ++e) {
                const bool keep = lane < nc && e < cn0 && head[e].x < static_cast<uint32_t>(p.V) &&
                                  __uint_as_float(head[e].y) >= t_all;
                mask |= keep ? (1u << e) : 0u;
            }
            const int cnt = __popc(mask);
            int x = cnt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            kept = __shfl_sync(0xffffffffu, x, 31);
            int o0 = 0;
            if (lane == 0) o0 = atomicAdd(&s_alloc, kept);
            off = __shfl_sync(0xffffffffu, o0, 0);
            fits = off + kept <= lay.cap;
            if (fits) {
                int pos = off + x - cnt;
#pragma unroll
                for (int e = 0; e < kHead; ++e)
                    if (mask & (1u << e)) st_key[pos++] = head[e];
            }
        }
        for (int pass = 0; pass < 2 && fits && spill; ++pass) {
            int pos0 = 0;
            {
                for (int t0 = 0; t0 < run; t0 += 32 * kBatch) {
                    uint2 en[kBatch];
#pragma unroll
                    for (int q = 0; q < kBatch; ++q) {   // independent loads, all in flight
                        const int t = t0 + q * 32 + lane;
                        en[q] = make_uint2(0xffffffffu, 0u);
                        if (t < run) {
                            const int c = segment_of(pref, nc, t);
                            en[q] = p.cand[static_cast<size_t>(sg + c) * kSegCap + (t - pref[c])];
                        }
                    }
#pragma unroll
                    for (int q = 0; q < kBatch; ++q) {
                        const bool keep = en[q].x < static_cast<uint32_t>(p.V) && __uint_as_float(en[q].y) >= t_all;
                        const unsigned bal = __ballot_sync(0xffffffffu, keep);
                        if (pass == 1 && keep) st_key[off + pos0 + __popc(bal & ((1u << lane) - 1u))] = en[q];
                        pos0 += __popc(bal);
                    }
                }
            }
            if (pass == 0) {
                kept = pos0;
                int o = 0;
                if (lane == 0) o = atomicAdd(&s_alloc, kept);
                off = __shfl_sync(0xffffffffu, o, 0);
                fits = off + kept <= lay.cap;
            }
        }
        __syncwarp();
        if (fits) {
            for (int j = 0; j < kept; ++j) {
                const uint32_t v = st_key[off + j].x;
                const int slot = off + j;
                if (lane * 8 < r) {
                    cp_async_16(st_w + static_cast<size_t>(slot) * RS + lane * 8, p.Wt + static_cast<size_t>(v) * r + lane * 8, 16u);
                    cp_async_16(st_u + static_cast<size_t>(slot) * RS + lane * 8, p.U + static_cast<size_t>(v) * r + lane * 8, 16u);
                }
            }
            for (int j = lane; j < kept; j += 32) cp_async_4(st_c + off + j, p.c_bound + st_key[off + j].x);
        }
        if (lane == 0) {
            s_lmax[d] = m;
            s_over[d] = over;
            s_scnt[d] = kept;
            s_sbeg[d] = off;
            s_staged[d] = fits;
        }
    }
    cp_async_wait_all();   // the staged rows and bounds, and U[anchor]
    if (threadIdx.x == 0) {
        s_pk0 = 0;
        s_pkn = -1;
        if (p.pack_tok) {
            int n = pk_c1 - pk_c0 - 1;
            if (n > B || n < 0) {
                if (n > B) set_status(p.dev_status, SDM_DEV_BAD_WINDOW);
                n = n > B ? B : -1;
            }
            s_pk0 = pk_c0;
            s_pkn = n;
        }
    }
    __syncthreads();

    // Pair scores: for every step d whose ids are staged and whose possible
    // previous tokens are too (the anchor for d = 1, the staged ids of d - 1
    // otherwise), z[d][p][j] = L_j + U[p] . W^T[j] for all pairs, as 16 x 8
    // tensor-core tiles (mma.sync, bf16 in, fp32 accumulate) spread over the
    // warps.  The chain below then only looks scores up.
    if (warp == 0) {
        // per step (lane = step): whether it gets pair scores, its tiles and
        // winner rows as exclusive prefix sums.  The winner rows always fit:
        // they number 1 + (staged ids) <= cap + 1.
        int trun = 0, arun = 0;
        for (int d0 = 0; d0 < B; d0 += 32) {
            const int d = d0 + lane;
            int tiles = 0, rows = 0;
            bool ok = false;
            if (d < B) {
                const bool prev_ok = d == 0 || s_staged[d - 1];
                const int np = d == 0 ? 1 : s_scnt[d - 1];
                const int nq = s_scnt[d];
                ok = s_staged[d] && prev_ok && nq > 0 && np > 0;
                if (ok) {
                    tiles = ((np + 15) >> 4) * ((nq + 7) >> 3);
                    rows = np;
                }
            }
            int xt = tiles, xa = rows;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int yt = __shfl_up_sync(0xffffffffu, xt, o);
                const int ya = __shfl_up_sync(0xffffffffu, xa, o);
                if (lane >= o) {
                    xt += yt;
                    xa += ya;
                }
            }
            if (d < B) {
                s_paired[d] = ok;
                s_toff[d] = trun + xt - tiles;
                s_aoff[d] = arun + xa - rows;
            }
            trun += __shfl_sync(0xffffffffu, xt, 31);
            arun += __shfl_sync(0xffffffffu, xa, 31);
        }
        if (lane == 0) {
            s_toff[B] = trun;
            s_aoff[B] = arun;
        }
    }
    __syncthreads();
    {
        const int gid = lane >> 2, tig = lane & 3;
        const int n_tiles = s_toff[B];
        for (int t = warp; t < n_tiles; t += kWarps) {
            int d = 0;
            while (s_toff[d + 1] <= t) ++d;
            const int np = d == 0 ? 1 : s_scnt[d - 1];
            const int nq = s_scnt[d];
            const int tq = (nq + 7) >> 3;
            const int lt = t - s_toff[d];
            const int p0 = (lt / tq) * 16, j0 = (lt % tq) * 8;
            const uint16_t* ubase = d == 0 ? u_anchor : st_u + static_cast<size_t>(s_sbeg[d - 1]) * RS;
            // ldmatrix addresses: A (16 x 16) as matrices (rows 0-7 | 8-15) x (k 0-7 | 8-15),
            // B (16 x 8, the W^T rows of 8 candidates) as (k 0-7 | 8-15); rows past the set repeat its last row
            const int arow = min(p0 + (lane & 7) + ((lane >> 3) & 1) * 8, np - 1);
            const uint16_t* ua = ubase + static_cast<size_t>(arow) * RS + (lane >> 4) * 8;
            const int brow = min(j0 + (lane & 7), nq - 1);
            const uint16_t* wb = st_w + static_cast<size_t>(s_sbeg[d] + brow) * RS + ((lane >> 3) & 1) * 8;
            // two independent accumulator chains (even and odd k-steps), r % 64 == 0
            float acc[4] = {0.f, 0.f, 0.f, 0.f}, acc2[4] = {0.f, 0.f, 0.f, 0.f};
            for (int k0 = 0; k0 < r; k0 += 32) {
                uint32_t a0, a1, a2, a3, b0, b1, c0, c1, c2, c3, e0, e1;
                ldmatrix_x4(ua + k0, a0, a1, a2, a3);
                ldmatrix_x2(wb + k0, b0, b1);
                ldmatrix_x4(ua + k0 + 16, c0, c1, c2, c3);
                ldmatrix_x2(wb + k0 + 16, e0, e1);
                mma_16816(acc, a0, a1, a2, a3, b0, b1);
                mma_16816(acc2, c0, c1, c2, c3, e0, e1);
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[e] += acc2[e];
            // z = fp32(L) + Markov (one rounding); the winner of each row is
            // kept as a key ordered by (z desc, id asc) whose low byte is the
            // candidate's index in the step: ids < 2^24, at most 256 per step
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int pp = p0 + gid + h * 8;
                unsigned long long best = 0ull;
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int jj = j0 + tig * 2 + e;
                    if (jj < nq) {
                        const uint2 en = st_key[s_sbeg[d] + jj];
                        const float z = __uint_as_float(en.y) + acc[h * 2 + e];
                        const unsigned long long k = (static_cast<unsigned long long>(ordered_bits(z)) << 32) |
                                                     ((0xffffffu - en.x) << 8) | static_cast<uint32_t>(jj);
                        best = umax64(best, k);
                    }
                }
                best = umax64(best, __shfl_xor_sync(0xffffffffu, best, 1));
                best = umax64(best, __shfl_xor_sync(0xffffffffu, best, 2));
                if (tig == 0 && pp < np && best) atomicMax(&s_rowkey[s_aoff[d] + pp], best);
            }
        }
    }
    __syncthreads();
    // The chain.  A step with pair scores is a table lookup (the winner for
    // the previous token's row).  A staged step without them scores from
    // shared memory; either is warp 0's alone.  A step on the global path
    // uses every warp, warp 0 handing over its state first.
    if (s_aoff[B] > 0 && s_paired[B - 1]) {
        // fast path: every step has pair scores (then every step is staged) -
        // one thread walks the winner table, the warp writes the tokens
        bool all = true;
        for (int d = 0; d < B; ++d) all = all && s_paired[d];
        if (all) {
            if (warp == 0) {
                int tokv = 0;
                if (lane == 0) {
                    int pidx = 0;
                    for (int d = 0; d < B; ++d) {
                        pidx = static_cast<int>(s_rowkey[s_aoff[d] + pidx] & 0xffu);
                        s_ids[d].x = static_cast<uint32_t>(s_sbeg[d] + pidx);
                    }
                }
                __syncwarp();
                for (int d = lane; d < B; d += 32) {
                    tokv = static_cast<int>(st_key[s_ids[d].x].x);
                    if (tokv < 0 || tokv >= p.V) {
                        set_status(p.dev_status, SDM_DEV_BAD_TOKEN);
                        tokv = 0;
                    }
                    emit_token(p, row, d, tokv, s_pk0, s_pkn);
                }
            }
            return;
        }
    }
    const uint16_t* urow = u_anchor;   // U[y_{d-1}]: shared (staged) or global
    float cprev = s_cprev0;
    int pidx = 0;                      // index of y_{d-1} among the previous step's staged ids (-1: none)
    for (int d = 1; d <= B; ++d) {
        const float lmax = s_lmax[d - 1];
        if (s_staged[d - 1]) {
            if (warp != 0) continue;
            const int sb = s_sbeg[d - 1];
            const int n = s_scnt[d - 1];
            uint32_t bid = 0xffffffffu;
            int bslot = -1;
            if (s_paired[d - 1] && pidx >= 0) {
                bslot = sb + static_cast<int>(s_rowkey[s_aoff[d - 1] + pidx] & 0xffu);
                bid = st_key[bslot].x;
            } else {
                // staged, no pair scores: score the staged ids against U[y_{d-1}]
                const float tall = threshold(lmax, cprev);   // every id that can win has L >= tall
                float ubv[8];
                load_ub(urow, lane, r, ubv);
                unsigned long long best = 0ull;
                for (int j0 = 0; j0 < n; j0 += kGroup) {
                    uint2 en[kGroup];
                    float acc[kGroup];
#pragma unroll
                    for (int jj = 0; jj < kGroup; ++jj) {   // all row loads first, then the sums
                        const int j = j0 + jj;
                        en[jj] = j < n ? st_key[sb + j] : make_uint2(0xffffffffu, 0u);
                        const bool ok = j < n && __uint_as_float(en[jj].y) >= tall && lane * 8 < r;
                        const uint4 wv = ok ? *reinterpret_cast<const uint4*>(st_w + static_cast<size_t>(sb + j) * RS + lane * 8)
                                            : make_uint4(0, 0, 0, 0);
                        float a[8];
                        unpack<0>(wv, a);
                        acc[jj] = 0.f;
#pragma unroll
                        for (int q = 0; q < 8; ++q) acc[jj] = fmaf(a[q], ubv[q], acc[jj]);
                    }
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
                        for (int jj = 0; jj < kGroup; ++jj) acc[jj] += __shfl_xor_sync(0xffffffffu, acc[jj], o);
#pragma unroll
                    for (int jj = 0; jj < kGroup; ++jj) {
                        const float lv = __uint_as_float(en[jj].y);
                        if (j0 + jj < n && lv >= tall) {
                            const unsigned long long k = argmax_key(lv + acc[jj], en[jj].x);   // fp32(L) + Markov
                            if (k > best) {
                                best = k;
                                bslot = sb + j0 + jj;
                            }
                        }
                    }
                }
                bid = key_token(best);
            }
            int y = static_cast<int>(bid);
            if (bslot < 0 || y < 0 || y >= p.V) {
                if (lane == 0) set_status(p.dev_status, SDM_DEV_BAD_TOKEN);
                y = 0;
                bslot = -1;
            }
            if (lane == 0) emit_token(p, row, d - 1, y, s_pk0, s_pkn);
            if (bslot >= 0) {   // the winner's U row and bound were staged with it
                urow = st_u + static_cast<size_t>(bslot) * RS;
                cprev = st_c[bslot];
                pidx = bslot - sb;
            } else {
                urow = p.U + static_cast<size_t>(y) * r;
                cprev = p.c_bound[y];
                pidx = -1;
            }
            continue;
        }
        // global path: every warp, warp 0's state first
        const int par = d & 1;
        if (threadIdx.x == 0) {
            s_urow = urow;
            s_cprev = cprev;
            s_best[par] = 0ull;
        }
        __syncthreads();
        urow = s_urow;
        cprev = s_cprev;
        const int ds = (d - 1) * nc;
        const float tall = threshold(lmax, cprev);
        float ubv[8];
        load_ub(urow, lane, r, ubv);
        if (!s_over[d - 1]) {
            // the step's list entries in windows of kPickCap; ids with L >= tall scored
            const int* pref = s_pref + (d - 1) * (nc + 1);
            const int total = pref[nc];
            for (int w0 = 0; w0 < total; w0 += kPickCap) {
                if (threadIdx.x == 0) s_m = 0;
                __syncthreads();
                for (int t = w0 + threadIdx.x; t < min(total, w0 + kPickCap); t += kThreads) {
                    const int c = segment_of(pref, nc, t);
                    const uint2 en = p.cand[static_cast<size_t>(seg0 + ds + c) * kSegCap + (t - pref[c])];
                    if (en.x < static_cast<uint32_t>(p.V) && __uint_as_float(en.y) >= tall)
                        s_ids[atomicAdd(&s_m, 1)] = en;
                }
                __syncthreads();
                const unsigned long long b = warp_max_u64(score_global(p, s_ids, s_m, ubv, warp, lane));
                if (lane == 0 && b) atomicMax(&s_best[par], b);
                __syncthreads();
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
                const unsigned long long b = warp_max_u64(score_global(p, s_ids, s_m, ubv, warp, lane));
                if (lane == 0 && b) atomicMax(&s_best[par], b);
                __syncthreads();
            }
        }
        __syncthreads();
        const unsigned long long win = s_best[par];
        int y = static_cast<int>(key_token(win));
        if (win == 0ull || y < 0 || y >= p.V) {
            if (threadIdx.x == 0) set_status(p.dev_status, SDM_DEV_BAD_TOKEN);
            y = 0;
        }
        if (threadIdx.x == 0) emit_token(p, row, d - 1, y, s_pk0, s_pkn);
        urow = p.U + static_cast<size_t>(y) * r;
        cprev = p.c_bound[y];
        pidx = -1;
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

// c(y) = A(y) (1 + 2^-10) + 4 r 2^-24 |U[y]| max_v |W[:, v]| + 2^-20, rounded
// up, where A(y) = max_v |U[y] . W[:, v]| as the tensor cores accumulated it.
// Any fp32 evaluation of a dot product of length r differs from the exact
// one by at most about r 2^-24 |U[y]| |W[:, v]|, so 4 r 2^-24 |U| max|W|
// covers both the tensor-core maximum and the pick kernel's own dot products.
__global__ void bounds_kernel(const unsigned int* absmax_bits, const float* u_norm, const float* n_max, int V, int r,
                              float* c_bound, unsigned int* c_max_bits) {
    const int y = blockIdx.x * blockDim.x + threadIdx.x;
    if (y >= V) return;
    const double a = static_cast<double>(__uint_as_float(absmax_bits[y]));
    const double slack = 4.0 * r * 5.9604644775390625e-8 * static_cast<double>(u_norm[y]) * static_cast<double>(*n_max);
    const float c = __double2float_ru(a * (1.0 + 9.765625e-4) + slack + 9.5367431640625e-7);
    c_bound[y] = c;
    atomicMax(c_max_bits, __float_as_uint(c));
}

}  // namespace

int pruned_chunks(int V, int l_fp32) {
    const int per = kChunkBytes / (l_fp32 ? 4 : 2);
    return (V + per - 1) / per;
}

cudaError_t launch_chain_scan(const PrunedParams& p, cudaStream_t s) {
    const long long items = static_cast<long long>(p.R) * p.B * p.n_chunks;
    if (items > (1LL << 30)) return cudaErrorInvalidValue;
    // two CTAs per resident slot: a CTA that finishes early is replaced, which
    // evens out the tail better than one wave of equal shares
    const int grid = static_cast<int>(items < 8LL * num_sms() ? items : 8LL * num_sms());
    const size_t smem = p.fr.on ? chain_front_smem(p.R, p.B) : 0;
    if (smem > kFrontSmemMax) return cudaErrorInvalidValue;
    return p.l_fp32 ? launch_pdl(chain_scan_kernel<1>, dim3(grid + (p.fr.on ? 1 : 0)), dim3(kThreads), smem, s, p)
                    : launch_pdl(chain_scan_kernel<0>, dim3(grid + (p.fr.on ? 1 : 0)), dim3(kThreads), smem, s, p);
}

size_t chain_front_smem(int R, int B) {
    int n_pad = 1;
    while (n_pad < R * B) n_pad <<= 1;
    return schedule_smem_bytes(R, B, n_pad, kThreads);
}

cudaError_t launch_chain_pruned(const PrunedParams& p, cudaStream_t s) {
    cudaError_t e = launch_chain_scan(p, s);
    if (e != cudaSuccess) return e;
    return launch_chain_pick(p, s);
}

cudaError_t launch_chain_pick(const PrunedParams& p, cudaStream_t s) {
    cudaError_t e = cudaSuccess;
    const PickLayout lay = pick_layout(p.B, p.n_chunks, p.r);
    if (lay.cap < 1) return cudaErrorInvalidValue;
    static bool configured = false;
    if (!configured) {
        e = cudaFuncSetAttribute(chain_pick_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, kPickSmem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(chain_pick_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, kPickSmem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    return p.l_fp32 ? launch_pdl(chain_pick_kernel<1>, dim3(p.R), dim3(kThreads), lay.total, s, p)
                    : launch_pdl(chain_pick_kernel<0>, dim3(p.R), dim3(kThreads), lay.total, s, p);
}

cudaError_t launch_markov_prepare(const uint16_t* U, const uint16_t* W, int V, int r, uint16_t* Wt, float* u_norm,
                                  float* n_max, float* u_max, unsigned int* absmax_bits, cudaStream_t s) {
    transpose_kernel<<<dim3((V + 31) / 32, (r + 31) / 32), dim3(32, 8), 0, s>>>(W, r, V, Wt);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = cudaMemsetAsync(n_max, 0, sizeof(float), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(u_max, 0, sizeof(float), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(absmax_bits, 0, static_cast<size_t>(V) * sizeof(unsigned int), s);
    if (e != cudaSuccess) return e;
    const int blocks = (V * 32 + 255) / 256;
    row_norm_kernel<<<blocks, 256, 0, s>>>(U, V, r, u_norm, reinterpret_cast<unsigned int*>(u_max));
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    row_norm_kernel<<<blocks, 256, 0, s>>>(Wt, V, r, nullptr, reinterpret_cast<unsigned int*>(n_max));
    return cudaGetLastError();
}

cudaError_t launch_markov_bounds(const unsigned int* absmax_bits, const float* u_norm, const float* n_max, int V,
                                 int r, float* c_bound, float* c_max, cudaStream_t s) {
    cudaError_t e = cudaMemsetAsync(c_max, 0, sizeof(float), s);
    if (e != cudaSuccess) return e;
    bounds_kernel<<<(V + 255) / 256, 256, 0, s>>>(absmax_bits, u_norm, n_max, V, r, c_bound,
                                                  reinterpret_cast<unsigned int*>(c_max));
    return cudaGetLastError();
}

}  // namespace sdm
