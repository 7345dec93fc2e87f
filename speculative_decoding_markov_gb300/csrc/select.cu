// select.cu - categorical draws by the inverse CDF in vocabulary order.
//
// Every sampled token of the path (the draft y_d ~ q_d, the residual
// max(0, p - q) at the first rejection, the bonus ~ p) is the smallest id v
// with w_0 + ... + w_v > u S, S = sum of the nonnegative weights, one uniform
// u per draw (Philox word 0 of the draw's stream and row).  The weights are
// never materialised over the vocabulary.  The producing kernel leaves one
// record (m, s) per run of ids whose weights sum to s exp(m - M) on a common
// scale M: 16-column blocks from the Markov GEMM (draft and residual), or the
// streaming chunks of a target row (bonus).  One CTA per draw then
//   1. copies the request's records to shared memory (one bulk copy), splits
//      them into eight contiguous warp ranges (read 32 records at a time),
//      finds the maximum M and the warp weights (one 32-record chunk per
//      lane), and picks the warp holding u S from the eight sums;
//   2. that warp walks its range to the record holding the point (warp scan
//      + ballot);
//   3. the record's ids are recomputed (z = L + U[y] . W for a 16-column
//      block, the target row for a chunk) and walked to the id.
// Each level passes down the point as a fraction of the weight it selected,
// so the levels stay consistent whatever the rounding of the sums: a
// fraction that the recomputed weights cannot reach takes the last id of
// positive weight.
#include <algorithm>

#include "device.cuh"
#include "internal.h"

namespace sdm {
namespace {

constexpr int kSelThreads = 256;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kBlockCols = 16;   // ids per Markov GEMM record
constexpr float kBelowOne = 0.99999994f;
constexpr int kStageMaxRecords = 24576;   // records staged in shared memory (192 KB); more are read in place
constexpr uint32_t kBulkChunk = 32768;    // bytes per bulk copy instruction

constexpr int kMaxChunks = 1024;          // chunk sums of the walk kept in shared memory

struct SelShared {
    float csum[kMaxChunks];   // chunk sums of block_walk; chunk sums of the record walk
    float cmax[kMaxChunks];   // chunk maxima of the record walk
    float wmx[kSelWarps];
    float wsum[kSelWarps];
    float wmax[kSelWarps];
    uint64_t bar;
    int owner;
    float frac;
    int part;
    float part_frac;
    float red[kBlockCols][kBlockCols + 1];
};

__device__ __forceinline__ float clamp_frac(float f) { return fminf(fmaxf(f, 0.f), kBelowOne); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float block_max(float v, SelShared& sh) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if ((threadIdx.x & 31) == 0) sh.wmax[threadIdx.x >> 5] = v;
    __syncthreads();
    float m = sh.wmax[0];
#pragma unroll
    for (int q = 1; q < kSelWarps; ++q) m = fmaxf(m, sh.wmax[q]);
    __syncthreads();
    return m;
}

// One warp: the element of [lo, hi) holding fraction f of the range's total
// weight (weights from wfn(b)).  Returns the element (or the last one of
// positive weight, -1 if none) and *frac_in = the point's fraction of its
// weight; every lane gets the same result.  wfn is called by all 32 lanes
// together (it may shuffle), with indexes clamped into the range.
template <typename WFn>
__device__ __forceinline__ int warp_pick(int lo, int hi, float f, WFn wfn, float* frac_in) {
    const int lane = threadIdx.x & 31;
    auto wat = [&](int b0) {
        const float w = wfn(min(b0 + lane, hi - 1));
        return b0 + lane < hi ? w : 0.f;
    };
    float tot = 0.f;
    for (int b0 = lo; b0 < hi; b0 += 32) tot += wat(b0);
    tot = warp_sum(tot);
    const float T = f * tot;
    float c = 0.f;
    int last = -1;
    for (int b0 = lo; b0 < hi; b0 += 32) {
        const float w = wat(b0);
        float incl = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        const unsigned pass = __ballot_sync(0xffffffffu, w > 0.f && c + incl > T);
        const unsigned pos = __ballot_sync(0xffffffffu, w > 0.f);
        if (pos) last = b0 + 31 - __clz(pos);
        if (pass) {
            const int l = __ffs(pass) - 1;
            const float wl = __shfl_sync(0xffffffffu, w, l);
            const float il = __shfl_sync(0xffffffffu, incl, l);
            *frac_in = clamp_frac((T - (c + il - wl)) / wl);
            return b0 + l;
        }
        c += __shfl_sync(0xffffffffu, incl, 31);
    }
    *frac_in = kBelowOne;
    return last;
}

// Weight of record r on the scale M.
__device__ __forceinline__ float rec_weight(float2 r, float M) { return r.y > 0.f ? r.y * __expf(r.x - M) : 0.f; }

// Warp w's contiguous share [lo, hi) of n items.
__device__ __forceinline__ void warp_range(int n, int* lo, int* hi) {
    const int per = (n + kSelWarps - 1) / kSelWarps;
    *lo = min(n, (static_cast<int>(threadIdx.x) >> 5) * per);
    *hi = min(n, *lo + per);
}

// Levels 1 and 2 over n items with weights wfn(i) >= 0 (callable by all 32
// lanes together): sh.part = the item holding f S (-1 when S = 0), S = the
// sum of the weights, sh.part_frac = the point's fraction of that item's
// weight.  The items form chunks of 32 (more, a power of two, above 32768
// items); every warp sums its share of the chunks, one chunk per lane (chunk
// sums in shared memory); the warp holding the point is the last warp of positive weight
// whose exclusive prefix (the same sums in every thread) is <= f S, and
// it walks its chunk sums, then the chosen chunk's items.  Returns S.
template <typename WFn>
__device__ float block_walk(int n, float f, WFn wfn, SelShared& sh) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int cs = 32;   // chunk size: a power of two, at most kMaxChunks chunks
    while (cs * kMaxChunks < n) cs <<= 1;
    const int nch = (n + cs - 1) / cs;
    const int cpw = (nch + kSelWarps - 1) / kSelWarps;
    const int c0 = min(nch, warp * cpw), c1 = min(nch, c0 + cpw);
    // lane l sums chunk c0 + l (+ 32 ...) alone, starting at item l of the
    // chunk so that the lanes' reads fall in different banks
    float wt = 0.f;
    for (int cb = c0; cb < c1; cb += 32) {
        const int c = cb + lane;
        const int e0 = min(c, nch - 1) * cs, e1 = min(n, e0 + cs);
        float v = 0.f;
#pragma unroll 8
        for (int j = 0; j < cs; ++j) {
            const int e = e0 + ((j + lane) & (cs - 1));
            const float w = wfn(min(e, e1 - 1));
            v += e < e1 ? w : 0.f;
        }
        if (c < c1) {
            sh.csum[c] = v;
            wt += v;
        }
    }
    wt = warp_sum(wt);
    if (lane == 0) sh.wsum[warp] = wt;
    __syncthreads();
    // (fp32: eight partial sums; fp64 is a slow pipe on this part)
    float S = 0.f;
#pragma unroll
    for (int q = 0; q < kSelWarps; ++q) S += sh.wsum[q];
    const float T = f * S;
    int owner = -1;
    float excl = 0.f, run = 0.f;
#pragma unroll
    for (int q = 0; q < kSelWarps; ++q) {
        if (sh.wsum[q] > 0.f && run <= T) {
            owner = q;
            excl = run;
        }
        run += sh.wsum[q];
    }
    if (owner < 0) {
        if (threadIdx.x == 0) {
            sh.part = -1;
            sh.part_frac = 0.f;
        }
    } else if (warp == owner) {
        const float fw = clamp_frac((T - excl) / sh.wsum[owner]);
        float fc;
        const int c = warp_pick(c0, c1, fw, [&](int q) { return sh.csum[q]; }, &fc);
        int pick = -1;
        float pf = 0.f;
        if (c >= 0) pick = warp_pick(c * cs, min(n, (c + 1) * cs), fc, wfn, &pf);
        if (lane == 0) {
            sh.part = pick;
            sh.part_frac = pf;
        }
    }
    __syncthreads();
    return S;
}

// The (max, sum) pair of the 32 records of chunk c (records past n count as
// empty): sixteen 16-byte loads, issued in a lane-rotated order so that the
// lanes of a warp, which read sixteen different chunks, spread over the banks.
// rec is 16-byte aligned and holds at least n rounded up to even records.
__device__ __forceinline__ void chunk_pair(const float2* rec, int n, int c, float* cm, float* cs) {
    const int lane = threadIdx.x & 31;
    const float4* q = reinterpret_cast<const float4*>(rec + c * 32);
    float4 v[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const int jj = (j + lane) & 15;
        v[j] = (c * 32 + 2 * jj < n) ? q[jj] : make_float4(-INFINITY, 0.f, -INFINITY, 0.f);
        if (c * 32 + 2 * jj + 1 >= n) v[j].w = 0.f;   // odd n: the second record of the last pair is padding
    }
    float m = -INFINITY;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        if (v[j].y > 0.f) m = fmaxf(m, v[j].x);
        if (v[j].w > 0.f) m = fmaxf(m, v[j].z);
    }
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        if (v[j].y > 0.f) s += v[j].y * __expf(v[j].x - m);
        if (v[j].w > 0.f) s += v[j].w * __expf(v[j].z - m);
    }
    *cm = m;
    *cs = s;
}

// Levels 1-3 over n (m, s) records: every lane condenses one 32-record chunk
// to a (max, sum) pair (chunk pairs in shared memory), the warps' pairs give
// the scale M and the weights; the warp holding u S walks its chunks, then the
// chosen chunk's records.  sh.part / sh.part_frac as for block_walk; returns
// S, *M_out = M.
__device__ float walk_records(const float2* rec, int n, float u, SelShared& sh, float* M_out) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nch = (n + 31) / 32;
    const int cpw = (nch + kSelWarps - 1) / kSelWarps;
    const int c0 = min(nch, warp * cpw), c1 = min(nch, c0 + cpw);
    Lse acc{-INFINITY, 0.f};
    for (int cb = c0; cb < c1; cb += 32) {
        const int c = cb + lane;
        float cm = -INFINITY, cs = 0.f;
        if (c < c1) {
            chunk_pair(rec, n, c, &cm, &cs);
            sh.cmax[c] = cm;
            sh.csum[c] = cs;
        }
        if (cs > 0.f) acc = lse_merge(acc, Lse{cm, cs});
    }
    acc = warp_lse(acc);
    if (lane == 0) {
        sh.wmx[warp] = acc.m;
        sh.wsum[warp] = acc.s;
    }
    __syncthreads();
    float M = -INFINITY;
#pragma unroll
    for (int q = 0; q < kSelWarps; ++q)
        if (sh.wsum[q] > 0.f) M = fmaxf(M, sh.wmx[q]);
    float wq[kSelWarps], S = 0.f;
#pragma unroll
    for (int q = 0; q < kSelWarps; ++q) {
        wq[q] = sh.wsum[q] > 0.f ? sh.wsum[q] * __expf(sh.wmx[q] - M) : 0.f;
        S += wq[q];
    }
    const float T = u * S;
    int owner = -1;
    float excl = 0.f, run = 0.f, wo = 0.f;
#pragma unroll
    for (int q = 0; q < kSelWarps; ++q) {
        if (wq[q] > 0.f && run <= T) {
            owner = q;
            excl = run;
            wo = wq[q];
        }
        run += wq[q];
    }
    if (owner < 0) {
        if (threadIdx.x == 0) {
            sh.part = -1;
            sh.part_frac = 0.f;
        }
    } else if (warp == owner) {
        const float fw = clamp_frac((T - excl) / wo);
        float fc;
        const int c = warp_pick(c0, c1, fw,
                                [&](int q) { return sh.csum[q] > 0.f ? sh.csum[q] * __expf(sh.cmax[q] - M) : 0.f; },
                                &fc);
        int pick = -1;
        float pf = 0.f;
        if (c >= 0) pick = warp_pick(c * 32, min(n, c * 32 + 32), fc, [&](int b) { return rec_weight(rec[b], M); }, &pf);
        if (lane == 0) {
            sh.part = pick;
            sh.part_frac = pf;
        }
    }
    __syncthreads();
    *M_out = M;
    return S;
}

// Copies bytes (a multiple of 16, 16-byte aligned source) to dst with bulk
// copies on sh.bar; false if the copy did not complete in time.
__device__ bool stage_bulk(void* dst, const void* src, uint32_t bytes, SelShared& sh) {
    if (threadIdx.x == 0) {
        mbar_init(&sh.bar, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(&sh.bar, bytes);
        for (uint32_t off = 0; off < bytes; off += kBulkChunk)
            bulk_load(static_cast<uint8_t*>(dst) + off, static_cast<const uint8_t*>(src) + off,
                      bytes - off < kBulkChunk ? bytes - off : kBulkChunk, &sh.bar);
    }
    __syncthreads();
    if (mbar_wait(&sh.bar, 0)) return true;
    // the copy did not land in time: wait once more (bounded) so that the
    // CTA does not go on, or exit, while it may still write shared memory
    mbar_wait(&sh.bar, 0);
    return false;
}

// Markov logits of the 16 columns v0 .. v0 + 15 for token prev, without L:
// sh.red[ks][c] holds the K slice ks of column c (all threads take part).
__device__ __forceinline__ void markov16(const uint16_t* U, const uint16_t* W, int prev, int r, int V, int v0,
                                         SelShared& sh) {
    const int tid = threadIdx.x;
    const int col = tid & (kBlockCols - 1), ks = tid / kBlockCols;   // 16 K slices of r / 16 <= 16
    const int kper = r / kBlockCols;
    const int v = v0 + col;
    float acc = 0.f;
    if (v < V) {
        const uint16_t* u = U + static_cast<size_t>(prev) * r + ks * kper;
        const uint16_t* w = W + static_cast<size_t>(ks * kper) * V + v;
        float uu[16], ww[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {   // every load in flight at once
            uu[j] = j < kper ? bf16_bits_to_float(u[j]) : 0.f;
            ww[j] = j < kper ? bf16_bits_to_float(w[static_cast<size_t>(j) * V]) : 0.f;
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) acc += uu[j] * ww[j];
    }
    sh.red[ks][col] = acc;
    __syncthreads();
}

__device__ __forceinline__ float load_elem(const void* base, int fp32, size_t idx) {
    if (fp32) return static_cast<const float*>(base)[idx];
    return bf16_bits_to_float(static_cast<const uint16_t*>(base)[idx]);
}

// Records of one request row: staged in shared memory when they fit.
__device__ __forceinline__ const float2* records_of(const float2* row, int n_valid, int stride, float2* sm,
                                                    SelShared& sh, int32_t* dev_status) {
    if (stride > kStageMaxRecords) return row;
    if (!stage_bulk(sm, row, static_cast<uint32_t>(stride) * 8u, sh)) {
        if (threadIdx.x == 0) set_status(dev_status, SDM_DEV_TIMEOUT);
        return row;   // read in place (the records are in global memory either way)
    }
    (void)n_valid;
    return sm;
}

// ---------------------------------------------------------------------------
// Draft step d: y_d ~ softmax(z_d / T) for request blockIdx.x; writes the
// token, lse = log sum exp(z_d / T) and log q(y_d) = z_d[y_d] / T - lse.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kSelThreads) draft_select_kernel(const DraftSelectParams p) {
    __shared__ SelShared sh;
    extern __shared__ __align__(16) float2 sm_rec[];
    pdl_wait();
    pdl_trigger();
    const int i = blockIdx.x;
    const int tid = threadIdx.x;
    const size_t o = static_cast<size_t>(i) * p.B + (p.d - 1);
    int prev = (p.d == 1) ? p.anchor[i] : p.tokens[o - 1];
    if (prev < 0 || prev >= p.V) {
        if (tid == 0) set_status(p.dev_status, SDM_DEV_BAD_TOKEN);
        prev = 0;
    }
    const RngKey rk{p.k0, p.k1, p.cycle};
    const float u = uniform_at(rk, 0u, static_cast<uint32_t>(i), static_cast<uint32_t>(p.d), 0u);
    const int n = (p.V + kBlockCols - 1) / kBlockCols;
    const float2* rec = records_of(p.blk + static_cast<size_t>(i) * p.nb, n, p.nb, sm_rec, sh, p.dev_status);
    float M;
    const float S = walk_records(rec, n, u, sh, &M);
    const int b = sh.part;
    if (b < 0) {   // no positive weight: only a non-finite row gets here
        if (tid == 0) {
            set_status(p.dev_status, SDM_DEV_BAD_TOKEN);
            p.tokens[o] = 0;
            if (p.lse) p.lse[o] = NAN;
            if (p.logq) p.logq[o] = NAN;
        }
        return;
    }
    const int v0 = b * kBlockCols;
    const int v = v0 + tid;
    const float lv = (tid < kBlockCols && v < p.V) ? load_elem(p.L, p.l_fp32, o * p.V + v) : 0.f;
    if (p.a_rows)   // RNN head: the request's memo row stands where U[prev] does
        markov16(p.a_rows, p.W, i, p.r, p.V, v0, sh);
    else
        markov16(p.U, p.W, prev, p.r, p.V, v0, sh);
    if (tid < 32) {
        float zt = -INFINITY, w = 0.f;
        if (tid < kBlockCols && v < p.V) {
            float mk = 0.f;
#pragma unroll
            for (int ks = 0; ks < kBlockCols; ++ks) mk += sh.red[ks][tid];
            zt = (lv + mk) * p.inv_t;
            w = __expf(zt - rec[b].x);
        }
        float fi;
        const int c = warp_pick(0, kBlockCols, sh.part_frac, [&](int j) { return __shfl_sync(0xffffffffu, w, j); },
                                &fi);
        const int cc = c < 0 ? 0 : c;
        const float zy = __shfl_sync(0xffffffffu, zt, cc);
        if (tid == 0) {
            if (c < 0) set_status(p.dev_status, SDM_DEV_BAD_TOKEN);
            const float l = M + logf(S);
            p.tokens[o] = v0 + cc;
            if (p.lse) p.lse[o] = l;
            if (p.logq) p.logq[o] = zy - l;
        }
    }
}

// ---------------------------------------------------------------------------
// Rejection sampling, last step per request: the residual draw at the first
// rejection (position a) or the bonus draw from p at row a; then the
// committed tokens: a drafts and the drawn token.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kSelThreads) resample_kernel(const ResampleParams p) {
    __shared__ SelShared sh;
    extern __shared__ __align__(16) float2 sm_rec[];
    pdl_wait();
    pdl_trigger();
    const int i = blockIdx.x;
    const int tid = threadIdx.x;
    const RngKey rk{p.k0, p.k1, p.cycle};
    const int a = p.accept[i];
    int tok = 0;
    bool bad = false;
    if (p.res_tok[i] >= 0) {
        // residual: records of sum max(0, p - q) per 16-column block
        const int prev = p.res_tok[i];
        const int pos = p.res_pos[i];
        const float u = uniform_at(rk, 2u, static_cast<uint32_t>(i), static_cast<uint32_t>(pos), 0u);
        const int n = (p.V + kBlockCols - 1) / kBlockCols;
        const float2* rec = records_of(p.blk + static_cast<size_t>(i) * p.nb, n, p.nb, sm_rec, sh, p.dev_status);
        float M;
        walk_records(rec, n, u, sh, &M);
        const int b = sh.part;
        if (b >= 0) {
            const int v0 = b * kBlockCols;
            const int v = v0 + tid;
            const size_t lrow = static_cast<size_t>(i) * p.gamma + pos;
            float lv = 0.f, tv = 0.f;
            if (tid < kBlockCols && v < p.V) {
                lv = load_elem(p.L, p.l_fp32, lrow * p.V + v);
                tv = load_elem(p.target, p.t_fp32, static_cast<size_t>(p.res_trow[i]) * p.V + v);
            }
            markov16(p.U, p.W, prev, p.r, p.V, v0, sh);
            if (tid < 32) {
                float w = 0.f;
                if (tid < kBlockCols && v < p.V) {
                    float mk = 0.f;
#pragma unroll
                    for (int ks = 0; ks < kBlockCols; ++ks) mk += sh.red[ks][tid];
                    const float q = __expf((lv + mk) * p.inv_t - p.lse_q[lrow]);
                    const float pv = __expf(tv * p.inv_t - p.res_lse_p[i]);
                    w = fmaxf(pv - q, 0.f);
                }
                float fi;
                const int c = warp_pick(0, kBlockCols, sh.part_frac,
                                        [&](int j) { return __shfl_sync(0xffffffffu, w, j); }, &fi);
                tok = v0 + (c < 0 ? 0 : c);
            }
        } else {
            tok = 0;   // p = q everywhere (no residual mass): the first id, as an exact draw would
        }
    } else if (p.bonus_row[i] >= 0) {
        // bonus: chunk partials of target row / T, then the chunk's ids
        const int row = p.bonus_row[i];
        const float u = uniform_at(rk, 3u, static_cast<uint32_t>(i), static_cast<uint32_t>(p.bonus_pos[i]), 0u);
        {   // a few chunk records in global memory, not 16-byte aligned: scalar loads
            const float2* lp = p.lse_part + static_cast<size_t>(row) * p.n_chunks;
            float m = -INFINITY;
            for (int b = tid; b < p.n_chunks; b += kSelThreads)
                if (lp[b].y > 0.f) m = fmaxf(m, lp[b].x);
            const float M = block_max(m, sh);
            block_walk(p.n_chunks, u, [&](int b) { return rec_weight(lp[b], M); }, sh);
        }
        const int c = sh.part;
        if (c >= 0) {
            const float mc = p.lse_part[static_cast<size_t>(row) * p.n_chunks + c].x;
            const float f = sh.part_frac;
            const int e0 = c * p.chunk, e1 = min(p.V, e0 + p.chunk);
            const size_t esz = p.t_fp32 ? 4 : 2;
            const uint8_t* src = static_cast<const uint8_t*>(p.target) + (static_cast<size_t>(row) * p.V + e0) * esz;
            const uint32_t bytes = static_cast<uint32_t>((e1 - e0) * esz);
            const void* chunk_base = src;
            size_t chunk_off = 0;
            if (bytes <= static_cast<uint32_t>(kStageMaxRecords) * 8u && stage_bulk(sm_rec, src, bytes, sh)) {
                chunk_base = sm_rec;   // the chunk's ids, staged
            } else {
                chunk_base = p.target;
                chunk_off = static_cast<size_t>(row) * p.V + e0;
            }
            block_walk(e1 - e0, f,
                       [&](int e) { return __expf(load_elem(chunk_base, p.t_fp32, chunk_off + e) * p.inv_t - mc); }, sh);
            if (tid == 0 && sh.part >= 0) sh.part += e0;
            __syncthreads();
            tok = sh.part;
            if (tok < 0) {
                bad = true;
                tok = 0;
            }
        } else {
            bad = true;
        }
    }
    if (tid == 0) {
        if (bad) set_status(p.dev_status, SDM_DEV_BAD_TOKEN);
        int32_t* out = p.out_tok + static_cast<size_t>(i) * (p.gamma + 1);
        const int32_t* y = p.draft + static_cast<size_t>(i) * p.gamma;
        for (int q = 0; q < a; ++q) out[q] = y[q];
        out[a] = tok;
        for (int q = a + 1; q <= p.gamma; ++q) out[q] = -1;
        p.n_out[i] = a + 1;
    }
}

// ---------------------------------------------------------------------------
// PCTree level, one CTA per frontier row (request i, slot f) with a token:
// log-sum-exp of z over the vocabulary and the row's top-k children.  The
// top-k ids by z lie in the k 16-column blocks with the largest maxima (each
// of them is at most its block's maximum, and at most k blocks reach the
// k-th value), so the CTA ranks the records by maximum, keeps 2k blocks (a
// margin for the rounding of the GEMM's sums), recomputes their logits and
// ranks those by (z desc, id asc).
// ---------------------------------------------------------------------------
constexpr int kMaxCand = 16;   // candidate blocks per row

constexpr int kCandCap = 2048;   // records above the threshold: at most C x (records per lane) <= 16 x 128

struct TreeShared {
    unsigned long long wl[kSelWarps][kMaxCand];
    unsigned long long tau;
    int ncand;
    int cblk[kMaxCand];
    float fsum[kSelWarps];
    unsigned long long ckey[kMaxCand * kBlockCols];
    union {
        unsigned long long cand[kCandCap];
        float red[kBlockCols][kMaxCand * kBlockCols];
    };
};

// Warp bitonic sort of one 64-bit key per lane, descending (lane 0 largest).
__device__ __forceinline__ unsigned long long warp_sort_desc(unsigned long long key) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
            const unsigned long long other = __shfl_xor_sync(0xffffffffu, key, j);
            const bool take_max = (((lane & j) == 0) == ((lane & k) == 0));
            key = take_max ? umax64(key, other) : (key < other ? key : other);
        }
    }
    return key;
}

__global__ void __launch_bounds__(kSelThreads) tree_select_kernel(const TreeSelectParams p) {
    __shared__ SelShared sh;
    __shared__ TreeShared ts;
    extern __shared__ __align__(16) float2 sm_rec[];
    pdl_wait();
    pdl_trigger();
    const int row = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int tok = p.front_tok[row];
    if (tok < 0) return;   // an empty frontier slot
    if (tok >= p.V) {
        if (tid == 0) set_status(p.dev_status, SDM_DEV_BAD_TOKEN);
        return;
    }
    const int n = (p.V + kBlockCols - 1) / kBlockCols;
    const int C = min(min(2 * p.k, kMaxCand), n);
    if (tid < kMaxCand) ts.cblk[tid] = -1;   // (visible after the staging barrier)
    const float2* rec = records_of(p.blk + static_cast<size_t>(row) * p.nb, n, p.nb, sm_rec, sh, p.dev_status);
    // 1. per warp range, one record per lane at a time: the lanes'
    //    log-sum-exp partials and each lane's largest key (m, block id)
    int lo, hi;
    warp_range(n, &lo, &hi);
    float m = -INFINITY, s = 0.f;
    unsigned long long lmax = 0ull;
#pragma unroll 4
    for (int b = lo + lane; b < hi; b += 32) {
        const float2 r = rec[b];
        if (r.y > 0.f) {
            lmax = umax64(lmax, argmax_key(r.x, static_cast<uint32_t>(b)));
            if (r.x > m) {
                s = s * __expf(m - r.x) + r.y;
                m = r.x;
            } else {
                s += r.y * __expf(r.x - m);
            }
        }
    }
    // 2. the C blocks with the largest maxima.  tau = the C-th largest lane
    //    key: C records reach it, so every one of the top C does too, and
    //    only the C lanes at or above it can hold any.  Those lanes list
    //    their records >= tau, and the listed keys rank themselves.
    const unsigned long long sorted = warp_sort_desc(lmax);
    if (lane < C) ts.wl[warp][lane] = sorted;
    if (tid == 0) {
        ts.tau = 0ull;
        ts.ncand = 0;
    }
    const Lse part = warp_lse(Lse{m, s});
    const float M = block_max(part.m, sh);   // (synchronises: the lists, tau and ncand are visible after it)
    if (lane == 0) ts.fsum[warp] = part.s > 0.f ? part.s * __expf(part.m - M) : 0.f;
    if (tid < kSelWarps * kMaxCand) {
        const int wv = tid / kMaxCand, q = tid % kMaxCand;
        const unsigned long long me = q < C ? ts.wl[wv][q] : 0ull;
        if (me != 0ull) {
            int rank = 0;
            for (int x = 0; x < kSelWarps; ++x)
                for (int y = 0; y < C; ++y) rank += ts.wl[x][y] > me ? 1 : 0;
            if (rank == C - 1) ts.tau = me;   // fewer than C keys in all: tau stays 0, every record qualifies
        }
    }
    __syncthreads();
    const unsigned long long tau = ts.tau;
    if (lmax != 0ull && lmax >= tau) {
        for (int b = lo + lane; b < hi; b += 32) {
            const float2 r = rec[b];
            if (!(r.y > 0.f)) continue;
            const unsigned long long key = argmax_key(r.x, static_cast<uint32_t>(b));
            if (key >= tau) {
                const int slot = atomicAdd(&ts.ncand, 1);
                if (slot < kCandCap) ts.cand[slot] = key;
            }
        }
    }
    __syncthreads();
    const int ncand = min(ts.ncand, kCandCap);
    for (int t = tid; t < ncand; t += kSelThreads) {
        const unsigned long long me = ts.cand[t];
        int rank = 0;
        for (int x = 0; x < ncand; ++x) rank += ts.cand[x] > me ? 1 : 0;
        if (rank < C) ts.cblk[rank] = static_cast<int>(key_token(me));
    }
    if (tid == 0 && ts.ncand > kCandCap) set_status(p.dev_status, SDM_DEV_BAD_TOKEN);
    __syncthreads();
    float S = 0.f;
#pragma unroll
    for (int q = 0; q < kSelWarps; ++q) S += ts.fsum[q];
    // 3. recompute the candidates' Markov logits: thread (block c, K slice
    //    ks of r / 16 rows) loads its rows' 16 columns as two 16-byte
    //    vectors per row, eight rows in flight at a time
    {
        const int c = tid >> 4, ks = tid & 15;
        const int kper = p.r / kBlockCols;
        if (c < C) {
            const int cb = ts.cblk[c];
            float acc[kBlockCols];
#pragma unroll
            for (int q = 0; q < kBlockCols; ++q) acc[q] = 0.f;
            if (cb >= 0) {
                const int v0 = cb * kBlockCols;
                const bool second = v0 + 8 < p.V;   // V % 8 == 0: the block's second half exists or is wholly past V
                const uint16_t* urow = p.U + static_cast<size_t>(tok) * p.r + ks * kper;
#pragma unroll
                for (int jb = 0; jb < 16; jb += 8) {
                    uint4 lo8[8], hi8[8];
                    float uu[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        lo8[j] = make_uint4(0u, 0u, 0u, 0u);
                        hi8[j] = make_uint4(0u, 0u, 0u, 0u);
                        uu[j] = 0.f;
                        if (jb + j < kper) {
                            const uint16_t* wr = p.W + static_cast<size_t>(ks * kper + jb + j) * p.V + v0;
                            lo8[j] = __ldg(reinterpret_cast<const uint4*>(wr));
                            if (second) hi8[j] = __ldg(reinterpret_cast<const uint4*>(wr + 8));
                            uu[j] = bf16_bits_to_float(urow[jb + j]);
                        }
                    }
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint32_t a[4] = {lo8[j].x, lo8[j].y, lo8[j].z, lo8[j].w};
                        const uint32_t b[4] = {hi8[j].x, hi8[j].y, hi8[j].z, hi8[j].w};
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            acc[2 * q] += uu[j] * __uint_as_float(a[q] << 16);
                            acc[2 * q + 1] += uu[j] * __uint_as_float(a[q] & 0xffff0000u);
                            acc[8 + 2 * q] += uu[j] * __uint_as_float(b[q] << 16);
                            acc[8 + 2 * q + 1] += uu[j] * __uint_as_float(b[q] & 0xffff0000u);
                        }
                    }
                }
            }
#pragma unroll
            for (int q = 0; q < kBlockCols; ++q) ts.red[ks][c * kBlockCols + q] = acc[q];
        }
    }
    __syncthreads();
    // 4. candidate keys, then the top-k by rank
    const int nc = C * kBlockCols;
    float zc = -INFINITY;
    int vc = -1;
    if (tid < nc) {
        const int cb = ts.cblk[tid / kBlockCols];
        const int v = cb * kBlockCols + (tid % kBlockCols);
        unsigned long long key = 0ull;
        if (cb >= 0 && v < p.V) {
            float mk = 0.f;
#pragma unroll
            for (int q = 0; q < kBlockCols; ++q) mk += ts.red[q][tid];
            zc = load_elem(p.L, p.l_fp32, (static_cast<size_t>(row / p.P) * p.B + (p.d - 1)) * p.V + v) + mk;
            vc = v;
            key = argmax_key(zc, static_cast<uint32_t>(v));
        }
        ts.ckey[tid] = key;
    }
    __syncthreads();
    if (tid < nc && vc >= 0) {
        const unsigned long long me = ts.ckey[tid];
        int rank = 0;
        for (int q = 0; q < nc; ++q) rank += ts.ckey[q] > me ? 1 : 0;
        if (rank < p.k) p.row_top[static_cast<size_t>(row) * kMaxTopK + rank] = make_float2(zc, __int_as_float(vc));
    }
    if (tid == 0) p.row_lse[row] = M + logf(S);
}

size_t stage_bytes(int stride) {
    return stride > kStageMaxRecords ? 0 : static_cast<size_t>(stride) * sizeof(float2);
}

template <typename K>
cudaError_t allow_smem(K kernel, bool& done) {
    if (done) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(stage_bytes(kStageMaxRecords)));
    done = e == cudaSuccess;
    return e;
}

}  // namespace

cudaError_t launch_draft_select(const DraftSelectParams& p, cudaStream_t s) {
    if (p.R <= 0) return cudaSuccess;
    static bool configured = false;
    cudaError_t e = allow_smem(draft_select_kernel, configured);
    if (e != cudaSuccess) return e;
    return launch_pdl(draft_select_kernel, dim3(p.R), dim3(kSelThreads), stage_bytes(p.nb), s, p);
}

cudaError_t launch_tree_select(const TreeSelectParams& p, cudaStream_t s) {
    if (p.rows <= 0) return cudaSuccess;
    static bool configured = false;
    cudaError_t e = allow_smem(tree_select_kernel, configured);
    if (e != cudaSuccess) return e;
    return launch_pdl(tree_select_kernel, dim3(p.rows), dim3(kSelThreads), stage_bytes(p.nb), s, p);
}

cudaError_t launch_resample(const ResampleParams& p, cudaStream_t s) {
    if (p.R <= 0) return cudaSuccess;
    static bool configured = false;
    cudaError_t e = allow_smem(resample_kernel, configured);
    if (e != cudaSuccess) return e;
    // the residual records, or the bonus draw's chunk of a target row (32 KB)
    const size_t smem = std::max(stage_bytes(p.nb), static_cast<size_t>(p.chunk) * (p.t_fp32 ? 4 : 2));
    return launch_pdl(resample_kernel, dim3(p.R), dim3(kSelThreads), std::min(smem, stage_bytes(kStageMaxRecords)), s,
                      p);
}

}  // namespace sdm
