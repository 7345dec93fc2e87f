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
//   1. splits the records into contiguous per-thread ranges, finds the
//      block-wide maximum M and the range weights, and locates the range
//      holding u S with a block scan in fp64;
//   2. the owning thread walks its range to the record holding the point;
//   3. the record's ids are recomputed (z = L + U[y] . W for a 16-column
//      block, the target row for a chunk) and walked to the id.
// Each level passes down the point as a fraction of the weight it selected,
// so the levels stay consistent whatever the rounding of the sums: a
// fraction that the recomputed weights cannot reach takes the last id of
// positive weight.
#include "device.cuh"
#include "internal.h"

namespace sdm {
namespace {

constexpr int kSelThreads = 256;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kBlockCols = 16;   // ids per Markov GEMM record
constexpr float kBelowOne = 0.99999994f;

struct SelShared {
    double wsum[kSelWarps];
    float wmax[kSelWarps];
    int owner;
    float frac;
    int part;
    float part_frac;
    float red[kBlockCols][kBlockCols + 1];
};

__device__ __forceinline__ float clamp_frac(float f) { return fminf(fmaxf(f, 0.f), kBelowOne); }

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

// Thread weights w >= 0 in thread order; the point f * S (S = their sum, in
// fp64) falls in the range of sh.owner, the last thread of positive weight
// whose exclusive prefix is <= f S (-1 when S = 0), at fraction sh.frac of its
// weight.  Returns S.
__device__ double block_locate(float w, float f, SelShared& sh) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    double x = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sh.wsum[warp] = x;
    if (tid == 0) sh.owner = -1;
    __syncthreads();
    double off = 0.0, S = 0.0;
#pragma unroll
    for (int q = 0; q < kSelWarps; ++q) {
        if (q < warp) off += sh.wsum[q];
        S += sh.wsum[q];
    }
    const double excl = off + (x - static_cast<double>(w));
    const double T = static_cast<double>(f) * S;
    if (w > 0.f && excl <= T) atomicMax(&sh.owner, tid);
    __syncthreads();
    if (tid == sh.owner) sh.frac = clamp_frac(static_cast<float>((T - excl) / static_cast<double>(w)));
    __syncthreads();
    return S;
}

// Weight of record r on the scale M.
__device__ __forceinline__ float rec_weight(float2 r, float M) { return r.y > 0.f ? r.y * __expf(r.x - M) : 0.f; }

// Level 1 and 2 over n records: sh.part = the record holding u S (-1 when
// S = 0), sh.part_frac = the point's fraction of that record's weight.
// Returns S; *M_out = the scale M.
__device__ double walk_records(const float2* rec, int n, float u, SelShared& sh, float* M_out) {
    const int tid = threadIdx.x;
    const int per = (n + kSelThreads - 1) / kSelThreads;
    const int lo = min(n, tid * per), hi = min(n, lo + per);
    float m = -INFINITY, s = 0.f;
    for (int b = lo; b < hi; ++b) {
        const float2 r = rec[b];
        if (!(r.y > 0.f)) continue;
        if (r.x > m) {
            s = s * __expf(m - r.x) + r.y;
            m = r.x;
        } else {
            s += r.y * __expf(r.x - m);
        }
    }
    const float M = block_max(m, sh);
    const float wt = s > 0.f ? s * __expf(m - M) : 0.f;
    const double S = block_locate(wt, u, sh);
    if (tid == sh.owner) {
        float tot = 0.f;
        for (int b = lo; b < hi; ++b) tot += rec_weight(rec[b], M);
        const float T = sh.frac * tot;
        float c = 0.f, pf = kBelowOne;
        int pick = -1, last = -1;
        for (int b = lo; b < hi; ++b) {
            const float w = rec_weight(rec[b], M);
            if (!(w > 0.f)) continue;
            last = b;
            if (pick < 0 && c + w > T) {
                pick = b;
                pf = (T - c) / w;
            }
            c += w;
        }
        if (pick < 0) pick = last;
        sh.part = pick;
        sh.part_frac = clamp_frac(pf);
    }
    if (tid == 0 && sh.owner < 0) {
        sh.part = -1;
        sh.part_frac = 0.f;
    }
    __syncthreads();
    *M_out = M;
    return S;
}

// Within one warp: lanes 0..15 hold the weights of a record's columns; the
// column holding fraction f of their sum (the first lane whose running sum
// passes it, else the last lane of positive weight; -1 if none is positive).
__device__ __forceinline__ int warp_walk16(float w, float f) {
    const int lane = threadIdx.x & 31;
    float c = w;
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, c, o);
        if (lane >= o) c += y;
    }
    const float tot = __shfl_sync(0xffffffffu, c, 15);
    const float T = f * tot;
    const unsigned pass = __ballot_sync(0xffffffffu, lane < 16 && w > 0.f && c > T);
    if (pass) return __ffs(pass) - 1;
    const unsigned pos = __ballot_sync(0xffffffffu, lane < 16 && w > 0.f);
    return pos ? 31 - __clz(pos) : -1;
}

// Markov logits of the 16 columns v0 .. v0 + 15 for token prev, without L:
// sh.red[ks][c] holds the K slice ks of column c (all threads take part).
__device__ __forceinline__ void markov16(const uint16_t* U, const uint16_t* W, int prev, int r, int V, int v0,
                                         SelShared& sh) {
    const int tid = threadIdx.x;
    const int col = tid & (kBlockCols - 1), ks = tid / kBlockCols;   // 16 K slices of r / 16
    const int kper = r / kBlockCols;
    const int v = v0 + col;
    float acc = 0.f;
    if (v < V) {
        const uint16_t* u = U + static_cast<size_t>(prev) * r + ks * kper;
        const uint16_t* w = W + static_cast<size_t>(ks * kper) * V + v;
#pragma unroll 4
        for (int j = 0; j < kper; ++j) acc += bf16_bits_to_float(u[j]) * bf16_bits_to_float(w[static_cast<size_t>(j) * V]);
    }
    sh.red[ks][col] = acc;
    __syncthreads();
}

__device__ __forceinline__ float load_elem(const void* base, int fp32, size_t idx) {
    if (fp32) return static_cast<const float*>(base)[idx];
    return bf16_bits_to_float(static_cast<const uint16_t*>(base)[idx]);
}

// ---------------------------------------------------------------------------
// Draft step d: y_d ~ softmax(z_d / T) for request blockIdx.x; writes the
// token, lse = log sum exp(z_d / T) and log q(y_d) = z_d[y_d] / T - lse.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kSelThreads) draft_select_kernel(const DraftSelectParams p) {
    __shared__ SelShared sh;
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
    const float2* rec = p.blk + static_cast<size_t>(i) * p.nb;
    float M;
    const double S = walk_records(rec, p.nb, u, sh, &M);
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
    markov16(p.U, p.W, prev, p.r, p.V, v0, sh);
    if (tid < 32) {
        const int lane = tid;
        const int v = v0 + lane;
        float zt = -INFINITY, w = 0.f;
        if (lane < kBlockCols && v < p.V) {
            float mk = 0.f;
#pragma unroll
            for (int ks = 0; ks < kBlockCols; ++ks) mk += sh.red[ks][lane];
            zt = (load_elem(p.L, p.l_fp32, o * p.V + v) + mk) * p.inv_t;
            w = __expf(zt - rec[b].x);
        }
        const int c = warp_walk16(w, sh.part_frac);
        const int cc = c < 0 ? 0 : c;
        const float zy = __shfl_sync(0xffffffffu, zt, cc);
        if (lane == 0) {
            if (c < 0) set_status(p.dev_status, SDM_DEV_BAD_TOKEN);
            const float l = M + logf(static_cast<float>(S));
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
        const float2* rec = p.blk + static_cast<size_t>(i) * p.nb;
        float M;
        walk_records(rec, p.nb, u, sh, &M);
        const int b = sh.part;
        if (b >= 0) {
            const int v0 = b * kBlockCols;
            markov16(p.U, p.W, prev, p.r, p.V, v0, sh);
            if (tid < 32) {
                const int v = v0 + tid;
                float w = 0.f;
                if (tid < kBlockCols && v < p.V) {
                    float mk = 0.f;
#pragma unroll
                    for (int ks = 0; ks < kBlockCols; ++ks) mk += sh.red[ks][tid];
                    const size_t lrow = static_cast<size_t>(i) * p.gamma + pos;
                    const float q = __expf((load_elem(p.L, p.l_fp32, lrow * p.V + v) + mk) * p.inv_t - p.lse_q[lrow]);
                    const float pv = __expf(load_elem(p.target, p.t_fp32, static_cast<size_t>(p.res_trow[i]) * p.V + v) *
                                                p.inv_t -
                                            p.res_lse_p[i]);
                    w = fmaxf(pv - q, 0.f);
                }
                const int c = warp_walk16(w, sh.part_frac);
                tok = v0 + (c < 0 ? 0 : c);
            }
        } else {
            tok = 0;   // p = q everywhere (no residual mass): the first id, as an exact draw would
        }
    } else if (p.bonus_row[i] >= 0) {
        // bonus: chunk partials of target row / T, then the chunk's ids
        const int row = p.bonus_row[i];
        const float u = uniform_at(rk, 3u, static_cast<uint32_t>(i), static_cast<uint32_t>(p.bonus_pos[i]), 0u);
        float M;
        walk_records(p.lse_part + static_cast<size_t>(row) * p.n_chunks, p.n_chunks, u, sh, &M);
        const int c = sh.part;
        if (c >= 0) {
            const float mc = p.lse_part[static_cast<size_t>(row) * p.n_chunks + c].x;
            const float f = sh.part_frac;
            const int e0 = c * p.chunk, e1 = min(p.V, e0 + p.chunk);
            const int per = (e1 - e0 + kSelThreads - 1) / kSelThreads;
            const int lo = min(e1, e0 + tid * per), hi = min(e1, lo + per);
            const size_t base = static_cast<size_t>(row) * p.V;
            float wt = 0.f;
            for (int v = lo; v < hi; ++v) wt += __expf(load_elem(p.target, p.t_fp32, base + v) * p.inv_t - mc);
            block_locate(wt, f, sh);
            if (tid == sh.owner) {
                const float T = sh.frac * wt;
                float cum = 0.f;
                int pick = -1, last = -1;
                for (int v = lo; v < hi; ++v) {
                    const float w = __expf(load_elem(p.target, p.t_fp32, base + v) * p.inv_t - mc);
                    if (!(w > 0.f)) continue;
                    last = v;
                    if (cum + w > T) {
                        pick = v;
                        break;
                    }
                    cum += w;
                }
                sh.part = pick >= 0 ? pick : last;
            }
            if (tid == 0 && sh.owner < 0) sh.part = -1;
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

}  // namespace

cudaError_t launch_draft_select(const DraftSelectParams& p, cudaStream_t s) {
    if (p.R <= 0) return cudaSuccess;
    return launch_pdl(draft_select_kernel, dim3(p.R), dim3(kSelThreads), 0, s, p);
}

cudaError_t launch_resample(const ResampleParams& p, cudaStream_t s) {
    if (p.R <= 0) return cudaSuccess;
    return launch_pdl(resample_kernel, dim3(p.R), dim3(kSelThreads), 0, s, p);
}

}  // namespace sdm
