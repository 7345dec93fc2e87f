// stream.cu - HBM-bound reductions over vocab rows of the packed target
// logits: argmax (greedy verification, PCTree verification) and log-sum-exp
// partials per chunk (rejection sampling: the normaliser of p, and the chunk
// weights the bonus draw walks).
//
// Work item = (row, chunk of `chunk` ids).  A persistent grid of CTAs walks
// the items; each thread streams 16-byte vectors (8 bf16 or 4 fp32) with four
// loads in flight and cache-streaming hints, so a row is read from HBM exactly
// once.  The number of rows can come from device memory (cu_seqlens[R]), so a
// captured launch covers any packed total up to the tier.
#include "device.cuh"
#include "internal.h"

namespace sdm {
namespace {

constexpr int kThreads = 256;
// Vectors in flight per thread: the log-sum-exp stream keeps a whole 32 KB
// item in flight per CTA (measured 10 % faster on fp32 rows); the argmax
// stream does better with more CTAs per SM at half that.
template <int OP>
constexpr int unroll_of() { return OP == STREAM_LSE ? 8 : 4; }

struct Argmax {
    float best = -INFINITY;
    uint32_t bv = 0;
    __device__ __forceinline__ void add(float x, uint32_t v) {
        if (x > best) {   // ids arrive in increasing order per thread: ties keep the lowest
            best = x;
            bv = v;
        }
    }
};

struct OnlineLse {
    float m = -INFINITY;
    float s = 0.f;
    template <int N>
    __device__ __forceinline__ void add(const float (&x)[N]) {
        float mx = x[0];
#pragma unroll
        for (int i = 1; i < N; ++i) mx = fmaxf(mx, x[i]);
        if (mx > m) {
            s *= __expf(m - mx);
            m = mx;
        }
#pragma unroll
        for (int i = 0; i < N; ++i) s += __expf(x[i] - m);
    }
};

template <int OP, int FP32>
__global__ void __launch_bounds__(kThreads) row_stream_kernel(const StreamParams p) {
    constexpr int VEC = FP32 ? 4 : 8;
    constexpr int kUnroll = unroll_of<OP>();
    __shared__ unsigned long long red_key[kThreads / 32];
    __shared__ float red_m[kThreads / 32], red_s[kThreads / 32];
    pdl_wait();
    pdl_trigger();
    const int n_items = p.count ? min(max(*p.count, 0), p.n_items) : p.n_items;   // never past the buffer
    const long long total = static_cast<long long>(n_items) * p.n_chunks;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    for (long long w = blockIdx.x; w < total; w += gridDim.x) {
        const int item = static_cast<int>(w / p.n_chunks);
        const int chunk = static_cast<int>(w % p.n_chunks);
        const int row = p.row_of ? p.row_of[item] : item;
        if (row < 0) continue;
        const int v_begin = chunk * p.chunk;
        const int v_end = min(p.V, v_begin + p.chunk);
        const int n_vec = (v_end - v_begin) / VEC;
        const size_t esz = FP32 ? 4 : 2;
        const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(p.base) +
                                                          (static_cast<size_t>(row) * p.V + v_begin) * esz);

        Argmax am;
        OnlineLse ls;
        for (int i0 = threadIdx.x; i0 < n_vec; i0 += kThreads * kUnroll) {
            uint4 x[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int i = i0 + u * kThreads;
                if (i < n_vec) x[u] = __ldcs(src + i);
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int i = i0 + u * kThreads;
                if (i >= n_vec) break;
                const uint32_t v0 = static_cast<uint32_t>(v_begin + i * VEC);
                float val[VEC];
                if (FP32) {
                    val[0] = __uint_as_float(x[u].x);
                    val[1] = __uint_as_float(x[u].y);
                    val[2] = __uint_as_float(x[u].z);
                    val[3] = __uint_as_float(x[u].w);
                } else {
                    const uint32_t ww[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        val[2 * q] = __uint_as_float(ww[q] << 16);
                        val[2 * q + 1] = __uint_as_float(ww[q] & 0xffff0000u);
                    }
                }
                if (OP == STREAM_ARGMAX) {
#pragma unroll
                    for (int q = 0; q < VEC; ++q) am.add(val[q], v0 + q);
                } else {
#pragma unroll
                    for (int q = 0; q < VEC; ++q) val[q] *= p.inv_t;
                    ls.add(val);
                }
            }
        }
        if (OP == STREAM_LSE) {
            OnlineLse r = ls;
            Lse t = warp_lse(Lse{r.m, r.s});
            if (lane == 0) {
                red_m[warp] = t.m;
                red_s[warp] = t.s;
            }
            __syncthreads();
            if (threadIdx.x == 0) {
                Lse acc{red_m[0], red_s[0]};
                for (int q = 1; q < kThreads / 32; ++q) acc = lse_merge(acc, Lse{red_m[q], red_s[q]});
                p.part[static_cast<size_t>(item) * p.n_chunks + chunk] = make_float2(acc.m, acc.s);
            }
            __syncthreads();
        } else {
            unsigned long long k = warp_max_u64(argmax_key(am.best, am.bv));
            if (lane == 0) red_key[warp] = k;
            __syncthreads();
            if (threadIdx.x == 0) {
                unsigned long long acc = red_key[0];
                for (int q = 1; q < kThreads / 32; ++q) acc = umax64(acc, red_key[q]);
                p.keys[static_cast<size_t>(item) * p.n_chunks + chunk] = acc;   // one partial per chunk
            }
            __syncthreads();
        }
    }
}

template <int OP>
cudaError_t launch_op(const StreamParams& p, int max_items, cudaStream_t s) {
    const long long work = static_cast<long long>(max_items) * p.n_chunks;
    if (work <= 0) return cudaSuccess;
    const int grid = static_cast<int>(work < 8LL * num_sms() ? work : 8LL * num_sms());
    return p.fp32 ? launch_pdl(row_stream_kernel<OP, 1>, dim3(grid), dim3(kThreads), 0, s, p)
                  : launch_pdl(row_stream_kernel<OP, 0>, dim3(grid), dim3(kThreads), 0, s, p);
}

}  // namespace

cudaError_t launch_stream(int op, const StreamParams& p, int max_items, cudaStream_t s) {
    switch (op) {
        case STREAM_ARGMAX: return launch_op<STREAM_ARGMAX>(p, max_items, s);
        case STREAM_LSE: return launch_op<STREAM_LSE>(p, max_items, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace sdm
