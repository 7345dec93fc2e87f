// observe.cu - the observability side of verification: the row list and the
// reductions around the soft-label GEMM passes (DSpark notes sec. 5.1: the
// confidence head's label is the single-token acceptance rate 1 - TV(q, p)),
// and the per-cycle statistics (SGLang "observability": acceptance ceilings,
// calibration; DSpark notes sec. 8.1: position d counts only where 1..d-1
// were accepted).
#include "device.cuh"
#include "internal.h"

namespace sdm {
namespace {

constexpr int kPrepThreads = 256;
constexpr int kRowWarps = 8;            // rows per CTA in the per-row reductions
constexpr int kObserveThreads = 1024;

// ---------------------------------------------------------------------------
// Row list of the soft-label passes.  Thread (i, p): window row p of request
// i becomes GEMM row g = cu[i] - i + p when p < w_i (every slot was marked
// unused, res_tok = -1, before this kernel).  Every label starts at -1; the
// target row's log-sum-exp is combined from the streaming partials here.
// ---------------------------------------------------------------------------
__global__ void label_prep_kernel(const int32_t* __restrict__ cu, const int32_t* __restrict__ anchor,
                                  const int32_t* __restrict__ draft, const float* __restrict__ lse_q,
                                  const float2* __restrict__ lse_part, int n_chunks, int R, int gamma, int V,
                                  int row_capacity, int32_t* res_req, int32_t* res_pos, int32_t* res_tok,
                                  int32_t* res_trow, float* res_lse_p, float* row_lse_q, float* label,
                                  int32_t* dev_status) {
    pdl_wait();
    pdl_trigger();
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    const int slots = R * gamma;
    if (t >= slots) return;
    const int i = t / gamma, p = t % gamma;
    label[t] = -1.f;
    const int c0 = cu[i];
    int w = cu[i + 1] - c0 - 1;
    if (w < 0 || w > gamma) {
        if (p == 0) set_status(dev_status, SDM_DEV_BAD_WINDOW);
        w = w < 0 ? 0 : gamma;
    }
    if (p >= w) return;
    const int g = c0 - i + p;
    if (g < 0 || g >= slots) {
        set_status(dev_status, SDM_DEV_BAD_WINDOW);
        return;
    }
    const int trow = c0 + p;
    const int prev = p == 0 ? anchor[i] : draft[static_cast<size_t>(i) * gamma + p - 1];
    // the log-sum-exp stream wrote partials for rows below min(cu[R], row_capacity) only
    const int total = cu[R];
    if (trow < 0 || trow >= row_capacity || trow >= total || prev < 0 || prev >= V) {
        set_status(dev_status, trow >= row_capacity ? SDM_DEV_CAPACITY
                               : (trow < 0 || trow >= total) ? SDM_DEV_BAD_WINDOW : SDM_DEV_BAD_TOKEN);
        res_tok[g] = -1;
        return;
    }
    res_req[g] = i;
    res_pos[g] = p;
    res_tok[g] = prev;
    res_trow[g] = trow;
    row_lse_q[g] = lse_q ? lse_q[static_cast<size_t>(i) * gamma + p] : 0.f;
    const float2* part = lse_part + static_cast<size_t>(trow) * n_chunks;
    float m = -INFINITY;
    for (int c = 0; c < n_chunks; ++c) m = fmaxf(m, part[c].x);
    double s = 0.0;   // fp32 terms, summed in fp64
    for (int c = 0; c < n_chunks; ++c) s += static_cast<double>(part[c].y * expf(part[c].x - m));
    res_lse_p[g] = static_cast<float>(static_cast<double>(m) + log(s));
}

__device__ __forceinline__ double warp_sum_f64(double s) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    return s;
}

// One warp per listed row: the row maximum of the partials first, then each
// partial's sum rescaled to it (an fp32 exponential) and summed in fp64, lanes
// taking partials lane, lane + 32, ... and a fixed butterfly combining them
// (the order does not depend on timing).
__global__ void label_lse_q_kernel(const float2* __restrict__ part, int n_part, int rows,
                                   const int32_t* __restrict__ res_tok, float* row_lse_q) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int g = blockIdx.x * kRowWarps + (threadIdx.x >> 5);
    if (g >= rows || res_tok[g] < 0) return;
    const float2* pr = part + static_cast<size_t>(g) * n_part;
    float m = -INFINITY;
    for (int k = lane; k < n_part; k += 32) {
        const float2 x = pr[k];
        if (x.y > 0.f) m = fmaxf(m, x.x);   // a thread that consumed no column left (-inf, 0)
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    double s = 0.0;
    for (int k = lane; k < n_part; k += 32) {
        const float2 x = pr[k];
        if (x.y > 0.f) s += static_cast<double>(x.y * expf(x.x - m));
    }
    s = warp_sum_f64(s);
    if (lane == 0) row_lse_q[g] = static_cast<float>(static_cast<double>(m) + log(s));
}

__global__ void label_finalize_kernel(const float2* __restrict__ part, int n_part, int rows,
                                      const int32_t* __restrict__ res_tok, const int32_t* __restrict__ res_req,
                                      const int32_t* __restrict__ res_pos, int gamma, float* label) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int g = blockIdx.x * kRowWarps + (threadIdx.x >> 5);
    if (g >= rows || res_tok[g] < 0) return;
    const float2* pr = part + static_cast<size_t>(g) * n_part;
    double s = 0.0;   // the per-thread fp32 partial sums, added in fp64
    for (int k = lane; k < n_part; k += 32) s += static_cast<double>(pr[k].y);
    s = warp_sum_f64(s);
    if (lane == 0) label[static_cast<size_t>(res_req[g]) * gamma + res_pos[g]] = static_cast<float>(s);
}

// ---------------------------------------------------------------------------
// Verify-cycle statistics, one CTA: counters in shared memory, one thread per
// request at a time.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kObserveThreads)
observe_kernel(const float* __restrict__ conf, const int32_t* __restrict__ cu, const int32_t* __restrict__ ceiling,
               const int32_t* __restrict__ cls, int R, int gamma, int n_class, int n_bins, int32_t* hist,
               int32_t* reached, int32_t* hits, int32_t* bin_n, int32_t* bin_hit, double* bin_conf, double* ece,
               int32_t* dev_status) {
    extern __shared__ __align__(16) uint8_t sm_raw[];
    double* s_conf = reinterpret_cast<double*>(sm_raw);
    int* s_bn = reinterpret_cast<int*>(s_conf + n_bins);
    int* s_bh = s_bn + n_bins;
    int* s_hist = s_bh + n_bins;
    int* s_reach = s_hist + n_class * (gamma + 1);
    int* s_hit = s_reach + n_class * gamma;
    const int n_int = 2 * n_bins + n_class * (3 * gamma + 1);
    for (int k = threadIdx.x; k < n_bins; k += blockDim.x) s_conf[k] = 0.0;
    for (int k = threadIdx.x; k < n_int; k += blockDim.x) s_bn[k] = 0;
    pdl_wait();
    pdl_trigger();
    __syncthreads();
    const float fb = static_cast<float>(n_bins);
    for (int i = threadIdx.x; i < R; i += blockDim.x) {
        const int c = cls[i];
        if (c < 0 || c >= n_class) {
            set_status(dev_status, SDM_DEV_BAD_CLASS);
            continue;
        }
        int w = cu[i + 1] - cu[i] - 1;
        int A = ceiling[i];
        if (w < 0 || w > gamma || A < 0 || A > w) {
            set_status(dev_status, SDM_DEV_BAD_WINDOW);
            w = w < 0 ? 0 : (w > gamma ? gamma : w);
            A = A < 0 ? 0 : (A > w ? w : A);
        }
        atomicAdd(&s_hist[c * (gamma + 1) + A], 1);
        const int last = A + 1 < w ? A + 1 : w;
        for (int d = 1; d <= last; ++d) {
            const int hit = d <= A;
            atomicAdd(&s_reach[c * gamma + d - 1], 1);
            if (hit) atomicAdd(&s_hit[c * gamma + d - 1], 1);
            float x = conf[static_cast<size_t>(i) * gamma + d - 1];
            x = fminf(fmaxf(x, 0.f), 1.f);            // NaN -> 0
            int b = static_cast<int>(floorf(__fmul_rn(x, fb)));
            b = b > n_bins - 1 ? n_bins - 1 : b;
            atomicAdd(&s_bn[b], 1);
            if (hit) atomicAdd(&s_bh[b], 1);
            atomicAdd(&s_conf[b], static_cast<double>(x));
        }
    }
    __syncthreads();
    for (int k = threadIdx.x; k < n_class * (gamma + 1); k += blockDim.x) hist[k] = s_hist[k];
    for (int k = threadIdx.x; k < n_class * gamma; k += blockDim.x) {
        reached[k] = s_reach[k];
        hits[k] = s_hit[k];
    }
    for (int k = threadIdx.x; k < n_bins; k += blockDim.x) {
        bin_n[k] = s_bn[k];
        bin_hit[k] = s_bh[k];
        bin_conf[k] = s_conf[k];
    }
    if (threadIdx.x == 0) {   // bins in order, as the definition sums them
        long long n = 0;
        double e = 0.0;
        for (int b = 0; b < n_bins; ++b) {
            n += s_bn[b];
            e += fabs(static_cast<double>(s_bh[b]) - s_conf[b]);
        }
        *ece = n > 0 ? e / static_cast<double>(n) : 0.0;
    }
}

}  // namespace

size_t observe_smem_bytes(int gamma, int n_class, int n_bins) {
    return static_cast<size_t>(n_bins) * 8 +
           static_cast<size_t>(2 * n_bins + n_class * (3 * gamma + 1)) * 4;
}

cudaError_t launch_label_prep(const int32_t* cu, const int32_t* anchor, const int32_t* draft, const float* lse_q,
                              const float2* lse_part, int n_chunks, int R, int gamma, int V, int row_capacity,
                              int32_t* res_req, int32_t* res_pos, int32_t* res_tok, int32_t* res_trow,
                              float* res_lse_p, float* row_lse_q, float* label, int32_t* dev_status, cudaStream_t s) {
    const int slots = R * gamma;
    return launch_pdl(label_prep_kernel, dim3((slots + kPrepThreads - 1) / kPrepThreads), dim3(kPrepThreads), 0, s,
                      cu, anchor, draft, lse_q, lse_part, n_chunks, R, gamma, V, row_capacity, res_req, res_pos,
                      res_tok, res_trow, res_lse_p, row_lse_q, label, dev_status);
}

cudaError_t launch_label_lse_q(const float2* part, int n_part, int rows, const int32_t* res_tok, float* row_lse_q,
                               cudaStream_t s) {
    return launch_pdl(label_lse_q_kernel, dim3((rows + kRowWarps - 1) / kRowWarps), dim3(32 * kRowWarps), 0, s, part,
                      n_part, rows, res_tok, row_lse_q);
}

cudaError_t launch_label_finalize(const float2* part, int n_part, int rows, const int32_t* res_tok,
                                  const int32_t* res_req, const int32_t* res_pos, int gamma, float* label,
                                  cudaStream_t s) {
    return launch_pdl(label_finalize_kernel, dim3((rows + kRowWarps - 1) / kRowWarps), dim3(32 * kRowWarps), 0, s,
                      part, n_part, rows, res_tok, res_req, res_pos, gamma, label);
}

cudaError_t launch_observe(const float* conf, const int32_t* cu, const int32_t* ceiling, const int32_t* cls, int R,
                           int gamma, int n_class, int n_bins, int32_t* hist, int32_t* reached, int32_t* hits,
                           int32_t* bin_n, int32_t* bin_hit, double* bin_conf, double* ece, int32_t* dev_status,
                           cudaStream_t s) {
    const size_t smem = observe_smem_bytes(gamma, n_class, n_bins);
    return launch_pdl(observe_kernel, dim3(1), dim3(kObserveThreads), smem, s, conf, cu, ceiling, cls, R, gamma,
                      n_class, n_bins, hist, reached, hits, bin_n, bin_hit, bin_conf, ece, dev_status);
}

}  // namespace sdm
