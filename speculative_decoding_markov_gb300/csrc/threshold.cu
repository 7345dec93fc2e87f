// threshold.cu - the conventional fixed-threshold verify length and its sweep
// (DSpark notes sec. 5.2: a fixed threshold on the confidences decides how
// many drafts are verified; sec. 8.3, Fig. 5: sweeping the threshold, 0 =
// the whole block).
#include "device.cuh"
#include "internal.h"

namespace sdm {
namespace {

constexpr int kThrThreads = 1024;
constexpr int kSweepThreads = 256;

// The longest prefix of c[0..gamma) whose every confidence is >= tau (an
// fp32 comparison; a NaN ends the prefix).
__device__ __forceinline__ int threshold_len(const float* c, int gamma, float tau) {
    int n = 0;
    while (n < gamma && c[n] >= tau) ++n;
    return n;
}

__global__ void __launch_bounds__(kThrThreads)
schedule_threshold_kernel(const float* __restrict__ conf, int R, int gamma, float tau, int32_t* budget,
                          int32_t* total_tokens) {
    __shared__ int s_total;
    if (threadIdx.x == 0) s_total = 0;
    pdl_wait();
    pdl_trigger();
    __syncthreads();
    int local = 0;
    for (int i = threadIdx.x; i < R; i += blockDim.x) {
        const int n = threshold_len(conf + static_cast<size_t>(i) * gamma, gamma, tau);
        budget[i] = n;
        local += n;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) local += __shfl_xor_sync(0xffffffffu, local, o);
    if ((threadIdx.x & 31) == 0) atomicAdd(&s_total, local);
    __syncthreads();
    if (threadIdx.x == 0) *total_tokens = R + s_total;   // every request sends its root token
}

// One CTA per threshold.  The expected count is summed exactly: a survival
// S >= 2^-24 is a whole multiple of 2^-47, so S 2^48 is an integer (formed in
// fp32, a power-of-two scaling) and the integer sum does not depend on order.
__global__ void __launch_bounds__(kSweepThreads)
threshold_sweep_kernel(const float* __restrict__ conf, const int32_t* __restrict__ ceiling, int R, int gamma,
                       const float* __restrict__ taus, int32_t* drafts, int32_t* accepted, double* expected) {
    __shared__ int s_nd, s_na;
    __shared__ unsigned long long s_units;
    if (threadIdx.x == 0) {
        s_nd = s_na = 0;
        s_units = 0ull;
    }
    pdl_wait();
    pdl_trigger();
    __syncthreads();
    const float tau = taus[blockIdx.x];
    const float tiny = 1.0f / 16777216.0f;      // 2^-24
    const float scale = 281474976710656.0f;     // 2^48
    int nd = 0, na = 0;
    unsigned long long units = 0ull;
    for (int i = threadIdx.x; i < R; i += blockDim.x) {
        const float* c = conf + static_cast<size_t>(i) * gamma;
        const int n = threshold_len(c, gamma, tau);
        float s = 1.0f;
        for (int d = 0; d < n; ++d) {
            s = __fmul_rn(s, c[d]);
            if (s >= tiny) units += static_cast<unsigned long long>(__float2ll_rn(s * scale));
        }
        nd += n;
        if (ceiling) na += min(ceiling[i], n);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        nd += __shfl_xor_sync(0xffffffffu, nd, o);
        na += __shfl_xor_sync(0xffffffffu, na, o);
        units += __shfl_xor_sync(0xffffffffu, units, o);
    }
    if ((threadIdx.x & 31) == 0) {
        atomicAdd(&s_nd, nd);
        atomicAdd(&s_na, na);
        atomicAdd(&s_units, units);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        drafts[blockIdx.x] = s_nd;
        accepted[blockIdx.x] = ceiling ? s_na : -1;
        expected[blockIdx.x] = static_cast<double>(static_cast<long long>(s_units)) * 3.552713678800501e-15;   // 2^-48
    }
}

}  // namespace

cudaError_t launch_schedule_threshold(const float* conf, int R, int gamma, float tau, int32_t* budget,
                                      int32_t* total_tokens, cudaStream_t s) {
    return launch_pdl(schedule_threshold_kernel, dim3(1), dim3(kThrThreads), 0, s, conf, R, gamma, tau, budget,
                      total_tokens);
}

cudaError_t launch_threshold_sweep(const float* conf, const int32_t* ceiling, int R, int gamma, const float* taus,
                                   int K, int32_t* drafts, int32_t* accepted, double* expected, cudaStream_t s) {
    return launch_pdl(threshold_sweep_kernel, dim3(K), dim3(kSweepThreads), 0, s, conf, ceiling, R, gamma, taus,
                      drafts, accepted, expected);
}

}  // namespace sdm
