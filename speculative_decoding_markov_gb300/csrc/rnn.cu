// rnn.cu - the RNN sequential head's memo update (DSpark notes sec. 4, "RNN
// head": a memo that carries the whole draft so far, updated once per step
// from the previous memo, the previous word and the current backbone state):
//     m_d = tanh(A m_{d-1} + U[y_{d-1}] + x_d),   m_0 = 0,
// kept in fp32 between steps and handed to the tensor-core projection as
// bf16(m_d) (the A rows of the Markov GEMM, in place of U[y_{d-1}]).
#include "device.cuh"
#include "internal.h"

namespace sdm {
namespace {

constexpr int kRnnThreads = 256;   // 8 warps; r <= 256

__device__ __forceinline__ uint16_t bf16_rne(float f) {
    uint32_t b = __float_as_uint(f);
    if ((b & 0x7F800000u) == 0x7F800000u && (b & 0x007FFFFFu)) return static_cast<uint16_t>((b >> 16) | 0x40u);
    b += 0x7FFFu + ((b >> 16) & 1u);
    return static_cast<uint16_t>(b >> 16);
}

// One CTA per request: the previous memo in shared memory; warp w forms rows
// j = w + 8 t (t < r / 8 <= 32) of A m, lane l holding K elements 8 l ..
// 8 l + 7, the loads of 16 rows issued before any is used; a transposing
// butterfly leaves row t's sum in lane t, which finishes that row.
__global__ void __launch_bounds__(kRnnThreads) rnn_step_kernel(const RnnStepParams p) {
    __shared__ float sm[256], sux[256];   // previous memo; U[y_{d-1}] + x_d
    const int i = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_wait();
    pdl_trigger();
    for (int j = tid; j < p.r; j += blockDim.x) sm[j] = p.d == 1 ? 0.f : p.m[static_cast<size_t>(i) * p.r + j];
    int prev = p.anchor[i];
    if (p.d > 1)
        prev = p.keys ? static_cast<int>(key_token(p.keys[static_cast<size_t>(p.d - 2) * p.R + i]))
                      : p.tokens[static_cast<size_t>(i) * p.B + (p.d - 2)];
    if (prev < 0 || prev >= p.V) {
        if (tid == 0) set_status(p.dev_status, SDM_DEV_BAD_TOKEN);
        prev = 0;
    }
    {   // all threads are past the token read; stage U[prev] + x_d for the row sums
        __syncthreads();
        const uint16_t* urow = p.U + static_cast<size_t>(prev) * p.r;
        const uint16_t* xrow = p.X + (static_cast<size_t>(i) * p.B + (p.d - 1)) * p.r;
        for (int j = tid; j < p.r; j += blockDim.x) sux[j] = bf16_bits_to_float(urow[j]) + bf16_bits_to_float(xrow[j]);
        __syncthreads();
    }
    const int k0 = lane * 8;
    const bool kl = k0 < p.r;
    float mk[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) mk[q] = kl ? sm[k0 + q] : 0.f;
    // partial dot products of the warp's rows t = 0..31 (row j = warp + 8 t;
    // rows past r / 8 are zero) over this lane's 8 K elements
    const int nt = p.r / 8;
    float acc[32];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint4 a[16];
#pragma unroll
        for (int b = 0; b < 16; ++b) {
            const int t = h * 16 + b;
            a[b] = (kl && t < nt) ? __ldg(reinterpret_cast<const uint4*>(p.A + static_cast<size_t>(warp + 8 * t) * p.r + k0))
                                  : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int b = 0; b < 16; ++b) {
            const uint32_t w[4] = {a[b].x, a[b].y, a[b].z, a[b].w};
            float x = 0.f;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                x = fmaf(__uint_as_float(w[q] << 16), mk[2 * q], x);
                x = fmaf(__uint_as_float(w[q] & 0xffff0000u), mk[2 * q + 1], x);
            }
            acc[h * 16 + b] = x;
        }
    }
    // transposing butterfly: after the stage with offset s every lane keeps
    // the half of its rows selected by bit s of its lane id, summed with its
    // partner's; at the end lane l holds the full sum of row t = l
#pragma unroll
    for (int s = 16; s >= 1; s >>= 1) {
        const bool up = (lane & s) != 0;
#pragma unroll
        for (int t = 0; t < s; ++t) {
            const float send = up ? acc[t] : acc[t + s];
            const float keep = up ? acc[t + s] : acc[t];
            acc[t] = keep + __shfl_xor_sync(0xffffffffu, send, s);
        }
    }
    if (lane < nt) {
        const int j = warp + 8 * lane;
        const float mj = tanhf(acc[0] + sux[j]);
        p.m[static_cast<size_t>(i) * p.r + j] = mj;
        p.a_rows[static_cast<size_t>(i) * p.r + j] = bf16_rne(mj);
        if (p.memo_out) p.memo_out[(static_cast<size_t>(i) * p.B + (p.d - 1)) * p.r + j] = mj;
    }
}

}  // namespace

cudaError_t launch_rnn_step(const RnnStepParams& p, cudaStream_t s) {
    return launch_pdl(rnn_step_kernel, dim3(p.R), dim3(kRnnThreads), 0, s, p);
}

}  // namespace sdm
