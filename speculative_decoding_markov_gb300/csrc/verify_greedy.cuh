// verify_greedy.cuh - greedy verification of one request from the per-chunk
// argmax keys of its window rows ([DSpark notes] sec. 1: left-to-right
// acceptance, discard after the first mismatch, one bonus token; [SGLang]
// "three verify modes").  Run by the finalize kernel, one warp per request,
// after the argmax stream has written every row's per-chunk keys.
#pragma once
#include "device.cuh"
#include "internal.h"

namespace sdm {

// Argmax token of a row from its per-chunk partial keys (sixteen loads in
// flight at a time, through L2).
__device__ __forceinline__ int row_token(const unsigned long long* part, size_t row, int n_chunks) {
    const unsigned long long* q = part + row * n_chunks;
    unsigned long long k[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) k[j] = 0ull;
    for (int c0 = 0; c0 < n_chunks; c0 += 16) {
#pragma unroll
        for (int j = 0; j < 16; ++j)
            if (c0 + j < n_chunks) k[j] = umax64(k[j], __ldcg(q + c0 + j));
    }
#pragma unroll
    for (int j = 1; j < 16; ++j) k[0] = umax64(k[0], k[j]);
    return static_cast<int>(key_token(k[0]));
}

// Request i, resolved by one warp (lane p checks window rows p, p + 32, ...):
//   A = the first p < w with y_{p+1} != argmax of row p, else w;
//   commit a = A (min(A, budget) in CAP_ACCEPT) drafts and the target token
//   of row a; ceiling = A.
// The argmax stream wrote keys for rows [0, min(cu[R], rows_avail)) only
// (rows_avail: the rows the key buffer holds; total: cu[R]).  A request
// without rows, with rows past the buffer (SDM_DEV_CAPACITY) or past cu[R]
// (a non-monotone cu_seqlens, SDM_DEV_BAD_WINDOW) is flagged and commits one
// token (0) with accept 0, so no key this call did not write is read; a
// window longer than gamma is flagged and cut to gamma.
__device__ __forceinline__ void greedy_resolve(int i, int lane, int mode, const int32_t* cu, const int32_t* draft,
                                               const int32_t* budget, const unsigned long long* row_keys,
                                               int n_chunks, int gamma, int V, int rows_avail, int total,
                                               int32_t* accept, int32_t* ceiling, int32_t* out_tok, int32_t* n_out,
                                               int32_t* dev_status) {
    // the first 32 drafts load with the window's bounds (independent loads)
    const int32_t* y = draft + static_cast<size_t>(i) * gamma;
    const int y0 = lane < gamma ? y[lane] : -1;
    const int row0 = cu[i];
    const int row1 = cu[i + 1];
    int32_t* o = out_tok + static_cast<size_t>(i) * (gamma + 1);
    if (row1 <= row0 || row0 < 0 || row1 > rows_avail || row1 > total) {
        for (int p = lane; p <= gamma; p += 32) o[p] = p == 0 ? 0 : -1;
        if (lane == 0) {
            set_status(dev_status, row1 > rows_avail ? SDM_DEV_CAPACITY : SDM_DEV_BAD_WINDOW);
            accept[i] = 0;
            n_out[i] = 1;
            if (ceiling) ceiling[i] = 0;
        }
        return;
    }
    int w = row1 - row0 - 1;
    if (w > gamma) {
        if (lane == 0) set_status(dev_status, SDM_DEV_BAD_WINDOW);
        w = gamma;
    }
    int cap = w;
    if (mode == SDM_CAP_ACCEPT) {
        cap = budget[i];
        if (cap < 0 || cap > w) {
            if (lane == 0) set_status(dev_status, SDM_DEV_BAD_WINDOW);
            cap = cap < 0 ? 0 : w;
        }
    }
    // the first 32 window rows (the row after the last draft included) in
    // one round: lane p holds row p's target token
    const int t0 = lane <= w ? row_token(row_keys, static_cast<size_t>(row0 + lane), n_chunks) : -1;
    int A = w;
    for (int base = 0; base < w && A == w; base += 32) {
        const int p = base + lane;
        const int tp = base == 0 ? t0 : (p < w ? row_token(row_keys, static_cast<size_t>(row0 + p), n_chunks) : -1);
        const bool mism = p < w && (base == 0 ? y0 : y[p]) != tp;
        const unsigned bal = __ballot_sync(0xffffffffu, mism);
        if (bal) A = base + __ffs(bal) - 1;
    }
    const int a = A < cap ? A : cap;
    const int ta = __shfl_sync(0xffffffffu, t0, a & 31);
    for (int p = lane; p <= gamma; p += 32) {
        if (p < a) {
            o[p] = p < 32 ? y0 : y[p];   // p < 32: p is this lane
        } else if (p == a) {
            int t = a < 32 ? ta : row_token(row_keys, static_cast<size_t>(row0 + a), n_chunks);
            if (t < 0 || t >= V) {
                set_status(dev_status, SDM_DEV_BAD_TOKEN);
                t = 0;
            }
            o[p] = t;
        } else {
            o[p] = -1;
        }
    }
    if (lane == 0) {
        accept[i] = a;
        n_out[i] = a + 1;
        if (ceiling) ceiling[i] = A;
    }
}

}  // namespace sdm
