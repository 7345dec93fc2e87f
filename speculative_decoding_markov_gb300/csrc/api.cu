// api.cu - the extern "C" entry points of libsdm.so (declared in include/sdm.h):
// argument validation, tensor-map encoding, workspace carving and the launch
// sequence of each operation.  Every operation is enqueued on the caller's
// stream and allocates nothing.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>

#include "internal.h"

namespace {
using namespace sdm;

constexpr int kMaxGx = 256;           // upper bound of vocab splits per GEMM launch
constexpr int kMaxSampleV = 524288;   // 32768 records of 16 ids: the select kernels' chunk tables
inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct Carver {
    uint8_t* base;
    size_t off = 0;
    template <typename T>
    T* take(size_t count) {
        T* p = reinterpret_cast<T*>(base + off);
        off = align256(off + count * sizeof(T));
        return p;
    }
};

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// W [r, V] bf16 as a 2-D map (V innermost), box 64 ids x 64 K rows, 128-byte swizzle.
bool map_w(CUtensorMap* m, const uint16_t* W, int r, int V) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(V), static_cast<cuuint64_t>(r)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(V) * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(kBoxN), 64u};
    cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(W), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// L [R, B, V] as a 3-D map (V, B, R), box (128 bytes of V) x 1 x l_rows.
bool map_l(CUtensorMap* m, const void* L, int fp32, int R, int B, int V, int l_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t es = fp32 ? 4 : 2;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(V), static_cast<cuuint64_t>(B), static_cast<cuuint64_t>(R)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(V) * es, static_cast<cuuint64_t>(V) * B * es};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(fp32 ? 32 : 64), 1, static_cast<cuuint32_t>(l_rows)};
    cuuint32_t el[3] = {1, 1, 1};
    return fn(m, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(L),
              dims, strides, box, el, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline int gemm_grid_x(int n_tiles, int grid_y) {
    int gx = std::max(1, num_sms() / grid_y);
    gx = std::min(gx, n_tiles);
    return std::min(gx, kMaxGx);
}

inline bool vocab_ok(int V) { return V >= 8 && V % 8 == 0; }
inline bool rank_ok(int r) { return r >= 64 && r <= 256 && r % 64 == 0; }

#define SDM_CHECK_CUDA(x)                          \
    do {                                           \
        if ((x) != cudaSuccess) return SDM_ERR_CUDA; \
    } while (0)

// Row stride of the (m, s) records, one per 16-column block: rounded up to an
// even count so that every row starts on a 16-byte boundary (bulk copies).
inline int n_blocks16(int V) { return (((V + 15) / 16) + 1) & ~1; }

// greedy: argmax keys [B][R]; sampling: one (m, s) record per request and
// 16-column block, reused by every step
size_t ws_chain_dense(int R, int B, int V) {
    return align256(static_cast<size_t>(B) * R * 8) + align256(static_cast<size_t>(R) * n_blocks16(V) * 8);
}

// candidate lists of the pruned greedy chain (sized for the larger fp32 split)
size_t ws_chain_pruned(int R, int B, int V) {
    const size_t segs = static_cast<size_t>(R) * B * pruned_chunks(V, 1);
    return align256(segs * kSegCap * 8) + align256(segs * 4) + align256(segs * 4);
}

size_t ws_chain(int R, int B, int V) { return std::max(ws_chain_dense(R, B, V), ws_chain_pruned(R, B, V)); }

// RNN head: the dense chain's scratch, then the fp32 memo and its bf16 rows
size_t ws_chain_rnn(int R, int B, int V, int r) {
    return ws_chain_dense(R, B, V) + align256(static_cast<size_t>(R) * r * 4) + align256(static_cast<size_t>(R) * r * 2);
}

// frontier and pool, then either the record path's block records [rows][nb],
// per-row top-k and log-sum-exp, or the pruned path's scan lists (sized for
// the larger fp32 chunk count) and the GEMM's log-sum-exp partials
size_t ws_tree_common(int R, int B, int P) {
    const size_t rows = static_cast<size_t>(R) * P;
    const size_t pool = static_cast<size_t>(R) * (1 + static_cast<size_t>(P) * B);
    return 3 * align256(rows * 4) + align256(R * 4) + 4 * align256(pool * 4) + align256(R * 4);
}

int tree_n_part(int R, int P, int V) {   // one partial per GEMM CTA column: the most either sub-tile layout gives
    const int gy = (R * P + kTileM - 1) / kTileM;
    const int gy2 = (R * P + 2 * kTileM - 1) / (2 * kTileM);
    return std::max(gemm_grid_x((V + kTileN - 1) / kTileN, gy), gemm_grid_x((V + kTileN - 1) / kTileN, gy2));
}

size_t ws_tree(int R, int B, int P, int V) {
    const size_t rows = static_cast<size_t>(R) * P;
    const size_t records = align256(rows * n_blocks16(V) * 8) + align256(rows * kMaxTopK * 8) + align256(rows * 4);
    const size_t lrows = static_cast<size_t>(R) * B;
    const size_t pruned = ws_chain_pruned(R, B, V) + align256(rows * tree_n_part(R, P, V) * 8) +
                          align256(lrows * kTreeKeep * 8) + 3 * align256(lrows * 4);
    return ws_tree_common(R, B, P) + std::max(records, pruned);
}

size_t ws_verify(int R, int rows, int V) {
    const int nc = n_chunks_of(V, 0) > n_chunks_of(V, 1) ? n_chunks_of(V, 0) : n_chunks_of(V, 1);
    return align256(static_cast<size_t>(rows) * nc * 8) + align256(static_cast<size_t>(rows) * nc * 8) +
           6 * align256(static_cast<size_t>(R) * 4) + align256(static_cast<size_t>(R) * n_blocks16(V) * 8);
}

// soft label: target LSE partials, the row list, and one partial per listed
// row, GEMM CTA column and column group
int label_n_part(int R, int gamma, int V) {
    const int rows = R * gamma;
    const int gy = (rows + kTileM - 1) / kTileM;
    return gemm_grid_x((V + kTileN - 1) / kTileN, gy) * kColGroups;
}

size_t ws_tv_label(int R, int gamma, int V, int row_capacity) {
    const int nc = std::max(n_chunks_of(V, 0), n_chunks_of(V, 1));
    const size_t slots = static_cast<size_t>(R) * gamma;
    return align256(static_cast<size_t>(row_capacity) * nc * 8) + 6 * align256(slots * 4) +
           align256(slots * label_n_part(R, gamma, V) * 8);
}

// The dense chain draft: per step one tensor-core GEMM over all requests
// (argmax keys, or block records and an inverse-CDF select).  With rnn set,
// each step first updates the RNN head's memo and the GEMM's A rows are the
// memo's (scratch after the chain's: fp32 memo [R, r], bf16 rows [R, r]).
sdm_status draft_chain_dense(const void* L, sdm_dtype dtL, const uint16_t* U, const uint16_t* W,
                             const RnnStepParams* rnn, const int32_t* anchor, int R, int B, int V, int r,
                             sdm_decode decode, float temperature, sdm_rng rng, int32_t* tokens, float* logq,
                             float* lse, void* ws, int32_t* dev_status, cudaStream_t s) {
    Carver c{static_cast<uint8_t*>(ws)};
    auto* keys = c.take<unsigned long long>(static_cast<size_t>(B) * R);
    const int nb = n_blocks16(V);
    auto* blk = c.take<float2>(static_cast<size_t>(R) * nb);

    RnnStepParams rp;
    std::memset(&rp, 0, sizeof rp);
    if (rnn) {   // the memo state and its bf16 rows follow the chain's scratch
        rp = *rnn;
        rp.m = c.take<float>(static_cast<size_t>(R) * r);
        rp.a_rows = c.take<uint16_t>(static_cast<size_t>(R) * r);
        rp.R = R;
        rp.B = B;
        rp.V = V;
        rp.r = r;
        rp.anchor = anchor;
        rp.keys = decode == SDM_GREEDY ? keys : nullptr;
        rp.tokens = tokens;
        rp.dev_status = dev_status;
    }
    const int fp32 = dtL == SDM_FP32;
    const int l_rows = std::min(R, kTileM);
    CUtensorMap tmW, tmL;
    if (!map_w(&tmW, W, r, V) || !map_l(&tmL, L, fp32, R, B, V, l_rows)) return SDM_ERR_CUDA;
    const int mode = decode == SDM_GREEDY ? MODE_CHAIN_GREEDY : MODE_CHAIN_SAMPLE;
    const int n_tiles = (V + kTileN - 1) / kTileN;
    const int gy = (R + kTileM - 1) / kTileM;
    const int gx = gemm_grid_x(n_tiles, gy);

    GemmParams p;
    std::memset(&p, 0, sizeof p);
    p.rows = R;
    p.R = R;
    p.B = B;
    p.V = V;
    p.r = r;
    p.n_tiles = n_tiles;
    p.l_fp32 = fp32;
    p.l_rows = l_rows;
    p.P = 1;
    p.k = 1;
    gemm_pick_stages(p, mode);
    p.inv_t = decode == SDM_SAMPLE ? 1.0f / temperature : 1.0f;
    p.U = U;
    p.a_rows = rnn ? rp.a_rows : nullptr;
    p.anchor = anchor;
    p.keys = keys;
    p.tok_in = tokens;
    p.blk = blk;
    p.nb = nb;
    p.dev_status = dev_status;

    if (decode == SDM_GREEDY) {
        SDM_CHECK_CUDA(launch_fill_u64(keys, static_cast<size_t>(B) * R, 0ull, s));
        for (int d = 1; d <= B; ++d) {
            p.d = d;
            if (rnn) {
                rp.d = d;
                SDM_CHECK_CUDA(launch_rnn_step(rp, s));
            }
            SDM_CHECK_CUDA(launch_markov_gemm(mode, tmW, tmL, p, gx, gy, s));
        }
        SDM_CHECK_CUDA(launch_chain_finalize(keys, R, B, V, tokens, dev_status, s));
        return SDM_OK;
    }
    // sampling: per step the GEMM writes the block records, then one CTA per
    // request draws y_d by the inverse CDF (the next step's GEMM reads it)
    DraftSelectParams sp;
    std::memset(&sp, 0, sizeof sp);
    sp.blk = blk;
    sp.nb = nb;
    sp.R = R;
    sp.B = B;
    sp.V = V;
    sp.r = r;
    sp.L = L;
    sp.l_fp32 = fp32;
    sp.U = U;
    sp.W = W;
    sp.a_rows = p.a_rows;
    sp.anchor = anchor;
    sp.inv_t = p.inv_t;
    sp.k0 = static_cast<uint32_t>(rng.seed);
    sp.k1 = static_cast<uint32_t>(rng.seed >> 32);
    sp.cycle = static_cast<uint32_t>(rng.cycle);
    sp.tokens = tokens;
    sp.logq = logq;
    sp.lse = lse;
    sp.dev_status = dev_status;
    for (int d = 1; d <= B; ++d) {
        p.d = d;
        sp.d = d;
        if (rnn) {
            rp.d = d;
            SDM_CHECK_CUDA(launch_rnn_step(rp, s));
        }
        SDM_CHECK_CUDA(launch_markov_gemm(mode, tmW, tmL, p, gx, gy, s));
        SDM_CHECK_CUDA(launch_draft_select(sp, s));
    }
    return SDM_OK;
}

}  // namespace

extern "C" {

size_t sdm_workspace_size(int op, int R, int B, int V, int r, int P, int k, int N) {
    (void)r;
    (void)k;
    if (R <= 0) return 0;
    switch (op) {
        case SDM_OP_DRAFT_CHAIN: return ws_chain(R, B, V);
        case SDM_OP_DRAFT_TREE: return ws_tree(R, B, P, V);
        case SDM_OP_VERIFY: return ws_verify(R, P, V);
        case SDM_OP_TV_LABEL: return ws_tv_label(R, B, V, P);
        case SDM_OP_DRAFT_CHAIN_RNN: return ws_chain_rnn(R, B, V, r);
        case SDM_OP_VERIFY_TREE:
            return align256(static_cast<size_t>(R) * (N + 1) * 8 * std::max(n_chunks_of(V, 0), n_chunks_of(V, 1)));
        default: return 0;
    }
}

const char* sdm_status_str(sdm_status st) {
    switch (st) {
        case SDM_OK: return "ok";
        case SDM_ERR_INVALID_ARG: return "invalid argument";
        case SDM_ERR_UNSUPPORTED: return "unsupported shape or alignment";
        case SDM_ERR_TIER_OVERFLOW: return "packed total above every tier";
        case SDM_ERR_CUDA: return "CUDA error";
        case SDM_ERR_WORKSPACE: return "workspace missing or too small";
        case SDM_ERR_DEVICE: return "device-side input check failed";
        case SDM_ERR_TIMEOUT: return "a bounded device wait ran out";
        default: return "unknown status";
    }
}

sdm_status sdm_status_of_device(int32_t bits) {
    if (bits & SDM_DEV_TIMEOUT) return SDM_ERR_TIMEOUT;
    if (bits & SDM_DEV_TIER_OVERFLOW) return SDM_ERR_TIER_OVERFLOW;
    if (bits & ~static_cast<int32_t>(SDM_DEV_TIER_UNCAPTURED)) return SDM_ERR_DEVICE;
    return SDM_OK;
}

int sdm_version(void) { return 100; }

size_t sdm_markov_prepared_size(int V, int r) {
    if (V <= 0 || r <= 0) return 0;
    return align256(static_cast<size_t>(V) * r * 2) + 3 * align256(static_cast<size_t>(V) * 4) + 3 * 256;
}

sdm_status sdm_markov_prepare(const uint16_t* U, const uint16_t* W, int V, int r, void* prepared,
                              size_t prepared_bytes, int32_t* dev_status, void* stream) {
    if (!U || !W || !prepared || V <= 0 || r <= 0) return SDM_ERR_INVALID_ARG;
    if (!vocab_ok(V) || !rank_ok(r) || !aligned16(U) || !aligned16(W) || !aligned16(prepared))
        return SDM_ERR_UNSUPPORTED;
    if (prepared_bytes < sdm_markov_prepared_size(V, r)) return SDM_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    Carver c{static_cast<uint8_t*>(prepared)};
    uint16_t* Wt = c.take<uint16_t>(static_cast<size_t>(V) * r);
    float* c_bound = c.take<float>(V);
    float* u_norm = c.take<float>(V);
    unsigned int* absmax = c.take<unsigned int>(V);
    float* c_max = c.take<float>(1);
    float* n_max = c.take<float>(1);
    float* u_max = c.take<float>(1);
    SDM_CHECK_CUDA(launch_markov_prepare(U, W, V, r, Wt, u_norm, n_max, u_max, absmax, s));
    // A(y) = max_v |U[y] . W[:, v]| for every token y: the Markov GEMM with
    // GEMM row y = token y and an absolute-maximum epilogue
    CUtensorMap tmW;
    if (!map_w(&tmW, W, r, V)) return SDM_ERR_CUDA;
    GemmParams p;
    std::memset(&p, 0, sizeof p);
    p.rows = V;
    p.R = V;
    p.B = 1;
    p.V = V;
    p.r = r;
    p.n_tiles = (V + kTileN - 1) / kTileN;
    p.l_rows = 1;
    p.P = 1;
    p.k = 1;
    p.d = 1;
    p.inv_t = 1.0f;
    gemm_pick_stages(p, MODE_ABSMAX);
    p.U = U;
    p.absmax_bits = absmax;
    p.dev_status = dev_status;
    const int gy = (V + kTileM - 1) / kTileM;
    const int gx = gemm_grid_x(p.n_tiles, gy);
    SDM_CHECK_CUDA(launch_markov_gemm(MODE_ABSMAX, tmW, tmW, p, gx, gy, s));
    SDM_CHECK_CUDA(launch_markov_bounds(absmax, u_norm, n_max, V, r, c_bound, c_max, s));
    return SDM_OK;
}

sdm_status sdm_draft_chain(const void* L, sdm_dtype dtL, const uint16_t* U, const uint16_t* W,
                           const void* prepared, const int32_t* anchor, int R, int B, int V, int r,
                           sdm_decode decode, float temperature, sdm_rng rng, int32_t* tokens, float* logq,
                           float* lse, void* ws, size_t ws_bytes, int32_t* dev_status, void* stream) {
    if (!L || !U || !W || !anchor || !tokens || R <= 0 || B <= 0 || V <= 0 || r <= 0) return SDM_ERR_INVALID_ARG;
    if (dtL != SDM_BF16 && dtL != SDM_FP32) return SDM_ERR_INVALID_ARG;
    if (decode != SDM_GREEDY && decode != SDM_SAMPLE) return SDM_ERR_INVALID_ARG;
    if (decode == SDM_SAMPLE && !(temperature > 0.f)) return SDM_ERR_INVALID_ARG;
    if (!vocab_ok(V) || !rank_ok(r) || !aligned16(L) || !aligned16(U) || !aligned16(W)) return SDM_ERR_UNSUPPORTED;
    if (decode == SDM_SAMPLE && V > kMaxSampleV) return SDM_ERR_UNSUPPORTED;   // the draw's chunk table
    if (!ws || ws_bytes < ws_chain(R, B, V)) return SDM_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (decode == SDM_GREEDY && prepared) {
        // greedy by bound pruning: one scan of L, then one CTA per request walks the B steps
        if (!aligned16(prepared)) return SDM_ERR_UNSUPPORTED;
        const int n_chunks = pruned_chunks(V, dtL == SDM_FP32);
        if (B > kMaxPickSteps || n_chunks > kMaxPickChunks || static_cast<long long>(R) * B * n_chunks > (1LL << 30))
            return SDM_ERR_UNSUPPORTED;
        Carver pc{static_cast<uint8_t*>(const_cast<void*>(prepared))};
        PrunedParams pp;
        std::memset(&pp, 0, sizeof pp);
        pp.L = L;
        pp.l_fp32 = dtL == SDM_FP32;
        pp.R = R;
        pp.B = B;
        pp.V = V;
        pp.r = r;
        pp.n_chunks = n_chunks;
        pp.anchor = anchor;
        pp.U = U;
        pp.Wt = pc.take<uint16_t>(static_cast<size_t>(V) * r);
        pp.c_bound = pc.take<float>(V);
        pc.take<float>(V);           // |U[v]|
        pc.take<unsigned int>(V);    // A(v)
        pp.c_max = pc.take<float>(1);
        Carver wc{static_cast<uint8_t*>(ws)};
        const size_t segs = static_cast<size_t>(R) * B * n_chunks;
        pp.cand = wc.take<uint2>(segs * kSegCap);
        pp.cand_n = wc.take<int32_t>(segs);
        pp.cmax = wc.take<float>(segs);
        pp.tokens = tokens;
        pp.dev_status = dev_status;
        SDM_CHECK_CUDA(launch_chain_pruned(pp, s));
        return SDM_OK;
    }
    return draft_chain_dense(L, dtL, U, W, nullptr, anchor, R, B, V, r, decode, temperature, rng, tokens, logq, lse,
                             ws, dev_status, s);
}

sdm_status sdm_draft_chain_packed(const void* L, sdm_dtype dtL, const uint16_t* U, const uint16_t* W,
                                  const void* prepared, const int32_t* anchor, int R, int B, int V, int r,
                                  const int32_t* cu_seqlens, int32_t* packed_tok, int capacity, void* layout_ready,
                                  int32_t* tokens, void* ws, size_t ws_bytes, int32_t* dev_status, void* stream) {
    if (!L || !U || !W || !prepared || !anchor || !cu_seqlens || !packed_tok || !tokens || R <= 0 || B <= 0 ||
        V <= 0 || r <= 0 || capacity <= 0)
        return SDM_ERR_INVALID_ARG;
    if (dtL != SDM_BF16 && dtL != SDM_FP32) return SDM_ERR_INVALID_ARG;
    if (!vocab_ok(V) || !rank_ok(r) || !aligned16(L) || !aligned16(U) || !aligned16(W) || !aligned16(prepared))
        return SDM_ERR_UNSUPPORTED;
    const int n_chunks = pruned_chunks(V, dtL == SDM_FP32);
    if (B > kMaxPickSteps || n_chunks > kMaxPickChunks || static_cast<long long>(R) * B * n_chunks > (1LL << 30))
        return SDM_ERR_UNSUPPORTED;
    if (!ws || ws_bytes < ws_chain(R, B, V)) return SDM_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    Carver pc{static_cast<uint8_t*>(const_cast<void*>(prepared))};
    PrunedParams pp;
    std::memset(&pp, 0, sizeof pp);
    pp.L = L;
    pp.l_fp32 = dtL == SDM_FP32;
    pp.R = R;
    pp.B = B;
    pp.V = V;
    pp.r = r;
    pp.n_chunks = n_chunks;
    pp.anchor = anchor;
    pp.U = U;
    pp.Wt = pc.take<uint16_t>(static_cast<size_t>(V) * r);
    pp.c_bound = pc.take<float>(V);
    pc.take<float>(V);           // |U[v]|
    pc.take<unsigned int>(V);    // A(v)
    pp.c_max = pc.take<float>(1);
    Carver wc{static_cast<uint8_t*>(ws)};
    const size_t segs = static_cast<size_t>(R) * B * n_chunks;
    pp.cand = wc.take<uint2>(segs * kSegCap);
    pp.cand_n = wc.take<int32_t>(segs);
    pp.cmax = wc.take<float>(segs);
    pp.tokens = tokens;
    pp.dev_status = dev_status;
    pp.pack_cu = cu_seqlens;
    pp.pack_tok = packed_tok;
    pp.pack_cap = capacity;
    // the scan reads only L: it runs before the layout is ready; the pick
    // writes into the layout, so it waits for it
    SDM_CHECK_CUDA(launch_chain_scan(pp, s));
    if (layout_ready) SDM_CHECK_CUDA(cudaStreamWaitEvent(s, static_cast<cudaEvent_t>(layout_ready), 0));
    SDM_CHECK_CUDA(launch_chain_pick(pp, s));
    return SDM_OK;
}

sdm_status sdm_draft_chain_front(const void* L, sdm_dtype dtL, const uint16_t* U, const uint16_t* W,
                                 const void* prepared, const int32_t* anchor, int R, int B, int V, int r,
                                 const float* conf, const double* cost, int use_budget, const int32_t* tiers,
                                 int n_tiers, int strict, float* survival, int32_t* budget, double* expected,
                                 int32_t* total_tokens, int32_t* cu_seqlens, int32_t* packed_tok, int32_t* packed_req,
                                 int32_t* packed_pos, int capacity, int32_t* tier, int32_t* tokens, void* ws,
                                 size_t ws_bytes, int32_t* dev_status, void* stream) {
    if (!L || !U || !W || !prepared || !anchor || !conf || !cost || !survival || !budget || !expected ||
        !total_tokens || !cu_seqlens || !packed_tok || !packed_req || !packed_pos || !tier || !tokens || R <= 0 ||
        B <= 0 || V <= 0 || r <= 0 || capacity <= 0 || n_tiers < 0 || (n_tiers > 0 && !tiers))
        return SDM_ERR_INVALID_ARG;
    if (dtL != SDM_BF16 && dtL != SDM_FP32) return SDM_ERR_INVALID_ARG;
    if ((strict != 0 && strict != 1) || (use_budget != 0 && use_budget != 1)) return SDM_ERR_INVALID_ARG;
    if (!vocab_ok(V) || !rank_ok(r) || !aligned16(L) || !aligned16(U) || !aligned16(W) || !aligned16(prepared))
        return SDM_ERR_UNSUPPORTED;
    const int n_chunks = pruned_chunks(V, dtL == SDM_FP32);
    if (B > kMaxPickSteps || n_chunks > kMaxPickChunks || static_cast<long long>(R) * B * n_chunks > (1LL << 30))
        return SDM_ERR_UNSUPPORTED;
    if (static_cast<long long>(R) * B > 8192 || chain_front_smem(R, B) > kFrontSmemMax) return SDM_ERR_UNSUPPORTED;
    if (!ws || ws_bytes < ws_chain(R, B, V)) return SDM_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    Carver pc{static_cast<uint8_t*>(const_cast<void*>(prepared))};
    PrunedParams pp;
    std::memset(&pp, 0, sizeof pp);
    pp.L = L;
    pp.l_fp32 = dtL == SDM_FP32;
    pp.R = R;
    pp.B = B;
    pp.V = V;
    pp.r = r;
    pp.n_chunks = n_chunks;
    pp.anchor = anchor;
    pp.U = U;
    pp.Wt = pc.take<uint16_t>(static_cast<size_t>(V) * r);
    pp.c_bound = pc.take<float>(V);
    pc.take<float>(V);           // |U[v]|
    pc.take<unsigned int>(V);    // A(v)
    pp.c_max = pc.take<float>(1);
    Carver wc{static_cast<uint8_t*>(ws)};
    const size_t segs = static_cast<size_t>(R) * B * n_chunks;
    pp.cand = wc.take<uint2>(segs * kSegCap);
    pp.cand_n = wc.take<int32_t>(segs);
    pp.cmax = wc.take<float>(segs);
    pp.tokens = tokens;
    pp.dev_status = dev_status;
    pp.pack_cu = cu_seqlens;
    pp.pack_tok = packed_tok;
    pp.pack_cap = capacity;
    FrontParams& fr = pp.fr;
    fr.on = 1;
    fr.conf = conf;
    fr.cost = cost;
    fr.survival = survival;
    fr.budget = budget;
    fr.expected = expected;
    fr.total_tokens = total_tokens;
    int n_pad = 1;
    while (n_pad < R * B) n_pad <<= 1;
    fr.n_pad = n_pad;
    fr.use_budget = use_budget;
    fr.tiers = tiers;
    fr.n_tiers = n_tiers;
    fr.strict = strict;
    fr.cu = cu_seqlens;
    fr.ptok = packed_tok;
    fr.preq = packed_req;
    fr.ppos = packed_pos;
    fr.capacity = capacity;
    fr.tier = tier;
    // one launch lists the candidates and, in its first CTA, schedules and
    // lays out the windows; the pick (programmatic launch) waits for all of it
    SDM_CHECK_CUDA(launch_chain_scan(pp, s));
    SDM_CHECK_CUDA(launch_chain_pick(pp, s));
    return SDM_OK;
}

sdm_status sdm_draft_chain_rnn(const void* L, sdm_dtype dtL, const uint16_t* U, const uint16_t* W, const uint16_t* A,
                               const uint16_t* X, const int32_t* anchor, int R, int B, int V, int r, sdm_decode decode,
                               float temperature, sdm_rng rng, int32_t* tokens, float* logq, float* lse, float* memo,
                               void* ws, size_t ws_bytes, int32_t* dev_status, void* stream) {
    if (!L || !U || !W || !A || !X || !anchor || !tokens || R <= 0 || B <= 0 || V <= 0 || r <= 0)
        return SDM_ERR_INVALID_ARG;
    if (dtL != SDM_BF16 && dtL != SDM_FP32) return SDM_ERR_INVALID_ARG;
    if (decode != SDM_GREEDY && decode != SDM_SAMPLE) return SDM_ERR_INVALID_ARG;
    if (decode == SDM_SAMPLE && !(temperature > 0.f)) return SDM_ERR_INVALID_ARG;
    if (!vocab_ok(V) || !rank_ok(r) || !aligned16(L) || !aligned16(U) || !aligned16(W) || !aligned16(A))
        return SDM_ERR_UNSUPPORTED;
    if (decode == SDM_SAMPLE && V > kMaxSampleV) return SDM_ERR_UNSUPPORTED;
    if (!ws || ws_bytes < ws_chain_rnn(R, B, V, r)) return SDM_ERR_WORKSPACE;
    RnnStepParams rp;
    std::memset(&rp, 0, sizeof rp);
    rp.A = A;
    rp.U = U;
    rp.X = X;
    rp.memo_out = memo;
    return draft_chain_dense(L, dtL, U, W, &rp, anchor, R, B, V, r, decode, temperature, rng, tokens, logq, lse, ws,
                             dev_status, static_cast<cudaStream_t>(stream));
}

sdm_status sdm_draft_tree(const void* L, sdm_dtype dtL, const uint16_t* U, const uint16_t* W, const void* prepared,
                          const int32_t* anchor, int R, int B, int V, int r, int k, int P, int N, int32_t* tok,
                          int32_t* parent, int32_t* depth, float* score, uint32_t* mask, int32_t* n_nodes, void* ws,
                          size_t ws_bytes, int32_t* dev_status, void* stream) {
    if (!L || !U || !W || !anchor || !tok || !parent || !depth || !score || !mask || !n_nodes) return SDM_ERR_INVALID_ARG;
    if (R <= 0 || B <= 0 || V <= 0 || r <= 0 || k <= 0 || P <= 0 || N <= 0) return SDM_ERR_INVALID_ARG;
    if (dtL != SDM_BF16 && dtL != SDM_FP32) return SDM_ERR_INVALID_ARG;
    if (!vocab_ok(V) || !rank_ok(r) || !aligned16(L) || !aligned16(U) || !aligned16(W)) return SDM_ERR_UNSUPPORTED;
    if (k > kMaxTopK || k > V || P * k > 64 || kTileM % P != 0 || N > P * B) return SDM_ERR_UNSUPPORTED;
    if (static_cast<long long>(P) * B + 1 > 8192) return SDM_ERR_UNSUPPORTED;   // the pool is ranked in shared memory
    if (V > kMaxSampleV) return SDM_ERR_UNSUPPORTED;   // the per-row chunk and candidate tables of the level select
    const int fp32 = dtL == SDM_FP32;
    const int n_chunks = pruned_chunks(V, fp32);
    if (prepared) {
        if (!aligned16(prepared)) return SDM_ERR_UNSUPPORTED;
        if (n_chunks > kMaxPickChunks || static_cast<long long>(R) * B * n_chunks > (1LL << 30))
            return SDM_ERR_UNSUPPORTED;
    }
    if (!ws || ws_bytes < ws_tree(R, B, P, V)) return SDM_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t rows = static_cast<size_t>(R) * P;
    const size_t pool = static_cast<size_t>(R) * (1 + static_cast<size_t>(P) * B);
    Carver c{static_cast<uint8_t*>(ws)};
    int32_t* front_tok = c.take<int32_t>(rows);
    int32_t* front_node = c.take<int32_t>(rows);
    float* front_score = c.take<float>(rows);
    int32_t* n_front = c.take<int32_t>(R);
    int32_t* pool_tok = c.take<int32_t>(pool);
    int32_t* pool_parent = c.take<int32_t>(pool);
    int32_t* pool_depth = c.take<int32_t>(pool);
    float* pool_score = c.take<float>(pool);
    int32_t* pool_n = c.take<int32_t>(R);

    // the bound-pruned level's GEMM takes two 128-row sub-tiles per CTA when
    // there are more than 128 frontier rows (every W tile feeds 256 rows)
    const int m_sub = (prepared && rows > static_cast<size_t>(kTileM)) ? 2 : 1;
    const int l_rows = std::min(kTileM * m_sub / P, R);
    CUtensorMap tmW, tmL;
    if (!map_w(&tmW, W, r, V) || !map_l(&tmL, L, fp32, R, B, V, l_rows)) return SDM_ERR_CUDA;
    const int n_tiles = (V + kTileN - 1) / kTileN;
    const int gy = static_cast<int>((rows + kTileM * m_sub - 1) / (kTileM * m_sub));
    const int gx = gemm_grid_x(n_tiles, gy);

    GemmParams p;
    std::memset(&p, 0, sizeof p);
    p.m_sub = m_sub;
    p.rows = static_cast<int>(rows);
    p.R = R;
    p.B = B;
    p.V = V;
    p.r = r;
    p.n_tiles = n_tiles;
    p.l_fp32 = fp32;
    p.l_rows = l_rows;
    p.P = P;
    p.k = k;
    p.inv_t = 1.0f;
    p.U = U;
    p.anchor = anchor;
    p.front_tok = front_tok;
    p.dev_status = dev_status;
    SDM_CHECK_CUDA(launch_tree_init(anchor, R, P, B, front_tok, front_node, front_score, n_front, pool_tok, pool_parent,
                                    pool_depth, pool_score, pool_n, dev_status, s));
    if (prepared) {
        // every (request, level) row of L listed once for the top k; per level
        // the GEMM's log-sum-exp partials, then one CTA per request ranks the
        // listed ids exactly and prunes
        Carver pc{static_cast<uint8_t*>(const_cast<void*>(prepared))};
        const uint16_t* Wt = pc.take<uint16_t>(static_cast<size_t>(V) * r);
        const float* c_bound = pc.take<float>(V);
        pc.take<float>(V);           // |U[v]|
        pc.take<unsigned int>(V);    // A(v)
        const float* c_max = pc.take<float>(1);
        PrunedParams pp;
        std::memset(&pp, 0, sizeof pp);
        pp.L = L;
        pp.l_fp32 = fp32;
        pp.R = R;
        pp.B = B;
        pp.V = V;
        pp.r = r;
        pp.n_chunks = n_chunks;
        pp.anchor = anchor;
        pp.U = U;
        pp.Wt = Wt;
        pp.c_bound = c_bound;
        pp.c_max = c_max;
        const size_t segs = static_cast<size_t>(R) * B * pruned_chunks(V, 1);   // carved as ws_chain_pruned sizes it
        pp.cand = c.take<uint2>(segs * kSegCap);
        pp.cand_n = c.take<int32_t>(segs);
        pp.cmax = c.take<float>(segs);
        pp.dev_status = dev_status;
        pp.kth = k;
        const int n_part = gx;   // one partial per frontier row and GEMM CTA
        auto* part = c.take<float2>(rows * n_part);
        TreeRowsParams rp;
        std::memset(&rp, 0, sizeof rp);
        rp.cand = pp.cand;
        rp.cand_n = pp.cand_n;
        rp.n_chunks = n_chunks;
        rp.rows = R * B;
        rp.V = V;
        rp.k = k;
        rp.c_max = c_max;
        rp.keep = c.take<uint2>(static_cast<size_t>(R) * B * kTreeKeep);
        rp.n_keep = c.take<int32_t>(static_cast<size_t>(R) * B);
        rp.lk = c.take<float>(static_cast<size_t>(R) * B);
        rp.cmax = pp.cmax;
        rp.lmax = c.take<float>(static_cast<size_t>(R) * B);
        SDM_CHECK_CUDA(launch_chain_scan(pp, s));
        SDM_CHECK_CUDA(launch_tree_rows(rp, s));
        p.part = part;
        p.n_part = n_part;
        p.row_lmax = rp.lmax;
        p.c_bound = c_bound;
        gemm_pick_stages(p, MODE_TREE_LSE);
        TreeLevelParams tl;
        std::memset(&tl, 0, sizeof tl);
        tl.keep = rp.keep;
        tl.n_keep = rp.n_keep;
        tl.lk = rp.lk;
        tl.L = L;
        tl.l_fp32 = fp32;
        tl.U = U;
        tl.Wt = Wt;
        tl.c_bound = c_bound;
        tl.R = R;
        tl.B = B;
        tl.V = V;
        tl.r = r;
        tl.P = P;
        tl.k = k;
        tl.part = part;
        tl.n_part = n_part;
        tl.front_tok = front_tok;
        tl.front_node = front_node;
        tl.front_score = front_score;
        tl.n_front = n_front;
        tl.pool_tok = pool_tok;
        tl.pool_parent = pool_parent;
        tl.pool_depth = pool_depth;
        tl.pool_score = pool_score;
        tl.pool_n = pool_n;
        tl.dev_status = dev_status;
        for (int d = 1; d <= B; ++d) {
            p.d = d;
            tl.d = d;
            SDM_CHECK_CUDA(launch_markov_gemm(MODE_TREE_LSE, tmW, tmL, p, gx, gy, s));
            SDM_CHECK_CUDA(launch_tree_level(tl, s));
        }
    } else {
        const int nb = n_blocks16(V);
        auto* blk = c.take<float2>(rows * nb);
        auto* row_top = c.take<float2>(rows * kMaxTopK);
        float* row_lse = c.take<float>(rows);
        p.blk = blk;
        p.nb = nb;
        gemm_pick_stages(p, MODE_TREE);
        TreeSelectParams tp;
        std::memset(&tp, 0, sizeof tp);
        tp.blk = blk;
        tp.nb = nb;
        tp.rows = static_cast<int>(rows);
        tp.P = P;
        tp.B = B;
        tp.V = V;
        tp.r = r;
        tp.k = k;
        tp.front_tok = front_tok;
        tp.L = L;
        tp.l_fp32 = fp32;
        tp.U = U;
        tp.W = W;
        tp.row_top = row_top;
        tp.row_lse = row_lse;
        tp.dev_status = dev_status;
        for (int d = 1; d <= B; ++d) {
            p.d = d;
            tp.d = d;
            SDM_CHECK_CUDA(launch_markov_gemm(MODE_TREE, tmW, tmL, p, gx, gy, s));
            SDM_CHECK_CUDA(launch_tree_select(tp, s));
            SDM_CHECK_CUDA(launch_tree_merge(row_top, row_lse, R, P, k, B, d, front_tok, front_node, front_score,
                                             n_front, pool_tok, pool_parent, pool_depth, pool_score, pool_n, s));
        }
    }
    SDM_CHECK_CUDA(launch_tree_finalize(R, P, B, N, pool_tok, pool_parent, pool_depth, pool_score, pool_n, tok, parent,
                                        depth, score, mask, n_nodes, s));
    return SDM_OK;
}

sdm_status sdm_check_timeout_path(const void* L, sdm_dtype dtL, const uint16_t* U, const uint16_t* W,
                                  const int32_t* anchor, int R, int B, int V, int r, unsigned long long wait_ns,
                                  void* ws, size_t ws_bytes, int32_t* dev_status, void* stream) {
    if (!L || !U || !W || !anchor || !dev_status || R <= 0 || B <= 0 || V <= 0 || r <= 0) return SDM_ERR_INVALID_ARG;
    if (dtL != SDM_BF16 && dtL != SDM_FP32) return SDM_ERR_INVALID_ARG;
    if (wait_ns < 1000ull || wait_ns > 1000000000ull) return SDM_ERR_INVALID_ARG;
    if (!vocab_ok(V) || !rank_ok(r) || !aligned16(L) || !aligned16(U) || !aligned16(W)) return SDM_ERR_UNSUPPORTED;
    if (!ws || ws_bytes < ws_chain_dense(R, B, V)) return SDM_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int fp32 = dtL == SDM_FP32;
    const int l_rows = std::min(R, kTileM);
    CUtensorMap tmW, tmL;
    if (!map_w(&tmW, W, r, V) || !map_l(&tmL, L, fp32, R, B, V, l_rows)) return SDM_ERR_CUDA;
    const int n_tiles = (V + kTileN - 1) / kTileN;
    const int gy = (R + kTileM - 1) / kTileM;
    const int gx = gemm_grid_x(n_tiles, gy);
    auto* keys = static_cast<unsigned long long*>(ws);
    GemmParams p;
    std::memset(&p, 0, sizeof p);
    p.rows = R;
    p.R = R;
    p.B = B;
    p.V = V;
    p.r = r;
    p.n_tiles = n_tiles;
    p.l_fp32 = fp32;
    p.l_rows = l_rows;
    p.P = 1;
    p.k = 1;
    p.d = 1;
    p.inv_t = 1.0f;
    gemm_pick_stages(p, MODE_CHAIN_GREEDY);
    p.U = U;
    p.anchor = anchor;
    p.keys = keys;
    p.dev_status = dev_status;
    p.wait_ns = wait_ns;
    p.withhold_loads = 1;   // nothing is loaded: every pipeline wait runs out
    SDM_CHECK_CUDA(launch_fill_u64(keys, static_cast<size_t>(B) * R, 0ull, s));
    SDM_CHECK_CUDA(launch_markov_gemm(MODE_CHAIN_GREEDY, tmW, tmL, p, gx, gy, s));
    return SDM_OK;
}

sdm_status sdm_schedule_budget(const float* conf, int R, int gamma, const double* cost, float* survival,
                               int32_t* budget, double* expected, int32_t* total_tokens, void* ws, size_t ws_bytes,
                               int32_t* dev_status, void* stream) {
    (void)ws;
    (void)ws_bytes;
    if (!conf || !cost || !survival || !budget || !expected || !total_tokens || R <= 0 || gamma <= 0)
        return SDM_ERR_INVALID_ARG;
    if (static_cast<long long>(R) * gamma > 8192) return SDM_ERR_UNSUPPORTED;
    SDM_CHECK_CUDA(launch_schedule(conf, R, gamma, cost, survival, budget, expected, total_tokens, nullptr, dev_status,
                                   static_cast<cudaStream_t>(stream)));
    return SDM_OK;
}

sdm_status sdm_schedule_dynamic(const float* conf, const float* conf_stale, int R, int gamma, const double* cost,
                                float* survival, int32_t* budget, double* expected, int32_t* total_tokens,
                                int32_t* capacity, int32_t* dev_status, void* stream) {
    (void)dev_status;
    if (!conf || !conf_stale || !cost || !survival || !budget || !expected || !total_tokens || !capacity || R <= 0 ||
        gamma <= 0)
        return SDM_ERR_INVALID_ARG;
    if (static_cast<long long>(R) * gamma > 8192) return SDM_ERR_UNSUPPORTED;
    SDM_CHECK_CUDA(launch_schedule_dynamic(conf, conf_stale, R, gamma, cost, survival, budget, expected, total_tokens,
                                           capacity, static_cast<cudaStream_t>(stream)));
    return SDM_OK;
}

sdm_status sdm_schedule_threshold(const float* conf, int R, int gamma, float tau, int32_t* budget,
                                  int32_t* total_tokens, int32_t* dev_status, void* stream) {
    (void)dev_status;
    if (!conf || !budget || !total_tokens || R <= 0 || gamma <= 0) return SDM_ERR_INVALID_ARG;
    if (static_cast<long long>(R) * gamma > (1LL << 30)) return SDM_ERR_UNSUPPORTED;
    SDM_CHECK_CUDA(launch_schedule_threshold(conf, R, gamma, tau, budget, total_tokens,
                                             static_cast<cudaStream_t>(stream)));
    return SDM_OK;
}

sdm_status sdm_threshold_sweep(const float* conf, const int32_t* ceiling, int R, int gamma, const float* taus, int K,
                               int32_t* drafts, int32_t* accepted, double* expected, int32_t* dev_status,
                               void* stream) {
    (void)dev_status;
    if (!conf || !taus || !drafts || !accepted || !expected || R <= 0 || gamma <= 0 || K <= 0)
        return SDM_ERR_INVALID_ARG;
    // the exact expected-count sum holds R gamma terms of at most 2^48 units
    if (static_cast<long long>(R) * gamma > 32768 || K > 65535) return SDM_ERR_UNSUPPORTED;
    SDM_CHECK_CUDA(launch_threshold_sweep(conf, ceiling, R, gamma, taus, K, drafts, accepted, expected,
                                          static_cast<cudaStream_t>(stream)));
    return SDM_OK;
}

sdm_status sdm_pack_ragged(const int32_t* anchor, const int32_t* draft, const int32_t* budget, int R, int gamma,
                           const int32_t* tiers, int n_tiers, int strict, int32_t* cu_seqlens, int32_t* packed_tok,
                           int32_t* packed_req, int32_t* packed_pos, int capacity, int32_t* tier, int32_t* tier_host,
                           int32_t* dev_status, void* stream) {
    if (!anchor || !cu_seqlens || !packed_tok || !packed_req || !packed_pos || !tier) return SDM_ERR_INVALID_ARG;
    if (R <= 0 || gamma < 0 || n_tiers < 0 || capacity <= 0 || (n_tiers > 0 && !tiers)) return SDM_ERR_INVALID_ARG;
    if (strict != 0 && strict != 1) return SDM_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    SDM_CHECK_CUDA(launch_pack(anchor, draft, budget, R, gamma, tiers, n_tiers, strict, cu_seqlens, packed_tok,
                               packed_req, packed_pos, capacity, tier, dev_status, s));
    if (tier_host) SDM_CHECK_CUDA(cudaMemcpyAsync(tier_host, tier, sizeof(int32_t), cudaMemcpyDeviceToHost, s));
    return SDM_OK;
}

sdm_status sdm_verify(sdm_vmode mode, sdm_decode decode, float temperature, sdm_rng rng, const void* target,
                      sdm_dtype dtT, int row_capacity, const int32_t* cu_seqlens, const int32_t* anchor,
                      const int32_t* draft, const int32_t* budget, const float* logq, const float* lse_q,
                      const void* L, sdm_dtype dtL, const uint16_t* U, const uint16_t* W, int r, int R, int gamma,
                      int V, int32_t* accept, int32_t* ceiling, int32_t* out_tok, int32_t* n_out, void* ws,
                      size_t ws_bytes, int32_t* dev_status, void* stream) {
    if (!target || !cu_seqlens || !anchor || !draft || !accept || !out_tok || !n_out) return SDM_ERR_INVALID_ARG;
    if (R <= 0 || gamma <= 0 || V <= 0 || row_capacity <= 0) return SDM_ERR_INVALID_ARG;
    if (mode != SDM_STATIC && mode != SDM_COMPACT && mode != SDM_CAP_ACCEPT) return SDM_ERR_INVALID_ARG;
    if (decode != SDM_GREEDY && decode != SDM_SAMPLE) return SDM_ERR_INVALID_ARG;
    if (dtT != SDM_BF16 && dtT != SDM_FP32) return SDM_ERR_INVALID_ARG;
    if (mode == SDM_CAP_ACCEPT && !budget) return SDM_ERR_INVALID_ARG;
    if (!vocab_ok(V) || !aligned16(target)) return SDM_ERR_UNSUPPORTED;
    if (decode == SDM_SAMPLE) {
        if (!logq || !lse_q || !L || !U || !W || !(temperature > 0.f)) return SDM_ERR_INVALID_ARG;
        if (dtL != SDM_BF16 && dtL != SDM_FP32) return SDM_ERR_INVALID_ARG;
        if (!rank_ok(r) || !aligned16(L) || !aligned16(U) || !aligned16(W)) return SDM_ERR_UNSUPPORTED;
        if (V > kMaxSampleV) return SDM_ERR_UNSUPPORTED;
    }
    if (!ws || ws_bytes < ws_verify(R, row_capacity, V)) return SDM_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int t_fp32 = dtT == SDM_FP32;
    const int nchunk_max = std::max(n_chunks_of(V, 0), n_chunks_of(V, 1));
    Carver c{static_cast<uint8_t*>(ws)};
    auto* row_keys = c.take<unsigned long long>(static_cast<size_t>(row_capacity) * nchunk_max);
    auto* lse_part = c.take<float2>(static_cast<size_t>(row_capacity) * nchunk_max);
    int32_t* res_tok = c.take<int32_t>(R);
    int32_t* res_pos = c.take<int32_t>(R);
    int32_t* res_trow = c.take<int32_t>(R);
    float* res_lse_p = c.take<float>(R);
    int32_t* bonus_row = c.take<int32_t>(R);
    int32_t* bonus_pos = c.take<int32_t>(R);
    const int nb = n_blocks16(V);
    auto* blk = c.take<float2>(static_cast<size_t>(R) * nb);

    StreamParams sp;
    std::memset(&sp, 0, sizeof sp);
    sp.base = target;
    sp.fp32 = t_fp32;
    sp.V = V;
    sp.chunk = t_fp32 ? kChunkFp32 : kChunkBf16;
    sp.n_chunks = n_chunks_of(V, t_fp32);
    sp.count = cu_seqlens + R;
    sp.n_items = row_capacity;
    sp.inv_t = decode == SDM_SAMPLE ? 1.0f / temperature : 1.0f;

    if (decode == SDM_GREEDY) {
        sp.keys = row_keys;
        SDM_CHECK_CUDA(launch_stream(STREAM_ARGMAX, sp, row_capacity, s));
        SDM_CHECK_CUDA(launch_verify_greedy_finalize(mode, cu_seqlens, draft, budget, row_keys, sp.n_chunks, R, gamma,
                                                     V, row_capacity, accept, ceiling, out_tok, n_out, dev_status, s));
        return SDM_OK;
    }
    // rejection sampling
    const uint32_t k0 = static_cast<uint32_t>(rng.seed), k1 = static_cast<uint32_t>(rng.seed >> 32);
    const uint32_t cyc = static_cast<uint32_t>(rng.cycle);
    sp.part = lse_part;
    SDM_CHECK_CUDA(launch_stream(STREAM_LSE, sp, row_capacity, s));
    SDM_CHECK_CUDA(launch_verify_sample_scan(mode, cu_seqlens, anchor, draft, budget, logq, target, t_fp32, V, lse_part,
                                             sp.n_chunks, sp.inv_t, k0, k1, cyc, R, gamma, accept, ceiling, res_tok,
                                             res_pos, res_trow, res_lse_p, bonus_row, bonus_pos, row_capacity,
                                             dev_status, s));
    // residual rows: recompute q with the Markov head; records of max(0, p - q)
    CUtensorMap tmW;
    if (!map_w(&tmW, W, r, V)) return SDM_ERR_CUDA;
    const int n_tiles = (V + kTileN - 1) / kTileN;
    const int gy = (R + kTileM - 1) / kTileM;
    const int gx = gemm_grid_x(n_tiles, gy);
    GemmParams p;
    std::memset(&p, 0, sizeof p);
    p.rows = R;
    p.R = R;
    p.B = gamma;
    p.V = V;
    p.r = r;
    p.n_tiles = n_tiles;
    p.l_fp32 = dtL == SDM_FP32;
    p.l_rows = 1;
    p.P = 1;
    p.k = 1;
    p.d = 1;
    gemm_pick_stages(p, MODE_RESID);
    p.inv_t = sp.inv_t;
    p.U = U;
    p.res_tok = res_tok;
    p.res_pos = res_pos;
    p.res_trow = res_trow;
    p.res_lse_p = res_lse_p;
    p.lse_q = lse_q;
    p.L = L;
    p.target = target;
    p.t_fp32 = t_fp32;
    p.gamma = gamma;
    p.blk = blk;
    p.nb = nb;
    p.dev_status = dev_status;
    SDM_CHECK_CUDA(launch_markov_gemm(MODE_RESID, tmW, tmW, p, gx, gy, s));
    // the residual or bonus draw of every request, then the committed tokens
    ResampleParams rp;
    std::memset(&rp, 0, sizeof rp);
    rp.blk = blk;
    rp.nb = nb;
    rp.res_tok = res_tok;
    rp.res_pos = res_pos;
    rp.res_trow = res_trow;
    rp.res_lse_p = res_lse_p;
    rp.lse_q = lse_q;
    rp.L = L;
    rp.l_fp32 = p.l_fp32;
    rp.U = U;
    rp.W = W;
    rp.r = r;
    rp.bonus_row = bonus_row;
    rp.bonus_pos = bonus_pos;
    rp.lse_part = lse_part;
    rp.n_chunks = sp.n_chunks;
    rp.chunk = sp.chunk;
    rp.target = target;
    rp.t_fp32 = t_fp32;
    rp.R = R;
    rp.gamma = gamma;
    rp.V = V;
    rp.inv_t = sp.inv_t;
    rp.k0 = k0;
    rp.k1 = k1;
    rp.cycle = cyc;
    rp.draft = draft;
    rp.accept = accept;
    rp.out_tok = out_tok;
    rp.n_out = n_out;
    rp.dev_status = dev_status;
    SDM_CHECK_CUDA(launch_resample(rp, s));
    return SDM_OK;
}

sdm_status sdm_verify_tree(const void* target, sdm_dtype dtT, const int32_t* tok, const int32_t* parent,
                           const int32_t* n_nodes, int R, int N, int B, int V, int32_t* accept, int32_t* out_tok,
                           int32_t* n_out, void* ws, size_t ws_bytes, int32_t* dev_status, void* stream) {
    if (!target || !tok || !parent || !n_nodes || !accept || !out_tok || !n_out) return SDM_ERR_INVALID_ARG;
    if (R <= 0 || N < 0 || B <= 0 || V <= 0) return SDM_ERR_INVALID_ARG;
    if (N >= 16384) return SDM_ERR_UNSUPPORTED;   // the tree is walked in shared memory
    if (dtT != SDM_BF16 && dtT != SDM_FP32) return SDM_ERR_INVALID_ARG;
    if (!vocab_ok(V) || !aligned16(target)) return SDM_ERR_UNSUPPORTED;
    const size_t rows = static_cast<size_t>(R) * (N + 1);
    const int nck = n_chunks_of(V, dtT == SDM_FP32);
    if (!ws || ws_bytes < align256(rows * 8 * nck)) return SDM_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    auto* row_keys = static_cast<unsigned long long*>(ws);
    StreamParams sp;
    std::memset(&sp, 0, sizeof sp);
    sp.base = target;
    sp.fp32 = dtT == SDM_FP32;
    sp.V = V;
    sp.chunk = sp.fp32 ? kChunkFp32 : kChunkBf16;
    sp.n_chunks = n_chunks_of(V, sp.fp32);
    sp.n_items = static_cast<int>(rows);
    sp.keys = row_keys;
    sp.inv_t = 1.0f;
    SDM_CHECK_CUDA(launch_stream(STREAM_ARGMAX, sp, static_cast<int>(rows), s));
    SDM_CHECK_CUDA(launch_tree_verify_walk(row_keys, sp.n_chunks, tok, parent, n_nodes, R, N, B, V, accept, out_tok, n_out,
                                           dev_status, s));
    return SDM_OK;
}

sdm_status sdm_tv_label(float temperature, const void* target, sdm_dtype dtT, int row_capacity,
                        const int32_t* cu_seqlens, const int32_t* anchor, const int32_t* draft, const float* lse_q,
                        const void* L, sdm_dtype dtL, const uint16_t* U, const uint16_t* W, int r, int R, int gamma,
                        int V, float* label, void* ws, size_t ws_bytes, int32_t* dev_status, void* stream) {
    if (!target || !cu_seqlens || !anchor || !draft || !L || !U || !W || !label) return SDM_ERR_INVALID_ARG;
    if (R <= 0 || gamma <= 0 || V <= 0 || row_capacity <= 0 || !(temperature > 0.f)) return SDM_ERR_INVALID_ARG;
    if ((dtT != SDM_BF16 && dtT != SDM_FP32) || (dtL != SDM_BF16 && dtL != SDM_FP32)) return SDM_ERR_INVALID_ARG;
    if (!vocab_ok(V) || !rank_ok(r) || !aligned16(target) || !aligned16(L) || !aligned16(U) || !aligned16(W))
        return SDM_ERR_UNSUPPORTED;
    if (static_cast<long long>(R) * gamma > (1 << 22)) return SDM_ERR_UNSUPPORTED;
    if (!ws || ws_bytes < ws_tv_label(R, gamma, V, row_capacity)) return SDM_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int slots = R * gamma;
    const int nchunk_max = std::max(n_chunks_of(V, 0), n_chunks_of(V, 1));
    const int n_part = label_n_part(R, gamma, V);
    Carver c{static_cast<uint8_t*>(ws)};
    auto* lse_part = c.take<float2>(static_cast<size_t>(row_capacity) * nchunk_max);
    int32_t* res_req = c.take<int32_t>(slots);
    int32_t* res_pos = c.take<int32_t>(slots);
    int32_t* res_tok = c.take<int32_t>(slots);
    int32_t* res_trow = c.take<int32_t>(slots);
    float* res_lse_p = c.take<float>(slots);
    float* row_lse_q = c.take<float>(slots);
    auto* part = c.take<float2>(static_cast<size_t>(slots) * n_part);

    // log-sum-exp of every packed target row over T, in streaming partials
    StreamParams sp;
    std::memset(&sp, 0, sizeof sp);
    sp.base = target;
    sp.fp32 = dtT == SDM_FP32;
    sp.V = V;
    sp.chunk = sp.fp32 ? kChunkFp32 : kChunkBf16;
    sp.n_chunks = n_chunks_of(V, sp.fp32);
    sp.count = cu_seqlens + R;
    sp.n_items = row_capacity;
    sp.inv_t = 1.0f / temperature;
    sp.part = lse_part;
    SDM_CHECK_CUDA(launch_stream(STREAM_LSE, sp, row_capacity, s));
    // every GEMM row unused until the row list names it
    SDM_CHECK_CUDA(cudaMemsetAsync(res_tok, 0xFF, static_cast<size_t>(slots) * sizeof(int32_t), s));
    SDM_CHECK_CUDA(launch_label_prep(cu_seqlens, anchor, draft, lse_q, lse_part, sp.n_chunks, R, gamma, V,
                                     row_capacity, res_req, res_pos, res_tok, res_trow, res_lse_p, row_lse_q, label,
                                     dev_status, s));
    CUtensorMap tmW;
    if (!map_w(&tmW, W, r, V)) return SDM_ERR_CUDA;
    const int n_tiles = (V + kTileN - 1) / kTileN;
    const int gy = (slots + kTileM - 1) / kTileM;
    const int gx = gemm_grid_x(n_tiles, gy);
    GemmParams p;
    std::memset(&p, 0, sizeof p);
    p.rows = slots;
    p.R = R;
    p.B = gamma;
    p.V = V;
    p.r = r;
    p.n_tiles = n_tiles;
    p.l_fp32 = dtL == SDM_FP32;
    p.l_rows = 1;
    p.P = 1;
    p.k = 1;
    p.d = 1;
    p.inv_t = sp.inv_t;
    p.U = U;
    p.res_req = res_req;
    p.res_tok = res_tok;
    p.res_pos = res_pos;
    p.res_trow = res_trow;
    p.res_lse_p = res_lse_p;
    p.row_lse_q = row_lse_q;
    p.L = L;
    p.target = target;
    p.t_fp32 = sp.fp32;
    p.gamma = gamma;
    p.part = part;
    p.n_part = n_part;
    p.dev_status = dev_status;
    if (!lse_q) {   // the draft's log-sum-exp, from one more pass over L
        gemm_pick_stages(p, MODE_QLSE);
        SDM_CHECK_CUDA(launch_markov_gemm(MODE_QLSE, tmW, tmW, p, gx, gy, s));
        SDM_CHECK_CUDA(launch_label_lse_q(part, n_part, slots, res_tok, row_lse_q, s));
    }
    const int tv_mode = p.l_fp32 ? MODE_TVMIN : (p.t_fp32 ? MODE_TVMIN_B32 : MODE_TVMIN_B16);
    gemm_pick_stages(p, tv_mode);
    SDM_CHECK_CUDA(launch_markov_gemm(tv_mode, tmW, tmW, p, gx, gy, s));
    SDM_CHECK_CUDA(launch_label_finalize(part, n_part, slots, res_tok, res_req, res_pos, gamma, label, s));
    return SDM_OK;
}

sdm_status sdm_observe(const float* conf, const int32_t* cu_seqlens, const int32_t* ceiling, const int32_t* cls, int R,
                       int gamma, int n_class, int n_bins, int32_t* hist, int32_t* reached, int32_t* hits,
                       int32_t* bin_n, int32_t* bin_hit, double* bin_conf, double* ece, int32_t* dev_status,
                       void* stream) {
    if (!conf || !cu_seqlens || !ceiling || !cls || !hist || !reached || !hits || !bin_n || !bin_hit || !bin_conf ||
        !ece)
        return SDM_ERR_INVALID_ARG;
    if (R <= 0 || gamma <= 0 || n_class <= 0 || n_bins <= 0) return SDM_ERR_INVALID_ARG;
    if (n_class > 4096 || n_bins > 4096 || gamma > 4096 || observe_smem_bytes(gamma, n_class, n_bins) > 49152 ||
        static_cast<long long>(R) * gamma > (1LL << 30))
        return SDM_ERR_UNSUPPORTED;
    SDM_CHECK_CUDA(launch_observe(conf, cu_seqlens, ceiling, cls, R, gamma, n_class, n_bins, hist, reached, hits,
                                  bin_n, bin_hit, bin_conf, ece, dev_status, static_cast<cudaStream_t>(stream)));
    return SDM_OK;
}

}  // extern "C"
