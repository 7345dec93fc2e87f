// internal.h - launch parameters and launcher declarations shared by the
// kernel translation units and the C-ABI layer (api.cu).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/sdm.h"

namespace sdm {

// Launch with programmatic stream serialization: the kernel may be scheduled
// while its predecessor in the stream drains, and waits for it in pdl_wait().
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// ---------------------------------------------------------------------------
// Markov GEMM (tcgen05): one CTA = one 128-row M tile x a round-robin set of
// 128-wide vocab tiles; K = r (<= 256, multiple of 64).
// ---------------------------------------------------------------------------
constexpr int kTileM = 128;        // GEMM rows per CTA (TMEM lanes)
constexpr int kTileN = 128;        // vocab ids per tile = N of one tcgen05.mma
constexpr int kBoxN = 64;          // vocab ids per TMA box (one 128-byte bf16 swizzle span)
constexpr int kColGroups = 4;      // epilogue column groups per box (16 columns each)
constexpr int kEpiCols = kBoxN / kColGroups;
constexpr int kEpiWarps = 4 * kColGroups;          // four TMEM sub-partitions x column groups
constexpr int kGemmThreads = 96 + 32 * kEpiWarps;  // warp 0 W loads, warp 1 MMA, warp 2 L loads, warps 3.. epilogue
constexpr int kMaxTopK = 8;

enum GemmMode {
    MODE_CHAIN_GREEDY = 0,
    MODE_CHAIN_SAMPLE = 1,
    MODE_TREE = 2,
    MODE_RESID = 3,
    MODE_ABSMAX = 4,
    MODE_QLSE = 5,    // soft label pass 1: log-sum-exp of the draft logits of listed rows
    MODE_TVMIN = 6,   // soft label pass 2: sum_v min(q_v, p_v) of listed rows
    MODE_TVMIN_B16 = 7,   // the same for bf16 L and bf16 target rows, loads a tile ahead of use
    MODE_TVMIN_B32 = 8,   // the same for bf16 L and fp32 target rows
    MODE_TREE_LSE = 9     // PCTree level, log-sum-exp only: one (max, sum) partial per frontier row, CTA and group
};

// Modes that stage a tile of L beside each W tile (the others read their L
// rows, if any, straight from global memory).
__host__ __device__ constexpr bool mode_reads_l(int mode) {
    return mode == MODE_CHAIN_GREEDY || mode == MODE_CHAIN_SAMPLE || mode == MODE_TREE || mode == MODE_TREE_LSE;
}
// PCTree modes: GEMM row = (request, frontier slot), L row = the request's.
__host__ __device__ constexpr bool mode_tree(int mode) { return mode == MODE_TREE || mode == MODE_TREE_LSE; }
// Modes whose GEMM rows come from an explicit row list (res_tok / res_req).
__host__ __device__ constexpr bool mode_row_list(int mode) {
    return mode == MODE_QLSE || mode == MODE_TVMIN || mode == MODE_TVMIN_B16 || mode == MODE_TVMIN_B32;
}
// Modes whose epilogue issues a whole tile's global loads before reading the
// accumulator, one slice at a time.
__host__ __device__ constexpr bool mode_loads_first(int mode) {
    return mode == MODE_QLSE || mode == MODE_TVMIN_B16 || mode == MODE_TVMIN_B32;
}

struct GemmParams {
    int rows;            // GEMM rows in use
    int R, B, V, r;
    int n_tiles;         // ceil(V / 64)
    int w_stages;        // W ring depth (64 K rows x 128 ids per stage)
    int l_stages;        // L ring depth (one 64-id box per stage)
    int l_fp32;          // L element type: 0 bf16, 1 fp32
    int l_rows;          // L rows per M tile in the TMA box (chain: min(R,128); tree: 128/P)
    int P;               // tree: GEMM rows per request (frontier slots)
    int k;               // tree: local top-k
    int d;               // 1-based draft position / tree level
    float inv_t;         // 1 / temperature
    const uint16_t* U;   // [V, r]
    const uint16_t* a_rows;     // chain modes: [R, r] bf16 A row of GEMM row m in place of U[tok(m)] (RNN memo), or NULL
    const int32_t* anchor;
    // chain
    unsigned long long* keys;   // greedy: [B][R] argmax keys
    const int32_t* tok_in;      // sample: [R, B] tokens drawn so far (step d reads column d - 2)
    // sampling and residual: one (m, s) record per GEMM row and 16-column block
    float2* blk;                // [rows][nb]
    int nb;                     // ceil(V / 16)
    // tree
    const int32_t* front_tok;   // [R][P] frontier tokens (-1: empty slot)
    // residual (sample verify): one GEMM row per request
    const int32_t* res_tok;     // [R] previous token of the rejected position, -1: none
    const int32_t* res_pos;     // [R] rejected window position j (L row j, stream row j)
    const int32_t* res_trow;    // [R] packed target row of position j
    const float* res_lse_p;     // [R] log-sum-exp of target row j / T
    const float* lse_q;         // [R, gamma] draft log-sum-exp
    const void* L;              // [R, gamma, V] (residual reads rows directly)
    const void* target;         // packed target rows
    int t_fp32;                 // target element type
    int gamma;
    // soft label (row list): GEMM row g = window row res_pos[g] of request
    // res_req[g] (previous token res_tok[g], -1: unused row; target row
    // res_trow[g], target log-sum-exp res_lse_p[g], draft log-sum-exp
    // row_lse_q[g]); one partial per row, CTA and column group in part
    const int32_t* res_req;
    const float* row_lse_q;
    float2* part;               // [rows][n_part]
    int n_part;                 // gridDim.x * kColGroups (MODE_TREE_LSE: gridDim.x, the groups merged)
    // absmax (prepared tables): GEMM row m = token m
    unsigned int* absmax_bits;      // [rows] max_v |U[m] . W[:, v]| as fp32 bits (atomic max)
    int32_t* dev_status;
    // wind-down check: a limit on every pipeline wait (0: the default), and
    // withheld loads (the producers arm nothing, so every wait runs out)
    unsigned long long wait_ns;
    int withhold_loads;
    // 128-row sub-tiles per CTA: 1, or 2 for PCTree levels (MODE_TREE_LSE)
    // of more than 128 frontier rows (every W tile then feeds 256 rows)
    int m_sub;
    // MODE_TREE_LSE with prepared tables: the bound max_v L_v + c(y) >= z
    // serves as the exponent reference (row_lmax [R * B], c_bound [V]), or NULL
    const float* row_lmax;
    const float* c_bound;
};

// Ring depths for the launch shape (written into p.w_stages / p.l_stages).
void gemm_pick_stages(GemmParams& p, int mode);
cudaError_t launch_markov_gemm(int mode, const CUtensorMap& tmW, const CUtensorMap& tmL, const GemmParams& p,
                               int grid_x, int grid_y, cudaStream_t s);

// ---------------------------------------------------------------------------
// Vocab-row streaming kernels (argmax / log-sum-exp partials over target rows)
// ---------------------------------------------------------------------------
constexpr int kChunkBf16 = 16384;     // ids per streaming work item (32 KB of bf16)
constexpr int kChunkFp32 = 8192;      // (32 KB of fp32)
// Streaming work items (and partials) per row of V elements.
inline int n_chunks_of(int V, int fp32) {
    const int c = fp32 ? kChunkFp32 : kChunkBf16;
    return (V + c - 1) / c;
}

enum StreamOp { STREAM_ARGMAX = 0, STREAM_LSE = 1 };

struct StreamParams {
    const void* base;       // row r starts at base + r * V elements
    int fp32;               // element type
    int V;
    int chunk;              // elements per work item (multiple of 8)
    int n_chunks;           // chunks per row
    int n_items;            // rows (items) when count == NULL, else the rows the buffer holds
    const int32_t* count;   // device item count (e.g. cu_seqlens + R), clamped to n_items; may be NULL
    const int32_t* row_of;  // item -> row index (NULL: identity; < 0: skip)
    float inv_t;
    unsigned long long* keys;   // ARGMAX: [n_items][n_chunks] partial keys
    float2* part;               // LSE: [n_items][n_chunks] (max, sum of exp(x - max)) of x = row / T
};

cudaError_t launch_stream(int op, const StreamParams& p, int max_items, cudaStream_t s);

// ---------------------------------------------------------------------------
// small kernels
// ---------------------------------------------------------------------------
cudaError_t launch_fill_u64(unsigned long long* p, size_t n, unsigned long long v, cudaStream_t s);

// greedy chain: tokens from the argmax keys [B][R]
cudaError_t launch_chain_finalize(const unsigned long long* keys, int R, int B, int V, int32_t* tokens,
                                  int32_t* dev_status, cudaStream_t s);

cudaError_t launch_schedule(const float* conf, int R, int gamma, const double* cost, float* survival,
                            int32_t* budget, double* expected, int32_t* total_tokens, unsigned long long* ws_keys,
                            int32_t* dev_status, cudaStream_t s);

cudaError_t launch_schedule_dynamic(const float* conf, const float* conf_stale, int R, int gamma, const double* cost,
                                    float* survival, int32_t* budget, double* expected, int32_t* total_tokens,
                                    int32_t* capacity, cudaStream_t s);

cudaError_t launch_pack(const int32_t* anchor, const int32_t* draft, const int32_t* budget, int R, int gamma,
                        const int32_t* tiers, int n_tiers, int strict, int32_t* cu, int32_t* ptok, int32_t* preq,
                        int32_t* ppos, int capacity, int32_t* tier, int32_t* dev_status, cudaStream_t s);

// rows_avail: the packed rows the keys cover (a window past them is flagged)
cudaError_t launch_verify_greedy_finalize(int mode, const int32_t* cu, const int32_t* draft, const int32_t* budget,
                                          const unsigned long long* row_keys, int n_chunks, int R, int gamma, int V,
                                          int rows_avail, int32_t* accept, int32_t* ceiling, int32_t* out_tok,
                                          int32_t* n_out, int32_t* dev_status, cudaStream_t s);

// Sample verify, step 2: per request, merge row LSE partials, run the
// left-to-right accept tests and choose the final row (residual or bonus).
cudaError_t launch_verify_sample_scan(int mode, const int32_t* cu, const int32_t* anchor, const int32_t* draft,
                                      const int32_t* budget, const float* logq, const void* target, int t_fp32,
                                      int V, const float2* lse_part, int n_chunks, float inv_t, uint32_t k0,
                                      uint32_t k1, uint32_t cycle, int R, int gamma, int32_t* accept,
                                      int32_t* ceiling, int32_t* res_tok, int32_t* res_pos, int32_t* res_trow,
                                      float* res_lse_p, int32_t* bonus_row, int32_t* bonus_pos, int rows_avail,
                                      int32_t* dev_status, cudaStream_t s);

// ---------------------------------------------------------------------------
// Inverse-CDF draws (select.cu).  A draw walks a row's (m, s) records, whose
// weights are s exp(m - max m), to the record holding u S, then recomputes
// the record's elements to find the id.
// ---------------------------------------------------------------------------
struct DraftSelectParams {
    const float2* blk;       // [R][nb] records of step d (MODE_CHAIN_SAMPLE)
    int nb;
    int R, B, V, r, d;       // d: 1-based draft position
    const void* L;           // [R, B, V]
    int l_fp32;
    const uint16_t* U;       // [V, r]
    const uint16_t* W;       // [r, V]
    const uint16_t* a_rows;  // [R, r] bf16 row of request i in place of U[prev] (RNN memo), or NULL
    const int32_t* anchor;
    float inv_t;
    uint32_t k0, k1, cycle;  // Philox key and cycle
    int32_t* tokens;         // [R, B]
    float* logq;             // [R, B] or NULL
    float* lse;              // [R, B] or NULL
    int32_t* dev_status;
};
cudaError_t launch_draft_select(const DraftSelectParams& p, cudaStream_t s);

struct ResampleParams {
    // residual rows (res_tok >= 0): records of MODE_RESID
    const float2* blk;       // [R][nb]
    int nb;
    const int32_t* res_tok;  // [R] token before the rejected position, -1: none
    const int32_t* res_pos;  // [R] rejected window position a
    const int32_t* res_trow; // [R] packed target row of position a
    const float* res_lse_p;  // [R]
    const float* lse_q;      // [R, gamma]
    const void* L;           // [R, gamma, V]
    int l_fp32;
    const uint16_t* U;
    const uint16_t* W;
    int r;
    // bonus rows (bonus_row >= 0): chunk log-sum-exp partials of the target row
    const int32_t* bonus_row;
    const int32_t* bonus_pos;
    const float2* lse_part;  // [rows][n_chunks]
    int n_chunks, chunk;
    const void* target;
    int t_fp32;
    int R, gamma, V;
    float inv_t;
    uint32_t k0, k1, cycle;
    const int32_t* draft;    // [R, gamma]
    const int32_t* accept;   // [R]
    int32_t* out_tok;        // [R, gamma + 1]
    int32_t* n_out;          // [R]
    int32_t* dev_status;
};
cudaError_t launch_resample(const ResampleParams& p, cudaStream_t s);

// PCTree level: per frontier row, log-sum-exp and the top-k children by z.
struct TreeSelectParams {
    const float2* blk;       // [rows][nb] records of this level (MODE_TREE)
    int nb;
    int rows, P, B, V, r, k, d;
    const int32_t* front_tok;   // [rows], -1: empty slot
    const void* L;              // [R, B, V]
    int l_fp32;
    const uint16_t* U;
    const uint16_t* W;
    float2* row_top;            // [rows][kMaxTopK] (z, id bits) in rank order
    float* row_lse;             // [rows]
    int32_t* dev_status;
};
cudaError_t launch_tree_select(const TreeSelectParams& p, cudaStream_t s);

// PCTree level by bound pruning (tree_pruned.cu): once per cycle, per
// (request, level) row, the ids any parent can need (from the scan's lists
// and the prepared tables); per level and request, the top-k children of
// every frontier parent, their scores from the MODE_TREE_LSE partials, the
// per-level prune.
constexpr int kMaxTreeSlots = 64;   // frontier slots P (P k <= 64, k >= 1)
constexpr int kTreeKeep = 192;      // ids kept per row (more: the exhaustive path)

struct TreeRowsParams {
    const uint2* cand;          // the scan's lists [rows][n_chunks][kSegCap]
    const int32_t* cand_n;      // [rows][n_chunks]
    int n_chunks, rows, V, k;
    const float* c_max;         // [1] (prepared)
    uint2* keep;                // [rows][kTreeKeep] (id, L bits), (L desc, id asc)
    int32_t* n_keep;            // [rows]; -1: the row takes the exhaustive path
    float* lk;                  // [rows] the row's k-th largest backbone logit
    const float* cmax;          // the scan's chunk maxima [rows][n_chunks]
    float* lmax;                // [rows] the row's largest backbone logit
};
cudaError_t launch_tree_rows(const TreeRowsParams& p, cudaStream_t s);

struct TreeLevelParams {
    const uint2* keep;          // tree_rows_kernel's outputs
    const int32_t* n_keep;
    const float* lk;
    const void* L;              // [R, B, V]
    int l_fp32;
    const uint16_t* U;          // [V, r]
    const uint16_t* Wt;         // [V, r] (prepared)
    const float* c_bound;       // [V] (prepared)
    int R, B, V, r, P, k, d;
    const float2* part;         // [R * P][n_part] (max, sum) partials of MODE_TREE_LSE
    int n_part;
    int32_t* front_tok;
    int32_t* front_node;
    float* front_score;
    int32_t* n_front;
    int32_t* pool_tok;
    int32_t* pool_parent;
    int32_t* pool_depth;
    float* pool_score;
    int32_t* pool_n;
    int32_t* dev_status;
};
size_t tree_level_smem(int P, int r);
cudaError_t launch_tree_level(const TreeLevelParams& p, cudaStream_t s);

// PCTree
cudaError_t launch_tree_init(const int32_t* anchor, int R, int P, int B, int32_t* front_tok, int32_t* front_node,
                             float* front_score, int32_t* n_front, int32_t* pool_tok, int32_t* pool_parent,
                             int32_t* pool_depth, float* pool_score, int32_t* pool_n, int32_t* dev_status,
                             cudaStream_t s);
cudaError_t launch_tree_merge(const float2* row_top, const float* row_lse, int R, int P, int k, int B, int d,
                              int32_t* front_tok, int32_t* front_node, float* front_score, int32_t* n_front,
                              int32_t* pool_tok, int32_t* pool_parent, int32_t* pool_depth, float* pool_score,
                              int32_t* pool_n, cudaStream_t s);
cudaError_t launch_tree_finalize(int R, int P, int B, int N, const int32_t* pool_tok, const int32_t* pool_parent,
                                 const int32_t* pool_depth, const float* pool_score, const int32_t* pool_n,
                                 int32_t* tok, int32_t* parent, int32_t* depth, float* score, uint32_t* mask,
                                 int32_t* n_nodes, cudaStream_t s);
cudaError_t launch_tree_verify_walk(const unsigned long long* row_keys, int n_chunks, const int32_t* tok, const int32_t* parent,
                                    const int32_t* n_nodes, int R, int N, int B, int V, int32_t* accept,
                                    int32_t* out_tok, int32_t* n_out, int32_t* dev_status, cudaStream_t s);

// ---------------------------------------------------------------------------
// Greedy chain by bound pruning: a scan of every row of L, then one CTA per
// request walks the B steps
// ---------------------------------------------------------------------------
constexpr int kChunkBytes = 32 * 1024;         // bytes of a row of L per scan work item
constexpr int kSegCap = 512;                   // listed ids per chunk
constexpr int kMaxPickSteps = 64;              // B limit of the pruned chain
constexpr int kMaxPickChunks = 64;             // chunks-per-row limit of the pruned chain

// The budget scheduler and the ragged layout run by one extra CTA of the
// greedy chain's scan (on != 0): from the confidences, costs and tiers alone,
// while the scan's other CTAs list the candidates; the pick then writes its
// drafts into that layout.
struct FrontParams {
    int on;
    const float* conf;        // [R, B] confidences
    const double* cost;       // [R (B + 1) + 1] step costs
    float* survival;          // [R, B]
    int32_t* budget;          // [R]
    double* expected;         // [1]
    int32_t* total_tokens;    // [1]
    int n_pad;                // R B rounded up to a power of two
    int use_budget;           // pack budget[i] drafts (compact) or all B (static)
    const int32_t* tiers;
    int n_tiers, strict;
    int32_t* cu;              // [R + 1]
    int32_t* ptok;            // [capacity]
    int32_t* preq;
    int32_t* ppos;
    int capacity;
    int32_t* tier;            // [1]
};

struct PrunedParams {
    const void* L;
    int l_fp32;
    int R, B, V, r;
    int n_chunks;           // scan work items per row
    const int32_t* anchor;
    const uint16_t* U;      // [V, r]
    const uint16_t* Wt;     // [V, r] (prepared)
    const float* c_bound;   // [V] bound on |Markov(y)| over the vocabulary (prepared)
    const float* c_max;     // [1] max_y c_bound[y] (prepared)
    uint2* cand;            // [R * B][n_chunks][kSegCap] listed (id, L bits)
    int32_t* cand_n;        // [R * B][n_chunks] list lengths (true counts)
    float* cmax;            // [R * B][n_chunks] chunk maxima
    int32_t* tokens;        // [R, B]
    int32_t* dev_status;
    int kth;                // lists for the k-th largest (PCTree, k > 1); 0 or 1: the chain's argmax
    // the pick's drafts also into a ragged layout (NULL: none): rows
    // pack_cu[i] + 1 .. pack_cu[i] + n_i of pack_tok, n_i = pack_cu[i+1] - pack_cu[i] - 1
    const int32_t* pack_cu;
    int32_t* pack_tok;
    int pack_cap;
    FrontParams fr;         // the scan's extra CTA (fr.on): scheduler and layout
};
// The scan alone, then (after the caller's dependency, e.g. an event wait)
// the pick alone.
cudaError_t launch_chain_pick(const PrunedParams& p, cudaStream_t s);

int pruned_chunks(int V, int l_fp32);
cudaError_t launch_chain_pruned(const PrunedParams& p, cudaStream_t s);
// The candidate lists alone (every (request, step) row), for a top-k of
// kth > 1 (PCTree levels); with p.fr.on one more CTA runs the scheduler and
// the ragged layout.
cudaError_t launch_chain_scan(const PrunedParams& p, cudaStream_t s);
// Dynamic shared memory of the scan's scheduler CTA (0 when off); the fused
// front is offered up to kFrontSmemMax.
size_t chain_front_smem(int R, int B);
constexpr size_t kFrontSmemMax = 48 * 1024;
// Prepared tables, step 1: W^T, |U[v]|, max |W[:, v]| and max |U[v]|; zeroes
// absmax_bits for the absmax GEMM.  Step 2 (after that GEMM): the bounds.
cudaError_t launch_markov_prepare(const uint16_t* U, const uint16_t* W, int V, int r, uint16_t* Wt, float* u_norm,
                                  float* n_max, float* u_max, unsigned int* absmax_bits, cudaStream_t s);
cudaError_t launch_markov_bounds(const unsigned int* absmax_bits, const float* u_norm, const float* n_max, int V,
                                 int r, float* c_bound, float* c_max, cudaStream_t s);

int num_sms();

// ---------------------------------------------------------------------------
// Observability (observe.cu): the soft-label row list and reductions, and the
// verify-cycle statistics
// ---------------------------------------------------------------------------
cudaError_t launch_label_prep(const int32_t* cu, const int32_t* anchor, const int32_t* draft, const float* lse_q,
                              const float2* lse_part, int n_chunks, int R, int gamma, int V, int row_capacity,
                              int32_t* res_req, int32_t* res_pos, int32_t* res_tok, int32_t* res_trow,
                              float* res_lse_p, float* row_lse_q, float* label, int32_t* dev_status, cudaStream_t s);
cudaError_t launch_label_lse_q(const float2* part, int n_part, int rows, const int32_t* res_tok, float* row_lse_q,
                               cudaStream_t s);
cudaError_t launch_label_finalize(const float2* part, int n_part, int rows, const int32_t* res_tok,
                                  const int32_t* res_req, const int32_t* res_pos, int gamma, float* label,
                                  cudaStream_t s);
size_t observe_smem_bytes(int gamma, int n_class, int n_bins);
cudaError_t launch_observe(const float* conf, const int32_t* cu, const int32_t* ceiling, const int32_t* cls, int R,
                           int gamma, int n_class, int n_bins, int32_t* hist, int32_t* reached, int32_t* hits,
                           int32_t* bin_n, int32_t* bin_hit, double* bin_conf, double* ece, int32_t* dev_status,
                           cudaStream_t s);

// RNN head memo update (rnn.cu): m_d = tanh(A m_{d-1} + U[y_{d-1}] + x_d)
struct RnnStepParams {
    const uint16_t* A;                 // [r, r] bf16, row j = output j
    const uint16_t* U;                 // [V, r] bf16 token table
    const uint16_t* X;                 // [R, B, r] bf16 projected backbone states
    const int32_t* anchor;             // [R] y_0
    const unsigned long long* keys;    // greedy: [B][R] argmax keys (y_{d-1} from keys[d-2]), else NULL
    const int32_t* tokens;             // sampling: [R, B] drawn tokens (y_{d-1} = column d-2)
    int R, B, V, r, d;
    float* m;                          // [R, r] fp32 memo: m_{d-1} in, m_d out
    uint16_t* a_rows;                  // [R, r] bf16(m_d)
    float* memo_out;                   // [R, B, r] fp32 trajectory, or NULL
    int32_t* dev_status;
};
cudaError_t launch_rnn_step(const RnnStepParams& p, cudaStream_t s);

// Fixed-threshold verify length and its sweep (threshold.cu)
cudaError_t launch_schedule_threshold(const float* conf, int R, int gamma, float tau, int32_t* budget,
                                      int32_t* total_tokens, cudaStream_t s);
cudaError_t launch_threshold_sweep(const float* conf, const int32_t* ceiling, int R, int gamma, const float* taus,
                                   int K, int32_t* drafts, int32_t* accepted, double* expected, cudaStream_t s);

}  // namespace sdm
