/*
 * sdm.h - C-ABI of the DSpark / PCTree speculative-decoding hot path on one
 * GB300 GPU (sm_103a).
 *
 * Library: libsdm.so (speculative_decoding_markov_gb300/libsdm.so).
 *
 * One decode cycle of semi-autoregressive speculative decoding is
 *   draft (Markov head, chain or PCTree)  ->  schedule (survival product and
 *   throughput-maximising prefix budget)  ->  pack (ragged front-pack into a
 *   captured tier)  ->  [target LLM forward: outside this library]  ->  verify.
 *
 * Sources, cited by page and section:
 *   [DSpark notes]  LayerX ML study-group notes (2026-06-30), summary of
 *                   "DSpark: Confidence-Scheduled Speculative Decoding with
 *                   Semi-Autoregressive Generation", sections 1-9.
 *   [PCTree]        Qiita article on PCTree (Parent-Conditioned Drafting Tree),
 *                   section on tree drafting with the Markov head.
 *   [SGLang]        "DSpark in SGLang" (winzheng.jp), sections on the SPS cost
 *                   table, ragged verify and the three verify modes.
 *
 * Conventions for every entry point:
 *   - Every pointer argument is a DEVICE pointer unless the comment says
 *     "host".  The caller owns every buffer; the library never allocates.
 *     Scratch memory is the caller's `ws` buffer of at least
 *     sdm_workspace_size(op, ...) bytes (256-byte aligned).
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t passed as
 *     void*; NULL is the legacy default stream).  The return value reports
 *     host-side validation and launch errors only.
 *   - Conditions found on the device (out-of-range token ids, a verify window
 *     that does not fit, a bounded wait that ran out, a packed total above
 *     every tier) are OR-ed into *dev_status (device int32, SDM_DEV_* bits);
 *     the caller reads it after synchronising.  No kernel traps.
 *   - Layouts are row-major.  bf16 arrays are raw 16-bit patterns.
 *     L is [R, B, V]: L[i, d-1, :] is the backbone logit row of draft
 *     position d of request i.  U is [V, r], W is [r, V].
 *   - Constraints: V % 8 == 0, r % 64 == 0 and r <= 256, L/U/W/target base
 *     addresses 16-byte aligned.  Anything else returns SDM_ERR_UNSUPPORTED.
 *   - Randomness (sampling only) is Philox4x32-10 with key (seed mod 2^32,
 *     seed >> 32) and counter (0, request, stream << 16 | row,
 *     cycle mod 2^32); its word 0, w, gives u = (2 (w >> 9) + 1) 2^-24, one
 *     uniform per decision.  Streams: 0 draft, 1 accept test, 2 residual,
 *     3 bonus.
 *   - Ties: argmax and top-k prefer the lowest token id; the scheduler ranks
 *     (survival desc, request asc, position asc); PCTree prunes by (score
 *     desc, parent slot asc, child rank asc) and selects by (score desc,
 *     depth asc, creation order asc).
 *   - Calls are independent (no global state); results are deterministic.
 */
#ifndef SDM_H
#define SDM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SDM_OK = 0,
    SDM_ERR_INVALID_ARG = 1,   /* null pointer, non-positive size, bad enum */
    SDM_ERR_UNSUPPORTED = 2,   /* shape or alignment outside the constraints */
    SDM_ERR_TIER_OVERFLOW = 3, /* strict tier mode: packed total above every tier (from sdm_status_of_device) */
    SDM_ERR_CUDA = 4,          /* a CUDA runtime or driver call failed */
    SDM_ERR_WORKSPACE = 5,     /* ws is NULL or smaller than required */
    SDM_ERR_DEVICE = 6,        /* a device-side input check failed (from sdm_status_of_device) */
    SDM_ERR_TIMEOUT = 7        /* a bounded device wait ran out (from sdm_status_of_device) */
} sdm_status;

typedef enum { SDM_BF16 = 0, SDM_FP32 = 1 } sdm_dtype;
typedef enum { SDM_GREEDY = 0, SDM_SAMPLE = 1 } sdm_decode;
typedef enum { SDM_STATIC = 0, SDM_COMPACT = 1, SDM_CAP_ACCEPT = 2 } sdm_vmode;

/* bits OR-ed into *dev_status */
enum {
    SDM_DEV_BAD_TOKEN = 1,        /* a token id outside [0, V) was read */
    SDM_DEV_TIER_UNCAPTURED = 2,  /* packed total above every tier: tier = total */
    SDM_DEV_TIMEOUT = 4,          /* a bounded pipeline wait ran out */
    SDM_DEV_BAD_WINDOW = 8,       /* budget or cu_seqlens window outside [0, gamma] */
    SDM_DEV_CAPACITY = 16,        /* packed rows would exceed the given capacity */
    SDM_DEV_BAD_CLASS = 32,       /* a request class id outside [0, n_class) */
    SDM_DEV_TIER_OVERFLOW = 64    /* strict pack: packed total above every tier */
};

/* The status a caller reports for the device bits it read back after
 * synchronising: SDM_OK for 0 or SDM_DEV_TIER_UNCAPTURED alone (informational:
 * the caller runs that cycle uncaptured); else, by precedence,
 * SDM_ERR_TIMEOUT (SDM_DEV_TIMEOUT), SDM_ERR_TIER_OVERFLOW
 * (SDM_DEV_TIER_OVERFLOW), SDM_ERR_DEVICE (any other bit). */
sdm_status sdm_status_of_device(int32_t dev_status_bits);

/* Philox key material: key = seed, counter word 3 = cycle. */
typedef struct {
    uint64_t seed;
    uint64_t cycle;
} sdm_rng;

/* Operation ids for sdm_workspace_size. */
enum {
    SDM_OP_DRAFT_CHAIN = 0,
    SDM_OP_DRAFT_TREE = 1,
    SDM_OP_SCHEDULE = 2,
    SDM_OP_PACK = 3,
    SDM_OP_VERIFY = 4,
    SDM_OP_VERIFY_TREE = 5,
    SDM_OP_TV_LABEL = 6,
    SDM_OP_DRAFT_CHAIN_RNN = 7
};

/* Bytes of scratch the operation needs for these sizes (0 if none).  Pass the
 * same sizes as the call; unused sizes may be 0.  For SDM_OP_VERIFY and
 * SDM_OP_TV_LABEL pass the packed row capacity as P. */
size_t sdm_workspace_size(int op, int R, int B, int V, int r, int P, int k, int N);

/*
 * markov_prepare: tables derived once from the Markov head (U, W), for the
 * greedy chain (no counterpart on the pages; a weight-preparation step, like
 * packing a weight matrix at load time).  Fills `prepared` (device, at least
 * sdm_markov_prepared_size(V, r) bytes, 256-byte aligned) with, in order,
 * each array starting on a 256-byte boundary:
 *   W^T [V, r] bf16;
 *   c [V] fp32: c(y) bounds |U[y] . W[:, v]| over every v, for the exact
 *     product and for any fp32 evaluation of it:
 *       c(y) = A(y) (1 + 2^-10) + 4 r 2^-24 |U[y]|_2 max_v |W[:, v]|_2 + 2^-20
 *     rounded up, A(y) = max_v |U[y] . W[:, v]| accumulated in fp32 by the
 *     tensor cores (one V x V x r product, about 12 TFLOP at V = 151,936,
 *     r = 256; nothing of it is stored);
 *   |U[v]|_2 [V] fp32 (fp64 accumulation, rounded up); A [V] (scratch);
 *   c_max = max_y c(y), max_v |W[:, v]|_2, max_v |U[v]|_2 (fp32 each).
 * A pipeline wait that runs out sets SDM_DEV_TIMEOUT in *dev_status (may be
 * NULL).  Enqueued on `stream`; valid until U or W change.
 */
size_t sdm_markov_prepared_size(int V, int r);
sdm_status sdm_markov_prepare(const uint16_t* U, const uint16_t* W, int V, int r, void* prepared,
                              size_t prepared_bytes, int32_t* dev_status, void* stream);

/*
 * draft_chain: the Markov-head sequential stage ([DSpark notes] sec. 4,
 * "Sequential stage" and "Markov head"; [PCTree] z_d = L_d + Markov(y_{d-1})).
 * For d = 1..B, with y_0 = anchor:
 *     z_d = fp32(L[i, d-1, :]) + U[y_{d-1}] . W          (fp32)
 *     greedy:  y_d = argmax_v z_d[v]
 *     sample:  y_d ~ softmax(z_d / T) by the inverse CDF in vocabulary
 *              order: the smallest v with sum_{j<=v} exp(z_d[j]/T) > u S,
 *              S the sum over all j, u = the uniform of (stream 0, row d);
 *              lse[i, d-1] = log sum_v exp(z_d[v]/T);
 *              logq[i, d-1] = z_d[y_d]/T - lse[i, d-1].
 * In:  L [R, B, V] (dtL), U [V, r] bf16, W [r, V] bf16, anchor [R] int32;
 *      prepared: NULL, or the tables sdm_markov_prepare built from U and W.
 * Out: tokens [R, B] int32; logq, lse [R, B] fp32 (sample only; may be NULL
 *      when greedy).
 * Sampling (and greedy without prepared tables): the product U[y] . W runs on
 * the tcgen05 tensor cores (bf16 in, fp32 accumulate in TMEM) and the +L /
 * argmax (greedy) or per-16-column (max, sum of exp) records (sampling) are
 * fused into its epilogue; z is never written to memory.  A sampled step
 * then walks the records of each request to the block holding u S and
 * recomputes that block's 16 logits to find the id (V <= 524288, else
 * SDM_ERR_UNSUPPORTED).
 * Greedy with prepared tables: since |U[y] . W[:, v]| <= c(y) for every v,
 * only ids with L[v] >= max L - 2 c(y) can win.  One HBM-bound pass over all
 * of L lists those ids for every (request, step) with the worst case c_max,
 * then one CTA per request stages the listed rows of W^T and U in shared
 * memory and walks the B steps, scoring exactly the ids that the previous
 * token's c(y) leaves.  L is read once and the result is the same argmax bit
 * for bit.  Needs B <= 64, V <= 64 * 16384 (bf16 L) or 64 * 8192 (fp32 L) and
 * R * B * ceil(V / 16384 or 8192) <= 2^30, else SDM_ERR_UNSUPPORTED.
 */
sdm_status sdm_draft_chain(const void* L, sdm_dtype dtL, const uint16_t* U, const uint16_t* W,
                           const void* prepared, const int32_t* anchor, int R, int B, int V, int r,
                           sdm_decode decode, float temperature, sdm_rng rng,
                           int32_t* tokens, float* logq, float* lse,
                           void* ws, size_t ws_bytes, int32_t* dev_status, void* stream);

/*
 * draft_chain_packed: the greedy chain of sdm_draft_chain with prepared
 * tables, writing its drafts also into the ragged verify layout (the pack of
 * [SGLang] "ragged verify" without a pass of its own after the draft).  The
 * layout is sdm_pack_ragged's with draft = NULL (cu_seqlens, the tier, the
 * row maps and the anchors, made from the budgets alone, e.g. on a second
 * stream while this draft runs); this call fills rows cu[i] + 1 .. cu[i] +
 * n_i of packed_tok with y_1 .. y_{n_i}, n_i = cu[i+1] - cu[i] - 1, so that
 * packed_tok ends as sdm_pack_ragged with the drafts would leave it.
 * layout_ready (a cudaEvent_t, may be NULL): recorded after the layout's
 * producer; the scan of L starts at once, the pass that writes the drafts
 * waits for the event on `stream`.  NULL: the layout is ordered before this
 * call on `stream`.
 * In/out as sdm_draft_chain (prepared required); cu_seqlens [R+1],
 * packed_tok [capacity] (device).  A window longer than B sets
 * SDM_DEV_BAD_WINDOW (cut to B); rows past capacity SDM_DEV_CAPACITY.
 */
sdm_status sdm_draft_chain_packed(const void* L, sdm_dtype dtL, const uint16_t* U, const uint16_t* W,
                                  const void* prepared, const int32_t* anchor, int R, int B, int V, int r,
                                  const int32_t* cu_seqlens, int32_t* packed_tok, int capacity, void* layout_ready,
                                  int32_t* tokens, void* ws, size_t ws_bytes, int32_t* dev_status, void* stream);

/*
 * draft_chain_front: the greedy chain draft together with the budget
 * scheduler and the ragged layout of its windows, in one call whose outputs
 * equal, bit for bit, those of
 *     sdm_schedule_budget(conf, R, B, cost, survival, budget, expected,
 *                         total_tokens)
 *     sdm_pack_ragged(anchor, NULL, use_budget ? budget : NULL, R, B, tiers,
 *                     n_tiers, strict, cu_seqlens, packed_tok, packed_req,
 *                     packed_pos, capacity, tier)
 *     sdm_draft_chain_packed(L, ..., prepared, anchor, R, B, V, r,
 *                            cu_seqlens, packed_tok, capacity, NULL, tokens)
 * ([DSpark notes] sec. 4, 5.1-5.2; [SGLang] "ragged verify").  The scheduler
 * and the layout need only the confidences, so they run in one extra CTA of
 * the draft's first (vocabulary-streaming) launch, beside its other CTAs,
 * and the pick writes the drafts into the layout; nothing runs on a second
 * stream.  It pays when the scan fills every SM (a side-stream scheduler
 * then waits for the scan to drain: 67.4 against 70.5 us per decode cycle
 * of 64 requests, B 7, V 151936); on a scan of a few CTAs the scheduler's
 * CTA is the longer path, and the three calls with the scheduler on a second
 * stream are faster.  Requires the prepared tables and R * B <= 8192 with the
 * scheduler's shared memory (about 16 (R B) bytes rounded up) within 48 KB,
 * else SDM_ERR_UNSUPPORTED (use the three calls).  Arguments as in those
 * calls; use_budget 1 packs budget[i] drafts per request (compact), 0 all B
 * (static); the tier's host copy is not offered.  Workspace: as
 * SDM_OP_DRAFT_CHAIN.
 */
sdm_status sdm_draft_chain_front(const void* L, sdm_dtype dtL, const uint16_t* U, const uint16_t* W,
                                 const void* prepared, const int32_t* anchor, int R, int B, int V, int r,
                                 const float* conf, const double* cost, int use_budget, const int32_t* tiers,
                                 int n_tiers, int strict, float* survival, int32_t* budget, double* expected,
                                 int32_t* total_tokens, int32_t* cu_seqlens, int32_t* packed_tok, int32_t* packed_req,
                                 int32_t* packed_pos, int capacity, int32_t* tier, int32_t* tokens, void* ws,
                                 size_t ws_bytes, int32_t* dev_status, void* stream);

/*
 * draft_chain_rnn: the chain draft with the RNN sequential head ([DSpark
 * notes] sec. 4, "RNN head": a memo that carries the whole draft so far,
 * updated once per step from the previous memo, the previous word and the
 * current backbone state; the page's formula is not legible, the reading
 * taken is)
 *     m_0 = 0,  m_d = tanh(A m_{d-1} + U[y_{d-1}] + x_d)
 *     z_d = L_d + bf16(m_d) . W
 * then y_d as in draft_chain (greedy argmax, or the inverse-CDF draw of
 * softmax(z_d / T) with the same random stream).  With A = 0 and x = 0 this
 * is the Markov head on the table bf16(tanh(U)).
 * In:  L [R, B, V] (dtL), U [V, r], W [r, V], A [r, r] (row j = output j),
 *      X [R, B, r] (x_d: the backbone state at position d projected to r),
 *      all bf16 but L; anchor [R].  Shapes and alignment as draft_chain.
 * Out: tokens [R, B]; logq, lse [R, B] fp32 (sampling; may be NULL);
 *      memo [R, B, r] fp32 = m_d per position (may be NULL).  The memo is
 *      formed in fp32 (tanhf); the projection on the tensor cores with fp32
 *      accumulation.
 * ws:  sdm_workspace_size(SDM_OP_DRAFT_CHAIN_RNN, R, B, V, r, 0, 0, 0).
 * Device checks as draft_chain (a token id outside [0, V) sets
 * SDM_DEV_BAD_TOKEN and is read as 0).
 */
sdm_status sdm_draft_chain_rnn(const void* L, sdm_dtype dtL, const uint16_t* U, const uint16_t* W, const uint16_t* A,
                               const uint16_t* X, const int32_t* anchor, int R, int B, int V, int r, sdm_decode decode,
                               float temperature, sdm_rng rng, int32_t* tokens, float* logq, float* lse, float* memo,
                               void* ws, size_t ws_bytes, int32_t* dev_status, void* stream);

/*
 * draft_tree: PCTree drafting ([PCTree]: per parent p, z_d(p) = L_d +
 * Markov(p) for every frontier parent in one batched Markov call; local top-k
 * per parent; path score s(c) = s(p) + log pi(v | p); top-P prune per level;
 * global top-N selection within the verify budget; the tree is verified in one
 * target forward with a tree-causal mask ([DSpark notes] JetSpec note: a node
 * attends to its ancestors only)).
 * Level 1 expands the root (token anchor[i], score 0); level d expands the
 * <= P nodes kept at level d-1.  Scores use T = 1 and are fp32.
 * Out (per request, N+1 slots; slot 0 = root, then the selected nodes in
 * rank order so parent[c] < c; unused slots hold -1 / 0):
 *   tok, parent, depth [R, N+1] int32; score [R, N+1] fp32;
 *   mask [R, N+1, ceil((N+1)/32)] uint32, bit j of row c set iff slot j is c
 *   or an ancestor of c; n_nodes [R] int32 (root included).
 * prepared: NULL, or the tables sdm_markov_prepare built from U and W.
 * With prepared tables: since |U[y] . W[:, v]| <= c(y) for every v, the top
 * k ids of parent y have L[v] >= L_(k) - 2 c(y), L_(k) the k-th largest
 * backbone logit of the row.  One HBM-bound pass over L lists, per 32 KB
 * chunk of every (request, level) row, the ids with L >= theta - 2 c_max
 * (theta a lower bound on the chunk's k-th largest value); each level then
 * runs the tcgen05 GEMM for every frontier row with only an online
 * log-sum-exp in its epilogue, and one CTA per request scores the listed ids
 * each parent can need exactly (z = L + U[y] . W^T[v]), takes each parent's
 * top k, the children's scores and the prune.  A row whose lists overflow
 * takes the exact top k over the whole vocabulary instead (slow).  Needs
 * V <= 64 * 16384 (bf16 L) or 64 * 8192 (fp32 L), R B ceil(V / 16384 or
 * 8192) <= 2^30.
 * Without: each level runs the tcgen05 GEMM for every frontier row with
 * per-16-column (max, sum of exp) records in its epilogue; the row's top-k
 * ids lie in the k blocks with the largest maxima, so one CTA per row ranks
 * the records, recomputes the logits of its 2k best blocks and ranks those.
 * Both give the same tree.
 * Constraints: 1 <= k <= 8, 1 <= P, P*k <= 64, 128 % P == 0, N <= P*B,
 * P*B + 1 <= 8192, V <= 524288 (else SDM_ERR_UNSUPPORTED).
 */
sdm_status sdm_draft_tree(const void* L, sdm_dtype dtL, const uint16_t* U, const uint16_t* W, const void* prepared,
                          const int32_t* anchor, int R, int B, int V, int r, int k, int P, int N,
                          int32_t* tok, int32_t* parent, int32_t* depth, float* score,
                          uint32_t* mask, int32_t* n_nodes,
                          void* ws, size_t ws_bytes, int32_t* dev_status, void* stream);

/*
 * schedule_budget: confidence survival and the hardware-aware prefix budget
 * ([DSpark notes] sec. 5.1 and 5.2; [SGLang] "SPS cost table").
 *   S[i, k] = S[i, k-1] * c[i, k]  (fp32, k = 1..gamma, S[i, 0] = 1)
 *   Survivals >= 2^-18 are ranked (S desc, request asc, position asc); with
 *   E(m) = R + sum of the top m and N(m) = R + m, the greedy adds the next
 *   survival while E(m+1)/cost[N(m+1)] > E(m)/cost[N(m)] and stops at the
 *   first that does not improve it.  budget[i] = request i's count in the
 *   top m*.  Sums are exact in fp64.
 * In:  conf [R, gamma] fp32 (post-sigmoid), cost [R*(gamma+1)+1] fp64 (step
 *      cost by total verify tokens).
 * Out: survival [R, gamma] fp32, budget [R] int32, expected [1] fp64 (E(m*)),
 *      total_tokens [1] int32 (N(m*)).
 * Constraint: R * gamma <= 8192.
 */
sdm_status sdm_schedule_budget(const float* conf, int R, int gamma, const double* cost,
                               float* survival, int32_t* budget, double* expected,
                               int32_t* total_tokens, void* ws, size_t ws_bytes,
                               int32_t* dev_status, void* stream);

/*
 * schedule_dynamic: the production scheduler ([DSpark notes] sec. 9.2,
 * "scheduler adaptation on real hardware").  The step's batch capacity must
 * be known before the step's own confidences are, so it comes from the
 * confidences of two steps before; the step's candidates are still ranked by
 * their own survivals (dynamic top-K); and because the capacity no longer
 * depends on this step's tokens, the search over the cost table is global,
 * which crosses the steps of a tiered table that an early stop would not.
 *   S'[i, k], S[i, k]: the survival products of conf_stale and conf (fp32,
 *   left to right), ranked as in schedule_budget (S desc, request asc,
 *   position asc; values below 2^-18 are left out).
 *   K = the m in 0 .. (ranked S') maximising E'(m) / cost[R + m], E'(m) =
 *   R + sum of the top m of S' (exact fp64), the smallest m on ties.
 *   budget[i] = request i's count in the top min(K, ranked S) of S.
 * In:  conf, conf_stale [R, gamma] fp32 (post-sigmoid), cost
 *      [R*(gamma+1)+1] fp64, every entry > 0 (it may step with the tier).
 * Out: survival [R, gamma] fp32 (of conf), budget [R] int32, expected [1]
 *      fp64 (R + the selected survivals), total_tokens [1] int32
 *      (R + min(K, ranked S)), capacity [1] int32 (K).
 * Constraint: R * gamma <= 8192.
 */
sdm_status sdm_schedule_dynamic(const float* conf, const float* conf_stale, int R, int gamma,
                                const double* cost, float* survival, int32_t* budget,
                                double* expected, int32_t* total_tokens, int32_t* capacity,
                                int32_t* dev_status, void* stream);

/*
 * pack_ragged: ragged front-pack of the verify windows ([SGLang] "ragged
 * verify": windows are front-packed into a compact cu_seqlens buffer whose
 * total is rounded up to the nearest captured tier).
 *   n_i = budget[i] (budget == NULL: n_i = gamma, the static block)
 *   cu_seqlens[0] = 0, cu_seqlens[i+1] = cu_seqlens[i] + n_i + 1
 *   rows cu[i] .. cu[i] + n_i hold y_0 (anchor), y_1 .. y_{n_i}, with
 *   packed_req = i and packed_pos = 0..n_i; rows total .. capacity-1 hold -1.
 *   tier = smallest tiers[q] >= total; above every tier: tier = total and
 *   SDM_DEV_TIER_UNCAPTURED is set (the caller runs uncaptured), or, with
 *   strict != 0, SDM_DEV_TIER_OVERFLOW instead (a caller that only runs
 *   captured tiers maps it to SDM_ERR_TIER_OVERFLOW with
 *   sdm_status_of_device; the rows are packed the same way).
 * In:  anchor [R], draft [R, gamma] or NULL (the layout alone: every draft
 *      row holds -1, for sdm_draft_chain_packed to fill), budget [R] or
 *      NULL, tiers [n_tiers] int32 (device), strict (0 or 1).
 * Out: cu_seqlens [R+1], packed_tok/req/pos [capacity], tier [1] (device);
 *      tier_host (host, may be NULL): if non-NULL it must be pinned host
 *      memory and receives the tier by an async copy on `stream`.
 * capacity >= max(max tier, R*(gamma+1)) guarantees every row fits; rows past
 * capacity are dropped and SDM_DEV_CAPACITY is set.
 */
sdm_status sdm_pack_ragged(const int32_t* anchor, const int32_t* draft, const int32_t* budget,
                           int R, int gamma, const int32_t* tiers, int n_tiers, int strict,
                           int32_t* cu_seqlens, int32_t* packed_tok, int32_t* packed_req,
                           int32_t* packed_pos, int capacity, int32_t* tier, int32_t* tier_host,
                           int32_t* dev_status, void* stream);

/*
 * verify: fused verification over the packed target logits ([DSpark notes]
 * sec. 1: left-to-right acceptance, discard after the first rejection, one
 * bonus token; [SGLang] "three verify modes").
 * Window of request i: w_i = cu[i+1] - cu[i] - 1 drafts, target rows
 * cu[i] .. cu[i] + w_i; row p is the target's prediction after y_p.
 *   greedy: t_p = argmax target row p; A = first p < w_i with y_{p+1} != t_p,
 *           else w_i; commit a = A drafts and t_a.
 *   sample: accept y_{p+1} iff u(stream 1, row p) < p_p(y)/q_p(y), with
 *           p = softmax(target row / T) and q_p(y) = exp(logq[i, p]); at the
 *           first rejection p = a, sample from max(0, p_a - q_a) where q_a is
 *           recomputed from L, U, W and lse_q (stream 2, row a); if all
 *           committed drafts pass, the bonus is drawn from p at row a
 *           (stream 3).  Every draw is the inverse CDF in vocabulary order
 *           with one uniform (word 0 of the Philox block of its stream and
 *           row; the row of a draft is d, of an accept test, residual or
 *           bonus the window position).  Sampling needs V <= 524288 (else
 *           SDM_ERR_UNSUPPORTED).
 *   modes: STATIC (w_i = gamma, commit A), COMPACT (w_i = budget, commit A),
 *          CAP_ACCEPT (w_i = gamma verified, commit a = min(A, budget[i]):
 *          the same output as compact; ceiling = A).
 * In:  target [rows, V] (dtT), cu_seqlens [R+1], anchor [R], draft [R, gamma];
 *      budget [R] (CAP_ACCEPT only); logq, lse_q [R, gamma] fp32, L [R, gamma,
 *      V], U, W, r (SAMPLE only, else may be NULL/0).  row_capacity = rows
 *      allocated in target (an upper bound on cu[R]).
 * Out: accept [R], ceiling [R] (may be NULL), out_tok [R, gamma+1] (-1
 *      padded), n_out [R] = accept + 1.
 * Only rows below min(cu[R], row_capacity) are read.  A request without
 * rows (cu[i+1] <= cu[i]) or whose rows end past cu[R] (a non-monotone
 * cu_seqlens) sets SDM_DEV_BAD_WINDOW, one whose rows run past row_capacity
 * sets SDM_DEV_CAPACITY; such a request commits one token (0) with accept 0
 * (greedy and sample).  A window longer than gamma is flagged
 * (SDM_DEV_BAD_WINDOW) and cut to gamma.
 */
sdm_status sdm_verify(sdm_vmode mode, sdm_decode decode, float temperature, sdm_rng rng,
                      const void* target, sdm_dtype dtT, int row_capacity, const int32_t* cu_seqlens,
                      const int32_t* anchor, const int32_t* draft, const int32_t* budget,
                      const float* logq, const float* lse_q,
                      const void* L, sdm_dtype dtL, const uint16_t* U, const uint16_t* W, int r,
                      int R, int gamma, int V,
                      int32_t* accept, int32_t* ceiling, int32_t* out_tok, int32_t* n_out,
                      void* ws, size_t ws_bytes, int32_t* dev_status, void* stream);

/*
 * verify_tree: greedy verification of a drafted tree in one target forward
 * ([PCTree]; greedy only).  Walk from the root: t = argmax of the current
 * slot's target row; move to the child whose token is t; stop when none is.
 * accept = depth reached; out_tok = accepted tokens then t (bonus).
 * In:  target [R, N+1, V] (dtT; slot c's row predicts c's child), tok, parent
 *      [R, N+1], n_nodes [R].
 * Out: accept [R], out_tok [R, B+1] (-1 padded), n_out [R].
 * When several children carry t, the lowest slot is taken.  N < 16384, else
 * SDM_ERR_UNSUPPORTED.
 */
sdm_status sdm_verify_tree(const void* target, sdm_dtype dtT, const int32_t* tok,
                           const int32_t* parent, const int32_t* n_nodes, int R, int N, int B, int V,
                           int32_t* accept, int32_t* out_tok, int32_t* n_out,
                           void* ws, size_t ws_bytes, int32_t* dev_status, void* stream);

/*
 * verify_greedy_static: greedy verification (as sdm_verify with SDM_GREEDY)
 * that allocates nothing and takes no workspace.  The pages have no
 * counterpart; this entry point exists for callers that cannot hand the
 * library scratch memory: a server that reserved all device memory up front,
 * a framework whose allocator must account for every byte, or a latency-bound
 * loop that cannot afford the device synchronisation of cudaMalloc/cudaFree.
 * Scratch: a fixed 1 MiB array in the library's own device memory (every GPU
 * that loads libsdm.so holds it until the process exits); row_capacity *
 * ceil(V / 16384) (bf16 target) or row_capacity * ceil(V / 8192) (fp32) must
 * be <= 131072, else SDM_ERR_WORKSPACE and nothing is launched.
 * The first call on a device looks the array's device address up (once per
 * device, with that device current, and again if the device's context has
 * changed since, e.g. after a device reset); make that first call before any
 * stream capture.  All calls share the one array and each call rewrites every
 * partial it reads (rows below min(cu[R], row_capacity); a window past them is
 * flagged as in sdm_verify), so nothing carries over between calls, but calls
 * that overlap on the GPU (concurrent streams) race on it: serialise them.
 * Arguments and outputs are those of sdm_verify.
 */
sdm_status sdm_verify_greedy_static(sdm_vmode mode, const void* target, sdm_dtype dtT, int row_capacity,
                                    const int32_t* cu_seqlens, const int32_t* draft, const int32_t* budget,
                                    int R, int gamma, int V, int32_t* accept, int32_t* ceiling,
                                    int32_t* out_tok, int32_t* n_out, int32_t* dev_status, void* stream);

/*
 * check_timeout_path: exercises the device-side timeout path on purpose (no
 * counterpart on the pages; a failure-detection check).  Every pipeline wait
 * of the tensor-core kernels is bounded by a wall-clock limit (2 s in normal
 * calls); when one runs out the kernel ORs SDM_DEV_TIMEOUT into *dev_status,
 * waits (bounded) for the copies and tensor-core work it has in flight, frees
 * its tensor memory and returns, so the context stays usable.  This call
 * launches the greedy chain's Markov GEMM for step 1 on the given inputs with
 * its loads withheld and every wait limited to wait_ns (1 us .. 1 s), so
 * every wait runs out: afterwards *dev_status holds SDM_DEV_TIMEOUT and
 * later calls on the stream run normally.  Nothing but the keys in ws is
 * written.
 * In:  as sdm_draft_chain (dense path); ws at least
 *      sdm_workspace_size(SDM_OP_DRAFT_CHAIN, R, B, V, r, 0, 0, 0) bytes;
 *      dev_status must not be NULL.
 */
sdm_status sdm_check_timeout_path(const void* L, sdm_dtype dtL, const uint16_t* U, const uint16_t* W,
                                  const int32_t* anchor, int R, int B, int V, int r, unsigned long long wait_ns,
                                  void* ws, size_t ws_bytes, int32_t* dev_status, void* stream);

/* Human-readable name of a status code (static string). */
const char* sdm_status_str(sdm_status status);

/* Library version, major * 10000 + minor * 100 + patch. */
int sdm_version(void);

/*
 * schedule_threshold: the conventional fixed-threshold verify length
 * ([DSpark notes] sec. 5.2: a fixed threshold on the confidences decides how
 * many drafts are verified; sec. 8.3, Fig. 5).  budget[i] = the longest
 * prefix n such that conf[i, d] >= tau for every d < n (fp32 comparison; a
 * NaN confidence ends the prefix); total_tokens = R + sum_i budget[i] (every
 * request sends its root token).
 * In:  conf [R, gamma] fp32 (device), tau.  R gamma <= 2^30.
 * Out: budget [R] int32, total_tokens [1] int32 (device).
 */
sdm_status sdm_schedule_threshold(const float* conf, int R, int gamma, float tau, int32_t* budget,
                                  int32_t* total_tokens, int32_t* dev_status, void* stream);

/*
 * threshold_sweep: the fixed-threshold rule at K thresholds at once
 * ([DSpark notes] sec. 8.3, Fig. 5: threshold 0 verifies the whole block).
 * With n_i(tau) as in schedule_threshold, for threshold k:
 *   drafts[k]   = sum_i n_i(tau_k)                     drafts verified
 *   accepted[k] = sum_i min(ceiling[i], n_i(tau_k))    drafts accepted, given
 *                 the acceptance count of the whole block (sdm_verify's
 *                 ceiling in CAP_ACCEPT or STATIC mode); -1 if ceiling NULL
 *   expected[k] = sum_i sum_{d <= n_i} S_{i,d}         expected accepted drafts,
 *                 S the fp32 running products of conf ([DSpark notes] sec.
 *                 5.1), summed exactly: each S >= 2^-24 as an integer count
 *                 of 2^-48, smaller survivals counted 0.
 * In:  conf [R, gamma] fp32, ceiling [R] int32 or NULL, taus [K] fp32
 *      (device).  R gamma <= 32768 (the exact sum stays below 2^63), K <= 65535.
 * Out: drafts, accepted [K] int32, expected [K] fp64 (device).
 */
sdm_status sdm_threshold_sweep(const float* conf, const int32_t* ceiling, int R, int gamma, const float* taus, int K,
                               int32_t* drafts, int32_t* accepted, double* expected, int32_t* dev_status,
                               void* stream);

/*
 * tv_label: the confidence head's soft label for every verified draft position
 * ([DSpark notes] sec. 5.1: the label is the single-token acceptance rate,
 * fixed by the total-variation distance between the draft and target
 * distributions):
 *     label[i, p] = sum_v min(q_v, p_v) = 1 - TV(q, p)         for p < w_i
 * with q = softmax((L[i, p] + U[y_p] . W) / T) the draft's distribution at
 * position p+1 (y_0 = anchor[i], y_p = draft[i, p-1]) and p = softmax(target
 * row cu[i] + p / T); w_i = cu[i+1] - cu[i] - 1.  label[i, p] = -1 for
 * p >= w_i.
 * In:  target [row_capacity, V] (dtT, the packed verify rows), cu_seqlens
 *      [R+1], anchor [R], draft [R, gamma]; lse_q [R, gamma] fp32 = the
 *      draft's log-sum-exp of (L + Markov) / T, as sampling drafts return it,
 *      or NULL: computed here by one more pass over L; L [R, gamma, V] (dtL),
 *      U [V, r], W [r, V] bf16, r in {64, 128, 192, 256}; temperature > 0 (1
 *      for greedy drafts).  target, L, U, W 16-byte aligned; V % 8 == 0;
 *      R gamma <= 2^22.
 * Out: label [R, gamma] fp32 (device).  Arithmetic in fp32 (exp, sums over
 *      16-column blocks, then over the vocabulary splits in a fixed order).
 * ws:  sdm_workspace_size(SDM_OP_TV_LABEL, R, gamma, V, r, row_capacity, 0, 0).
 * Device checks (OR-ed into *dev_status, the row keeps label -1): windows
 * outside [0, gamma] SDM_DEV_BAD_WINDOW, target rows past row_capacity
 * SDM_DEV_CAPACITY, previous tokens outside [0, V) SDM_DEV_BAD_TOKEN.
 */
sdm_status sdm_tv_label(float temperature, const void* target, sdm_dtype dtT, int row_capacity,
                        const int32_t* cu_seqlens, const int32_t* anchor, const int32_t* draft, const float* lse_q,
                        const void* L, sdm_dtype dtL, const uint16_t* U, const uint16_t* W, int r, int R, int gamma,
                        int V, float* label, void* ws, size_t ws_bytes, int32_t* dev_status, void* stream);

/*
 * observe: statistics of one verify cycle for offline analysis ([SGLang]
 * "observability": the acceptance ceiling that cap-accept exposes, the
 * per-request confidences and calibration metrics such as ECE; [DSpark
 * notes] sec. 8.1: position d counts only where positions 1..d-1 were all
 * accepted).  Position d = 1..gamma of request i is observed when
 * d <= min(A_i + 1, w_i), A_i = ceiling[i], w_i = cu[i+1] - cu[i] - 1; its
 * outcome is hit = (d <= A_i).
 * In:  conf [R, gamma] fp32 (the confidences the scheduler ranked),
 *      cu_seqlens [R+1] of the verify, ceiling [R] (sdm_verify's ceiling: the
 *      acceptance count of the whole verified window), cls [R] class ids in
 *      [0, n_class), n_bins >= 1.
 * Out (device): hist [n_class, gamma+1] int32: requests per class and
 *      ceiling; reached, hits [n_class, gamma] int32: observed positions and
 *      their hits per class and position; bin_n, bin_hit [n_bins] int32 and
 *      bin_conf [n_bins] fp64: per equal-width bin the observations, hits and
 *      the sum of the confidences (c clamped to [0, 1], NaN as 0, in bin
 *      floor(c n_bins) of an fp32 product, c = 1 in the top bin); ece [1]
 *      fp64 = sum_b |bin_hit_b - bin_conf_b| / N, N = sum_b bin_n_b (0 when
 *      N = 0).  bin_conf is summed by atomic adds: its last bits may differ
 *      between runs; the counts are exact.
 * Limits: 4 n_class (3 gamma + 1) + 16 n_bins <= 49152 bytes, else
 *      SDM_ERR_UNSUPPORTED.
 * Device checks: a class id outside [0, n_class) sets SDM_DEV_BAD_CLASS and
 * the request is skipped; a window outside [0, gamma] or a ceiling outside
 * [0, w_i] sets SDM_DEV_BAD_WINDOW and is clamped.
 */
sdm_status sdm_observe(const float* conf, const int32_t* cu_seqlens, const int32_t* ceiling, const int32_t* cls, int R,
                       int gamma, int n_class, int n_bins, int32_t* hist, int32_t* reached, int32_t* hits,
                       int32_t* bin_n, int32_t* bin_hit, double* bin_conf, double* ece, int32_t* dev_status,
                       void* stream);

#ifdef __cplusplus
}
#endif
#endif /* SDM_H */
