/*
 * oracle.h - CPU oracle for the DSpark / PCTree speculative-decoding hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  This is a plain, slow, single-threaded C
 * restatement of what the method computes, written from the pages that
 * describe it.  Only the tests, the smoke check and the benchmark's CPU
 * baseline leg may load it.  It shares no code, header or table with the
 * CUDA library (speculative_decoding_markov_gb300/csrc) and the library never
 * calls it.
 *
 * Page keys used in the citations below:
 *   [DSpark notes]  LayerX ML study-group notes 2026-06-30, "DSpark:
 *                   Confidence-Scheduled Speculative Decoding with
 *                   Semi-Autoregressive Generation", sections 1-9.
 *   [PCTree]        Qiita article on PCTree (Parent-Conditioned Drafting
 *                   Tree), section "a linear draft wastes everything after
 *                   the first miss".
 *   [SGLang]        winzheng.jp, "DSpark in SGLang", sections "SPS cost
 *                   table", "three verify modes", "ragged verify".
 *
 * Conventions shared with the library's C-ABI (they are conventions of the
 * interface, restated here independently):
 *   - bf16 values are passed as raw uint16 bit patterns;
 *   - L is [R, B, V] (request, draft position d-1, vocab), row-major;
 *   - U is [V, r], W is [r, V], both bf16;
 *   - the random numbers the method draws come from Philox4x32-10 (Salmon et
 *     al., SC'11) keyed by (seed, cycle); see orc_uniform().
 * Precision: the Markov product and every log/exp/ratio are in double; the
 * combined logit z = L + Markov is an fp32 addition (the pages keep logits in
 * the drafter's float type), so argmax decisions are taken on the same fp32
 * values the kernel sees.  Survival products are fp32 multiplies, expected
 * token counts fp64 sums.
 */
#ifndef SDM_ORACLE_H
#define SDM_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_BF16 = 0, ORC_FP32 = 1 };
enum { ORC_GREEDY = 0, ORC_SAMPLE = 1 };
enum { ORC_STATIC = 0, ORC_COMPACT = 1, ORC_CAP_ACCEPT = 2 };
enum { ORC_STREAM_DRAFT = 0, ORC_STREAM_ACCEPT = 1, ORC_STREAM_RESID = 2, ORC_STREAM_BONUS = 3 };
/* flag bits returned through *flags */
enum { ORC_FLAG_TIER_UNCAPTURED = 2, ORC_FLAG_INEXACT_MARKOV = 16, ORC_FLAG_TIER_OVERFLOW = 64 };

/* Philox4x32-10 block function, straight from its published definition. */
void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);
/* The uniform in (0,1) for (stream, request, row, vocab id v). */
double orc_uniform(uint64_t seed, uint64_t cycle, int stream, uint32_t req, uint32_t row, uint32_t v);

/* Markov-head chain draft.  req_ids (may be NULL = 0..R-1) gives the global
 * request index used for the random counters, so a subset of requests can be
 * drafted on its own.  logq, lse, margin may be NULL. */
int orc_draft_chain(const void* L, int dtL, const uint16_t* U, const uint16_t* W,
                    const int32_t* anchor, const int32_t* req_ids, int R, int B, int V, int r,
                    int decode, double temperature, uint64_t seed, uint64_t cycle,
                    int32_t* tokens, double* logq, double* lse, double* margin);

/* PCTree drafting.  Outputs hold N+1 slots per request (slot 0 = root);
 * mask holds ceil((N+1)/32) words per node row.  margin [R, B+2] (may be
 * NULL), one per decision: [i, d-1] the score gap at the prune boundary of
 * level d, [i, B] at the top-N boundary, [i, B+1] the smallest gap between
 * neighbours of the output ranking; INFINITY where nothing was cut. */
int orc_draft_tree(const void* L, int dtL, const uint16_t* U, const uint16_t* W,
                   const int32_t* anchor, int R, int B, int V, int r, int k, int P, int N,
                   int32_t* tok, int32_t* parent, int32_t* depth, double* score,
                   uint32_t* mask, int32_t* n_nodes, double* margin);

/* Survival product and the throughput-maximising prefix budget. */
int orc_schedule_budget(const float* conf, int R, int gamma, const double* cost,
                        float* survival, int32_t* budget, double* expected,
                        int32_t* total_tokens, int32_t* m_star);

/* The production scheduler: capacity K = the global argmax over m of
 * E'(m) / cost[R + m] on the survivals of conf_stale (the confidences of two
 * steps before), then the top K of the current survivals (all if fewer).
 * survival = the current products; capacity = K. */
int orc_schedule_dynamic(const float* conf, const float* conf_stale, int R, int gamma, const double* cost,
                         float* survival, int32_t* budget, double* expected, int32_t* total_tokens,
                         int32_t* capacity);

/* Ragged front-pack of the verify windows.  budget == NULL means the full
 * block (n_i = gamma).  Packed arrays need max(tiers[-1], R*(gamma+1)) slots.
 * A total above every tier is run uncaptured (tier = total,
 * ORC_FLAG_TIER_UNCAPTURED), or with strict != 0 reported as an overflow
 * (ORC_FLAG_TIER_OVERFLOW; the rows are packed the same way). */
int orc_pack_ragged(const int32_t* anchor, const int32_t* draft, const int32_t* budget,
                    int R, int gamma, const int32_t* tiers, int n_tiers, int strict,
                    int32_t* cu_seqlens, int32_t* packed_tok, int32_t* packed_req,
                    int32_t* packed_pos, int32_t* tier, int32_t* flags);

/* Verification over packed target logits [rows, V].  budget is only read in
 * cap-accept mode; logq/lse_q/L/U/W/r only in sample mode.  req_ids (may be
 * NULL) maps local request i to the global request id of the random counters.
 * margin [R, gamma+1] (may be NULL), one per decision: [i, p] the margin
 * |ln u - ln(p/q)| of the accept test of window row p, [i, gamma] that of the
 * final residual or bonus draw; INFINITY where no such decision was taken
 * (greedy decisions are exact: every entry INFINITY). */
int orc_verify(int mode, int decode, double temperature, uint64_t seed, uint64_t cycle,
               const int32_t* req_ids, const void* target, int dtT, const int32_t* cu_seqlens,
               const int32_t* anchor, const int32_t* draft, const int32_t* budget,
               const double* logq, const double* lse_q,
               const void* L, int dtL, const uint16_t* U, const uint16_t* W, int r,
               int R, int gamma, int V,
               int32_t* accept, int32_t* ceiling, int32_t* out_tok, int32_t* n_out,
               double* margin);

/* Greedy verification of a drafted tree: target is [R, N+1, V], one row per
 * tree slot.  out_tok holds B+1 slots per request. */
int orc_verify_tree(const void* target, int dtT, const int32_t* tok, const int32_t* parent,
                    const int32_t* n_nodes, int R, int N, int B, int V,
                    int32_t* accept, int32_t* out_tok, int32_t* n_out);

/* The confidence head's soft label 1 - TV(q, p) = sum_v min(q_v, p_v) for
 * every verified window row (label [R, gamma], -1 outside the window); q is
 * the draft's distribution at that position, p the target row's. */
int orc_tv_label(double temperature, const void* target, int dtT, const int32_t* cu_seqlens,
                 const int32_t* anchor, const int32_t* draft, const void* L, int dtL,
                 const uint16_t* U, const uint16_t* W, int r, int R, int gamma, int V, double* label);

/* Verify-cycle statistics: ceiling histogram per class [n_class, gamma+1],
 * per-position observed / accepted counts [n_class, gamma], equal-width
 * calibration bins of the confidences and their expected calibration error. */
int orc_observe(const float* conf, const int32_t* cu_seqlens, const int32_t* ceiling, const int32_t* cls,
                int R, int gamma, int n_class, int n_bins,
                int32_t* hist, int32_t* reached, int32_t* hits,
                int32_t* bin_n, int32_t* bin_hit, double* bin_conf, double* ece);

/* Fixed-threshold verify length: n_i = the longest prefix with every
 * confidence >= tau; total_tokens = R + sum n_i. */
int orc_schedule_threshold(const float* conf, int R, int gamma, float tau, int32_t* budget, int32_t* total_tokens);

/* Threshold sweep: per tau_k the verified drafts, the accepted drafts given
 * the whole-block ceilings (ceiling may be NULL: accepted = -1) and the
 * expected accepted drafts (exact sum of the survivals >= 2^-24). */
int orc_threshold_sweep(const float* conf, const int32_t* ceiling, int R, int gamma, const float* taus, int K,
                        int32_t* drafts, int32_t* accepted, double* expected);

/* RNN head: memo m_d = tanh(A m_{d-1} + U[y_{d-1}] + x_d), m_0 = 0, and
 * z_d = L_d + bf16(m_d) . W.  orc_rnn_memo gives the memo along a given
 * token sequence ([R, B, r] double); orc_draft_chain_rnn drafts with it
 * (outputs as orc_draft_chain).  A [r, r], X [R, B, r] bf16. */
int orc_rnn_memo(const uint16_t* A, const uint16_t* U, const uint16_t* X, const int32_t* anchor,
                 const int32_t* tokens, int R, int B, int r, double* memo);
int orc_draft_chain_rnn(const void* L, int dtL, const uint16_t* U, const uint16_t* W, const uint16_t* A,
                        const uint16_t* X, const int32_t* anchor, const int32_t* req_ids, int R, int B, int V, int r,
                        int decode, double temperature, uint64_t seed, uint64_t cycle,
                        int32_t* tokens, double* logq, double* lse, double* margin);

/* The RNN head's projection and decision for a given fp32 memo [R, B, r]:
 * z_d = L_d + bf16(memo_d) . W, then y_d, lse and logq as
 * orc_draft_chain_rnn forms them; margin[i, d-1] belongs to that position's
 * decision alone. */
int orc_rnn_project(const void* L, int dtL, const uint16_t* W, const float* memo, const int32_t* req_ids,
                    int R, int B, int V, int r, int decode, double temperature, uint64_t seed, uint64_t cycle,
                    int32_t* tokens, double* logq, double* lse, double* margin);

#ifdef __cplusplus
}
#endif
#endif
