/*
 * oracle.c - CPU oracle for the DSpark / PCTree speculative-decoding hot path.
 *
 * TEST INFRASTRUCTURE ONLY (see oracle.h): plain single-threaded loops that
 * follow each step of the method in the order the pages give it.  Nothing in
 * the CUDA library includes or calls this file.  Build with
 *     gcc -O2 -ffp-contract=off -fPIC -shared oracle.c -lm
 * so that every float expression is rounded exactly as written.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* Element access                                                       */
/* ------------------------------------------------------------------ */

/* bf16 is the upper half of an IEEE binary32. */
static float bf16_to_float(uint16_t h) {
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return f;
}

static float load_elem(const void* base, int dtype, size_t idx) {
    if (dtype == ORC_BF16) return bf16_to_float(((const uint16_t*)base)[idx]);
    return ((const float*)base)[idx];
}

/* ------------------------------------------------------------------ */
/* Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers:  */
/* as easy as 1, 2, 3", SC'11): ten rounds of the two-multiplier S-box,  */
/* with the Weyl key schedule between rounds.                            */
/* ------------------------------------------------------------------ */
void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
    const uint32_t mul0 = 0xD2511F53u, mul1 = 0xCD9E8D57u;
    const uint32_t weyl0 = 0x9E3779B9u, weyl1 = 0xBB67AE85u;
    uint32_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += weyl0;
            k1 += weyl1;
        }
        uint64_t p0 = (uint64_t)mul0 * x0;
        uint64_t p1 = (uint64_t)mul1 * x2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        uint32_t n0 = hi1 ^ x1 ^ k0;
        uint32_t n1 = lo1;
        uint32_t n2 = hi0 ^ x3 ^ k1;
        uint32_t n3 = lo0;
        x0 = n0; x1 = n1; x2 = n2; x3 = n3;
    }
    out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

/* Counter layout (a convention of this implementation; the pages only say
 * "Philox uniforms from the seed"):
 *   key     = (seed mod 2^32, seed >> 32)
 *   counter = (v >> 2, request, (stream << 16) | row, cycle mod 2^32)
 *   word    = v & 3 of the output block
 *   u       = (2 * (word >> 9) + 1) * 2^-24, an exact odd multiple of 2^-24
 *             strictly inside (0, 1). */
double orc_uniform(uint64_t seed, uint64_t cycle, int stream, uint32_t req, uint32_t row, uint32_t v) {
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t ctr[4] = {v >> 2, req, ((uint32_t)stream << 16) | row, (uint32_t)cycle};
    uint32_t out[4];
    orc_philox4x32_10(ctr, key, out);
    uint32_t word = out[v & 3u];
    return (double)(2u * (word >> 9) + 1u) / 16777216.0;
}

/* Categorical draw by the inverse CDF in index order (the pages leave the
 * sampler open; this is the plain textbook one): the smallest v with
 * w[0] + ... + w[v] > u S, S = sum of the nonnegative weights w, one uniform
 * u per draw.  *margin = the distance from u S to the nearer cumulative bound
 * around v, relative to S (how far u is from changing the draw). */
static int icdf_draw(const double* w, int V, double u, double* margin) {
    double S = 0.0;
    for (int v = 0; v < V; ++v) S += w[v];
    const double t = u * S;
    double c = 0.0;
    int last = -1;
    for (int v = 0; v < V; ++v) {
        if (!(w[v] > 0.0)) continue;
        last = v;
        const double c1 = c + w[v];
        if (c1 > t) {
            const double a = t - c, b = c1 - t;
            if (margin) *margin = (a < b ? a : b) / S;
            return v;
        }
        c = c1;
    }
    if (margin) *margin = 0.0;   /* u S at or above the rounded total: the last positive weight */
    return last < 0 ? 0 : last;
}

/* ------------------------------------------------------------------ */
/* Markov head: Markov(y) = U[y] . W, rank r  ([DSpark notes] sec. 4,    */
/* "Markov head"; [PCTree] z_d = L_d + Markov(y_{d-1})).                 */
/* ------------------------------------------------------------------ */

/* M[v] = sum_j U[prev, j] * W[j, v], accumulated in double.  Returns 0 when
 * every M[v] is exactly representable in fp32 (true for the grid-quantised
 * synthetic tables, whose partial sums are exact). */
static int markov_row(const uint16_t* U, const uint16_t* W, int prev, int r, int V, double* M) {
    int inexact = 0;
    for (int v = 0; v < V; ++v) M[v] = 0.0;
    for (int j = 0; j < r; ++j) {
        double u = (double)bf16_to_float(U[(size_t)prev * r + j]);
        if (u == 0.0) continue;
        const uint16_t* wrow = W + (size_t)j * V;
        for (int v = 0; v < V; ++v) M[v] += u * (double)bf16_to_float(wrow[v]);
    }
    for (int v = 0; v < V; ++v)
        if ((double)(float)M[v] != M[v]) inexact = 1;
    return inexact;
}

/* z_d[v] = L_d[v] + Markov(prev)[v], one fp32 addition per element. */
static void combine_logits(const void* L, int dtL, size_t row_off, const double* M, int V, float* z) {
    for (int v = 0; v < V; ++v) {
        float lv = load_elem(L, dtL, row_off + (size_t)v);
        float mv = (float)M[v];
        z[v] = lv + mv;
    }
}

/* argmax with the lowest id winning ties; *gap = best - second best. */
static int argmax_f32(const float* z, int V, double* gap) {
    int best = 0;
    for (int v = 1; v < V; ++v)
        if (z[v] > z[best]) best = v;
    double second = -INFINITY;
    for (int v = 0; v < V; ++v)
        if (v != best && (double)z[v] > second) second = (double)z[v];
    if (gap) *gap = (double)z[best] - second;
    return best;
}

/* log sum_v exp(x[v]) in double, max-shifted. */
static double logsumexp_scaled(const float* z, int V, double inv_t) {
    double m = -INFINITY;
    for (int v = 0; v < V; ++v)
        if ((double)z[v] * inv_t > m) m = (double)z[v] * inv_t;
    double s = 0.0;
    for (int v = 0; v < V; ++v) s += exp((double)z[v] * inv_t - m);
    return m + log(s);
}

/* ------------------------------------------------------------------ */
/* draft_chain                                                          */
/* ------------------------------------------------------------------ */
int orc_draft_chain(const void* L, int dtL, const uint16_t* U, const uint16_t* W,
                    const int32_t* anchor, const int32_t* req_ids, int R, int B, int V, int r,
                    int decode, double temperature, uint64_t seed, uint64_t cycle,
                    int32_t* tokens, double* logq, double* lse, double* margin) {
    int flags = 0;
    double* M = (double*)malloc(sizeof(double) * (size_t)V);
    double* wts = (double*)malloc(sizeof(double) * (size_t)V);
    float* z = (float*)malloc(sizeof(float) * (size_t)V);
    double inv_t = 1.0 / temperature;
    for (int i = 0; i < R; ++i) {
        uint32_t gid = req_ids ? (uint32_t)req_ids[i] : (uint32_t)i;
        int prev = anchor[i];                                   /* y_0: the anchor */
        for (int d = 1; d <= B; ++d) {
            /* z_d = L_d + Markov(y_{d-1}) */
            if (markov_row(U, W, prev, r, V, M)) flags |= ORC_FLAG_INEXACT_MARKOV;
            combine_logits(L, dtL, ((size_t)i * B + (size_t)(d - 1)) * V, M, V, z);
            size_t o = (size_t)i * B + (size_t)(d - 1);
            int y;
            double gap = 0.0;
            if (decode == ORC_GREEDY) {
                /* y_d = argmax_v z_d[v] */
                y = argmax_f32(z, V, &gap);
                if (logq) logq[o] = 0.0;
                if (lse) lse[o] = 0.0;
            } else {
                /* y_d ~ softmax(z_d / T): inverse CDF in vocabulary order,
                 * one uniform (stream 0, row d) */
                double zmax = -INFINITY;
                for (int v = 0; v < V; ++v)
                    if ((double)z[v] * inv_t > zmax) zmax = (double)z[v] * inv_t;
                for (int v = 0; v < V; ++v) wts[v] = exp((double)z[v] * inv_t - zmax);
                double u = orc_uniform(seed, cycle, ORC_STREAM_DRAFT, gid, (uint32_t)d, 0u);
                y = icdf_draw(wts, V, u, &gap);
                double l = logsumexp_scaled(z, V, inv_t);
                if (lse) lse[o] = l;
                if (logq) logq[o] = (double)z[y] * inv_t - l;     /* log q_d(y_d) */
            }
            tokens[o] = y;
            if (margin) margin[o] = gap;
            prev = y;
        }
    }
    free(M);
    free(wts);
    free(z);
    return flags;
}

/* ------------------------------------------------------------------ */
/* draft_tree (PCTree, [PCTree] section on tree drafting)               */
/* ------------------------------------------------------------------ */
typedef struct {
    int tok, parent, depth, creation;
    double score;
} tree_node;

typedef struct {
    double s;
    int slot, rank, tok, parent;
} tree_cand;

/* (s desc, parent slot asc, child rank asc) */
static int cand_before(const tree_cand* a, const tree_cand* b) {
    if (a->s != b->s) return a->s > b->s;
    if (a->slot != b->slot) return a->slot < b->slot;
    return a->rank < b->rank;
}

/* (s desc, depth asc, creation asc) */
static int node_before(const tree_node* a, const tree_node* b) {
    if (a->score != b->score) return a->score > b->score;
    if (a->depth != b->depth) return a->depth < b->depth;
    return a->creation < b->creation;
}

int orc_draft_tree(const void* L, int dtL, const uint16_t* U, const uint16_t* W,
                   const int32_t* anchor, int R, int B, int V, int r, int k, int P, int N,
                   int32_t* tok, int32_t* parent, int32_t* depth, double* score,
                   uint32_t* mask, int32_t* n_nodes, double* margin) {
    int flags = 0;
    int slots = N + 1;
    int words = (slots + 31) / 32;
    int pool_cap = 1 + P * B;
    double* M = (double*)malloc(sizeof(double) * (size_t)V);
    float* z = (float*)malloc(sizeof(float) * (size_t)V);
    tree_node* pool = (tree_node*)malloc(sizeof(tree_node) * (size_t)pool_cap);
    int* frontier = (int*)malloc(sizeof(int) * (size_t)P);
    int* next_frontier = (int*)malloc(sizeof(int) * (size_t)P);
    tree_cand* cand = (tree_cand*)malloc(sizeof(tree_cand) * (size_t)P * (size_t)k);
    int* top_id = (int*)malloc(sizeof(int) * (size_t)k);
    int* order = (int*)malloc(sizeof(int) * (size_t)pool_cap);
    int* out_slot = (int*)malloc(sizeof(int) * (size_t)pool_cap);

    for (int i = 0; i < R; ++i) {
        /* one margin per decision: [i, d-1] the prune boundary of level d,
         * [i, B] the top-N boundary, [i, B+1] the smallest score gap between
         * neighbours of the output ranking (their order); INFINITY where no
         * boundary was crossed */
        double* mg = margin ? margin + (size_t)i * (size_t)(B + 2) : NULL;
        if (mg)
            for (int q = 0; q < B + 2; ++q) mg[q] = INFINITY;
        int n_pool = 0;
        pool[n_pool++] = (tree_node){anchor[i], -1, 0, 0, 0.0};   /* root = anchor */
        int n_front = 1;
        frontier[0] = 0;
        for (int d = 1; d <= B; ++d) {
            int n_cand = 0;
            for (int slot = 0; slot < n_front; ++slot) {
                const tree_node* par = &pool[frontier[slot]];
                /* z_d(p) = L_d + Markov(p) for this frontier parent */
                if (markov_row(U, W, par->tok, r, V, M)) flags |= ORC_FLAG_INEXACT_MARKOV;
                combine_logits(L, dtL, ((size_t)i * B + (size_t)(d - 1)) * V, M, V, z);
                double l = logsumexp_scaled(z, V, 1.0);
                /* local top-k children by (z desc, id asc) */
                int kk = k < V ? k : V;
                int filled = 0;
                for (int v = 0; v < V; ++v) {
                    int pos = filled;
                    while (pos > 0 && z[v] > z[top_id[pos - 1]]) --pos;
                    if (pos >= kk) continue;
                    int last = filled < kk ? filled : kk - 1;
                    for (int q = last; q > pos; --q) top_id[q] = top_id[q - 1];
                    top_id[pos] = v;
                    if (filled < kk) ++filled;
                }
                for (int c = 0; c < filled; ++c) {
                    int v = top_id[c];
                    /* path score s(c) = s(p) + log pi(v | p) */
                    cand[n_cand++] = (tree_cand){par->score + ((double)z[v] - l), slot, c, v, frontier[slot]};
                }
            }
            /* per-level prune: keep the P best candidates */
            for (int a = 1; a < n_cand; ++a) {
                tree_cand t = cand[a];
                int b = a;
                while (b > 0 && cand_before(&t, &cand[b - 1])) {
                    cand[b] = cand[b - 1];
                    --b;
                }
                cand[b] = t;
            }
            int keep = n_cand < P ? n_cand : P;
            if (n_cand > keep && mg) mg[d - 1] = cand[keep - 1].s - cand[keep].s;
            for (int c = 0; c < keep; ++c) {
                pool[n_pool] = (tree_node){cand[c].tok, cand[c].parent, d, n_pool, cand[c].s};
                next_frontier[c] = n_pool;
                ++n_pool;
            }
            memcpy(frontier, next_frontier, sizeof(int) * (size_t)keep);
            n_front = keep;
        }
        /* global top-N over the pool (root excluded) */
        int n_order = 0;
        for (int p = 1; p < n_pool; ++p) {
            int b = n_order;
            while (b > 0 && node_before(&pool[p], &pool[order[b - 1]])) {
                order[b] = order[b - 1];
                --b;
            }
            order[b] = p;
            ++n_order;
        }
        int take = n_order < N ? n_order : N;
        if (n_order > take && mg) mg[B] = pool[order[take - 1]].score - pool[order[take]].score;
        for (int c = 1; c < take && mg; ++c) {
            double g = pool[order[c - 1]].score - pool[order[c]].score;
            if (g < mg[B + 1]) mg[B + 1] = g;
        }
        for (int p = 0; p < n_pool; ++p) out_slot[p] = -1;
        out_slot[0] = 0;
        size_t base = (size_t)i * slots;
        tok[base] = anchor[i];
        parent[base] = -1;
        depth[base] = 0;
        score[base] = 0.0;
        for (int c = 0; c < take; ++c) {
            const tree_node* nd = &pool[order[c]];
            out_slot[order[c]] = c + 1;
            tok[base + c + 1] = nd->tok;
            parent[base + c + 1] = out_slot[nd->parent];   /* ancestors rank earlier */
            if (out_slot[nd->parent] < 0) flags |= 1;      /* would break the tree */
            depth[base + c + 1] = nd->depth;
            score[base + c + 1] = nd->score;
        }
        for (int c = take + 1; c < slots; ++c) {
            tok[base + c] = -1;
            parent[base + c] = -1;
            depth[base + c] = -1;
            score[base + c] = 0.0;
        }
        n_nodes[i] = take + 1;
        /* tree-causal mask: row c sees itself and its ancestors */
        for (int c = 0; c < slots; ++c) {
            uint32_t* row = mask + (base + (size_t)c) * words;
            for (int w = 0; w < words; ++w) row[w] = 0u;
            if (c > take) continue;
            for (int a = c; a >= 0; a = parent[base + a]) row[a / 32] |= 1u << (a % 32);
        }
    }
    free(M); free(z); free(pool); free(frontier); free(next_frontier);
    free(cand); free(top_id); free(order); free(out_slot);
    return flags;
}

/* ------------------------------------------------------------------ */
/* schedule_budget ([DSpark notes] sec. 5.1 survival, 5.2 scheduler)    */
/* ------------------------------------------------------------------ */
typedef struct {
    float s;
    int req, pos;
} surv_entry;

/* (S desc, request asc, position asc) */
static int surv_before(const surv_entry* a, const surv_entry* b) {
    if (a->s != b->s) return a->s > b->s;
    if (a->req != b->req) return a->req < b->req;
    return a->pos < b->pos;
}

static int surv_cmp(const void* pa, const void* pb) {
    const surv_entry* a = (const surv_entry*)pa;
    const surv_entry* b = (const surv_entry*)pb;
    if (surv_before(a, b)) return -1;
    if (surv_before(b, a)) return 1;
    return 0;
}

int orc_schedule_budget(const float* conf, int R, int gamma, const double* cost,
                        float* survival, int32_t* budget, double* expected,
                        int32_t* total_tokens, int32_t* m_star) {
    /* Survivals below 2^-18 are never worth verifying at the tables used and
     * are left out of the ranking; what remains sums exactly in fp64. */
    const float floor_s = 1.0f / 262144.0f;
    surv_entry* e = (surv_entry*)malloc(sizeof(surv_entry) * (size_t)R * (size_t)gamma + 1);
    int n = 0;
    for (int i = 0; i < R; ++i) {
        float s = 1.0f;
        for (int k = 1; k <= gamma; ++k) {
            s = s * conf[(size_t)i * gamma + (size_t)(k - 1)];   /* S_{i,k} = S_{i,k-1} c_{i,k} */
            survival[(size_t)i * gamma + (size_t)(k - 1)] = s;
            if (s >= floor_s) e[n++] = (surv_entry){s, i, k};
        }
        budget[i] = 0;
    }
    qsort(e, (size_t)n, sizeof(surv_entry), surv_cmp);
    /* Greedy over the ranked survivals: every request always sends its root
     * token and always gets one token back, so E(m) = R + sum of the top m
     * survivals and N(m) = R + m verify tokens; add the next survival while
     * E/cost strictly improves and stop at the first one that does not. */
    double E = (double)R;
    double f = E / cost[R];
    int m = 0;
    while (m < n) {
        double E_next = E + (double)e[m].s;
        double f_next = E_next / cost[R + m + 1];
        if (!(f_next > f)) break;
        E = E_next;
        f = f_next;
        ++m;
    }
    for (int c = 0; c < m; ++c) budget[e[c].req] += 1;
    *expected = E;
    *total_tokens = R + m;
    if (m_star) *m_star = m;
    free(e);
    return 0;
}

/* ------------------------------------------------------------------ */
/* schedule_dynamic ([DSpark notes] sec. 9.2: the production scheduler)  */
/* ------------------------------------------------------------------ */
/* Ranked survivals of conf (the S_{i,k} products, those >= 2^-18) into e,
 * written to surv when not NULL; returns how many. */
static int ranked_survivals(const float* conf, int R, int gamma, float* surv, surv_entry* e) {
    const float floor_s = 1.0f / 262144.0f;
    int n = 0;
    for (int i = 0; i < R; ++i) {
        float s = 1.0f;
        for (int k = 1; k <= gamma; ++k) {
            s = s * conf[(size_t)i * gamma + (size_t)(k - 1)];
            if (surv) surv[(size_t)i * gamma + (size_t)(k - 1)] = s;
            if (s >= floor_s) e[n++] = (surv_entry){s, i, k};
        }
    }
    qsort(e, (size_t)n, sizeof(surv_entry), surv_cmp);
    return n;
}

int orc_schedule_dynamic(const float* conf, const float* conf_stale, int R, int gamma, const double* cost,
                         float* survival, int32_t* budget, double* expected, int32_t* total_tokens,
                         int32_t* capacity) {
    surv_entry* e = (surv_entry*)malloc(sizeof(surv_entry) * (size_t)R * (size_t)gamma + 1);
    /* 1. the verify capacity K from the confidences of two steps before: the
     *    global argmax over every m of E'(m) / cost[R + m], no early stop
     *    (the table may step), the smallest m on ties */
    int n_stale = ranked_survivals(conf_stale, R, gamma, NULL, e);
    double E = (double)R;
    double best = E / cost[R];
    int K = 0;
    for (int m = 1; m <= n_stale; ++m) {
        E += (double)e[m - 1].s;
        double f = E / cost[R + m];
        if (f > best) {
            best = f;
            K = m;
        }
    }
    /* 2. this step's candidates ranked by their current survivals; the top K
     *    (all of them if fewer) are verified */
    int n_now = ranked_survivals(conf, R, gamma, survival, e);
    int take = K < n_now ? K : n_now;
    for (int i = 0; i < R; ++i) budget[i] = 0;
    double En = (double)R;
    for (int c = 0; c < take; ++c) {
        budget[e[c].req] += 1;
        En += (double)e[c].s;
    }
    *expected = En;
    *total_tokens = R + take;
    *capacity = K;
    free(e);
    return 0;
}

/* ------------------------------------------------------------------ */
/* pack_ragged ([SGLang] "ragged verify")                               */
/* ------------------------------------------------------------------ */
int orc_pack_ragged(const int32_t* anchor, const int32_t* draft, const int32_t* budget,
                    int R, int gamma, const int32_t* tiers, int n_tiers, int strict,
                    int32_t* cu_seqlens, int32_t* packed_tok, int32_t* packed_req,
                    int32_t* packed_pos, int32_t* tier, int32_t* flags) {
    *flags = 0;
    cu_seqlens[0] = 0;
    for (int i = 0; i < R; ++i) {
        int n = budget ? budget[i] : gamma;
        if (n < 0 || n > gamma) return -1;
        cu_seqlens[i + 1] = cu_seqlens[i] + n + 1;                /* root + n drafts */
    }
    int total = cu_seqlens[R];
    int t = -1;
    for (int q = 0; q < n_tiers; ++q)
        if (tiers[q] >= total && (t < 0 || tiers[q] < t)) t = tiers[q];
    if (t < 0) {
        t = total;                                                /* above every captured tier */
        *flags |= strict ? ORC_FLAG_TIER_OVERFLOW : ORC_FLAG_TIER_UNCAPTURED;
    }
    *tier = t;
    for (int i = 0; i < R; ++i) {
        int n = cu_seqlens[i + 1] - cu_seqlens[i] - 1;
        for (int p = 0; p <= n; ++p) {
            int row = cu_seqlens[i] + p;
            packed_tok[row] = p == 0 ? anchor[i] : draft[(size_t)i * gamma + (size_t)(p - 1)];
            packed_req[row] = i;
            packed_pos[row] = p;
        }
    }
    for (int row = total; row < t; ++row) {
        packed_tok[row] = -1;
        packed_req[row] = -1;
        packed_pos[row] = -1;
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* verify ([DSpark notes] sec. 1; [SGLang] "three verify modes")        */
/* ------------------------------------------------------------------ */

static int row_argmax(const void* T, int dtT, size_t row, int V) {
    int best = 0;
    float bv = load_elem(T, dtT, row * (size_t)V);
    for (int v = 1; v < V; ++v) {
        float x = load_elem(T, dtT, row * (size_t)V + (size_t)v);
        if (x > bv) {
            bv = x;
            best = v;
        }
    }
    return best;
}

static double row_lse(const void* T, int dtT, size_t row, int V, double inv_t) {
    double m = -INFINITY;
    for (int v = 0; v < V; ++v) {
        double x = (double)load_elem(T, dtT, row * (size_t)V + (size_t)v) * inv_t;
        if (x > m) m = x;
    }
    double s = 0.0;
    for (int v = 0; v < V; ++v) s += exp((double)load_elem(T, dtT, row * (size_t)V + (size_t)v) * inv_t - m);
    return m + log(s);
}

int orc_verify(int mode, int decode, double temperature, uint64_t seed, uint64_t cycle,
               const int32_t* req_ids, const void* target, int dtT, const int32_t* cu_seqlens,
               const int32_t* anchor, const int32_t* draft, const int32_t* budget,
               const double* logq, const double* lse_q,
               const void* L, int dtL, const uint16_t* U, const uint16_t* W, int r,
               int R, int gamma, int V,
               int32_t* accept, int32_t* ceiling, int32_t* out_tok, int32_t* n_out,
               double* margin) {
    int flags = 0;
    double inv_t = 1.0 / temperature;
    double* M = (double*)malloc(sizeof(double) * (size_t)V);
    double* wts = (double*)malloc(sizeof(double) * (size_t)V);
    float* z = (float*)malloc(sizeof(float) * (size_t)V);
    for (int i = 0; i < R; ++i) {
        uint32_t gid = req_ids ? (uint32_t)req_ids[i] : (uint32_t)i;
        size_t row0 = (size_t)cu_seqlens[i];
        int w = cu_seqlens[i + 1] - cu_seqlens[i] - 1;           /* drafts in the window */
        int cap = (mode == ORC_CAP_ACCEPT) ? budget[i] : w;       /* drafts that may commit */
        if (cap > w) cap = w;
        const int32_t* y = draft + (size_t)i * gamma;             /* y[p] = y_{p+1} */
        /* one margin per decision: [i, p] the accept test of window row p,
         * [i, gamma] the final draw (residual or bonus); INFINITY where no
         * such decision was taken (and for every greedy decision) */
        double* mg = margin ? margin + (size_t)i * (size_t)(gamma + 1) : NULL;
        if (mg)
            for (int p = 0; p <= gamma; ++p) mg[p] = INFINITY;
        int A, a, last;
        if (decode == ORC_GREEDY) {
            /* accept while the draft equals the target's argmax; the first
             * mismatch is replaced by the target token there (bonus) */
            A = w;
            for (int p = 0; p < w; ++p) {
                if (y[p] != row_argmax(target, dtT, row0 + (size_t)p, V)) {
                    A = p;
                    break;
                }
            }
            a = A < cap ? A : cap;
            last = row_argmax(target, dtT, row0 + (size_t)a, V);
        } else {
            /* left to right: accept y_{p+1} iff u < p(y)/q(y).  In cap-accept
             * mode the tests run on past the commit window (the ceiling A);
             * rows inside the window use the same uniforms as compact. */
            A = w;
            for (int p = 0; p < w; ++p) {
                double lp = (double)load_elem(target, dtT, (row0 + (size_t)p) * (size_t)V + (size_t)y[p]) * inv_t
                            - row_lse(target, dtT, row0 + (size_t)p, V, inv_t);
                double lq = logq[(size_t)i * gamma + (size_t)p];
                double lu = log(orc_uniform(seed, cycle, ORC_STREAM_ACCEPT, gid, (uint32_t)p, 0u));
                if (mg) mg[p] = fabs(lu - (lp - lq));
                if (!(lu < lp - lq)) {
                    A = p;
                    break;
                }
            }
            a = A < cap ? A : cap;
            int row = a;
            double lse_p = row_lse(target, dtT, row0 + (size_t)row, V, inv_t);
            double gap = INFINITY;
            if (A < cap) {
                /* rejected at row a = A: resample from max(0, p - q), with q
                 * recomputed from the Markov head at that position (inverse
                 * CDF, one uniform: stream 2, row a) */
                int prev = row == 0 ? anchor[i] : y[row - 1];
                if (markov_row(U, W, prev, r, V, M)) flags |= ORC_FLAG_INEXACT_MARKOV;
                combine_logits(L, dtL, ((size_t)i * gamma + (size_t)row) * V, M, V, z);
                double lq_row = lse_q[(size_t)i * gamma + (size_t)row];
                for (int v = 0; v < V; ++v) {
                    double pv = exp((double)load_elem(target, dtT, (row0 + (size_t)row) * (size_t)V + (size_t)v) * inv_t - lse_p);
                    double qv = exp((double)z[v] * inv_t - lq_row);
                    double wv = pv - qv;
                    wts[v] = wv > 0.0 ? wv : 0.0;
                }
                last = icdf_draw(wts, V, orc_uniform(seed, cycle, ORC_STREAM_RESID, gid, (uint32_t)row, 0u), &gap);
            } else {
                /* every committed draft accepted: bonus token ~ p at row a
                 * (inverse CDF, stream 3, row a) */
                for (int v = 0; v < V; ++v)
                    wts[v] = exp((double)load_elem(target, dtT, (row0 + (size_t)row) * (size_t)V + (size_t)v) * inv_t - lse_p);
                last = icdf_draw(wts, V, orc_uniform(seed, cycle, ORC_STREAM_BONUS, gid, (uint32_t)row, 0u), &gap);
            }
            if (mg) mg[gamma] = gap;
        }
        size_t ob = (size_t)i * (size_t)(gamma + 1);
        for (int p = 0; p < a; ++p) out_tok[ob + (size_t)p] = y[p];
        out_tok[ob + (size_t)a] = last;
        for (int p = a + 1; p <= gamma; ++p) out_tok[ob + (size_t)p] = -1;
        accept[i] = a;
        n_out[i] = a + 1;
        if (ceiling) ceiling[i] = A;
    }
    free(M);
    free(wts);
    free(z);
    return flags;
}

/* ------------------------------------------------------------------ */
/* verify_tree: greedy longest accepted root path ([PCTree])            */
/* ------------------------------------------------------------------ */
int orc_verify_tree(const void* target, int dtT, const int32_t* tok, const int32_t* parent,
                    const int32_t* n_nodes, int R, int N, int B, int V,
                    int32_t* accept, int32_t* out_tok, int32_t* n_out) {
    int slots = N + 1;
    for (int i = 0; i < R; ++i) {
        size_t base = (size_t)i * slots;
        int cur = 0, a = 0;
        size_t ob = (size_t)i * (size_t)(B + 1);
        for (;;) {
            int t = row_argmax(target, dtT, base + (size_t)cur, V);
            int next = -1;
            for (int c = 1; c < n_nodes[i]; ++c)
                if (parent[base + c] == cur && tok[base + c] == t) {
                    next = c;
                    break;
                }
            if (next < 0 || a >= B) {
                out_tok[ob + (size_t)a] = t;                      /* bonus */
                break;
            }
            out_tok[ob + (size_t)a] = t;
            ++a;
            cur = next;
        }
        for (int p = a + 1; p <= B; ++p) out_tok[ob + (size_t)p] = -1;
        accept[i] = a;
        n_out[i] = a + 1;
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* Observability: the confidence head's soft label and the per-cycle    */
/* statistics of verification ([DSpark notes] sec. 5.1, sec. 8.1;        */
/* [SGLang] "observability").                                            */
/* ------------------------------------------------------------------ */

/* label[i, p] = sum_v min(q_v, p_v) = 1 - TV(q, p) for window row p < w_i,
 * the chance that one token drafted from q survives the accept test against
 * p ([DSpark notes] sec. 5.1: the soft acceptance label).  q is the draft's
 * distribution at position p+1, softmax((L[i, p] + Markov(y_p)) / T) with
 * y_0 the anchor, its log-sum-exp computed here in double; p is softmax of
 * target row cu[i] + p over T.  Rows outside the window get -1. */
int orc_tv_label(double temperature, const void* target, int dtT, const int32_t* cu_seqlens,
                 const int32_t* anchor, const int32_t* draft, const void* L, int dtL,
                 const uint16_t* U, const uint16_t* W, int r, int R, int gamma, int V, double* label) {
    int flags = 0;
    double inv_t = 1.0 / temperature;
    double* M = (double*)malloc(sizeof(double) * (size_t)V);
    float* z = (float*)malloc(sizeof(float) * (size_t)V);
    for (int i = 0; i < R; ++i) {
        int w = cu_seqlens[i + 1] - cu_seqlens[i] - 1;
        for (int p = 0; p < gamma; ++p) {
            double* out = label + (size_t)i * gamma + (size_t)p;
            if (p >= w) {
                *out = -1.0;
                continue;
            }
            int prev = p == 0 ? anchor[i] : draft[(size_t)i * gamma + (size_t)(p - 1)];
            if (markov_row(U, W, prev, r, V, M)) flags |= ORC_FLAG_INEXACT_MARKOV;
            combine_logits(L, dtL, ((size_t)i * gamma + (size_t)p) * V, M, V, z);
            double lq = logsumexp_scaled(z, V, inv_t);
            size_t trow = (size_t)cu_seqlens[i] + (size_t)p;
            double lp = row_lse(target, dtT, trow, V, inv_t);
            double s = 0.0;
            for (int v = 0; v < V; ++v) {
                double qv = exp((double)z[v] * inv_t - lq);
                double pv = exp((double)load_elem(target, dtT, trow * (size_t)V + (size_t)v) * inv_t - lp);
                s += qv < pv ? qv : pv;
            }
            *out = s;
        }
    }
    free(M);
    free(z);
    return flags;
}

/* Statistics of one verify cycle.  Position d = 1..gamma of request i is
 * observed when every earlier draft was accepted and d was verified:
 * d <= min(ceiling_i + 1, w_i); its outcome is hit = (d <= ceiling_i)
 * ([DSpark notes] sec. 8.1 counts position d only where 1..d-1 were all
 * accepted).  ceiling_i is the acceptance count of the whole verified window
 * (cap-accept's ceiling; in the other modes the accepted count).
 *   hist[c, k]      requests of class c whose ceiling is k (k = 0..gamma)
 *   reached[c, d-1] observed positions d of class c; hits[c, d-1] their hits
 *   calibration: confidence c clamped to [0, 1] (NaN as 0) falls in bin
 *   floor(c * n_bins) (fp32 product), the top bin taking c = 1;
 *   bin_n, bin_hit count observations and hits, bin_conf sums c;
 *   ece = sum_b |bin_hit_b - bin_conf_b| / N, N = sum_b bin_n_b (0 if N = 0),
 *   the expected calibration error with equal-width bins.
 * Returns -1 when a class id is out of range, else 0. */
int orc_observe(const float* conf, const int32_t* cu_seqlens, const int32_t* ceiling, const int32_t* cls,
                int R, int gamma, int n_class, int n_bins,
                int32_t* hist, int32_t* reached, int32_t* hits,
                int32_t* bin_n, int32_t* bin_hit, double* bin_conf, double* ece) {
    for (int k = 0; k < n_class * (gamma + 1); ++k) hist[k] = 0;
    for (int k = 0; k < n_class * gamma; ++k) reached[k] = hits[k] = 0;
    for (int b = 0; b < n_bins; ++b) {
        bin_n[b] = bin_hit[b] = 0;
        bin_conf[b] = 0.0;
    }
    for (int i = 0; i < R; ++i) {
        int c = cls[i];
        if (c < 0 || c >= n_class) return -1;
        int w = cu_seqlens[i + 1] - cu_seqlens[i] - 1;
        int A = ceiling[i];
        hist[(size_t)c * (gamma + 1) + (size_t)A] += 1;
        int last = A + 1 < w ? A + 1 : w;
        for (int d = 1; d <= last; ++d) {
            int hit = d <= A;
            reached[(size_t)c * gamma + (size_t)(d - 1)] += 1;
            hits[(size_t)c * gamma + (size_t)(d - 1)] += hit;
            float x = conf[(size_t)i * gamma + (size_t)(d - 1)];
            if (!(x > 0.0f)) x = 0.0f;
            if (x > 1.0f) x = 1.0f;
            float scaled = x * (float)n_bins;
            int b = (int)floorf(scaled);
            if (b > n_bins - 1) b = n_bins - 1;
            bin_n[b] += 1;
            bin_hit[b] += hit;
            bin_conf[b] += (double)x;
        }
    }
    long n = 0;
    double e = 0.0;
    for (int b = 0; b < n_bins; ++b) {
        n += bin_n[b];
        e += fabs((double)bin_hit[b] - bin_conf[b]);
    }
    *ece = n > 0 ? e / (double)n : 0.0;
    return 0;
}

/* ------------------------------------------------------------------ */
/* Fixed-threshold verify length and the threshold sweep                */
/* ([DSpark notes] sec. 5.2: the conventional rule puts a fixed         */
/* threshold on the confidences; sec. 8.3, Fig. 5: sweeping it,         */
/* threshold 0 = verify the whole block)                                */
/* ------------------------------------------------------------------ */

/* n_i = the longest prefix of request i whose every confidence is >= tau
 * (fp32 comparison; a NaN confidence ends the prefix). */
static int threshold_len(const float* c, int gamma, float tau) {
    int n = 0;
    while (n < gamma && c[n] >= tau) ++n;
    return n;
}

int orc_schedule_threshold(const float* conf, int R, int gamma, float tau, int32_t* budget, int32_t* total_tokens) {
    int32_t total = R;   /* every request sends its root token */
    for (int i = 0; i < R; ++i) {
        budget[i] = threshold_len(conf + (size_t)i * gamma, gamma, tau);
        total += budget[i];
    }
    *total_tokens = total;
    return 0;
}

/* For every tau_k: drafts[k] = sum_i n_i(tau_k) verified drafts;
 * accepted[k] = sum_i min(ceiling_i, n_i) (ceiling = what verifying the whole
 * block accepts; -1 when ceiling is NULL); expected[k] = sum_i sum_{d <= n_i}
 * S_{i,d}, the expected accepted drafts, with S_{i,d} the fp32 survival
 * products.  The sum is exact: each S >= 2^-24 is a whole multiple of 2^-47
 * and is added as an integer count of 2^-48; smaller survivals count 0. */
int orc_threshold_sweep(const float* conf, const int32_t* ceiling, int R, int gamma, const float* taus, int K,
                        int32_t* drafts, int32_t* accepted, double* expected) {
    const float tiny = 1.0f / 16777216.0f;   /* 2^-24 */
    for (int k = 0; k < K; ++k) {
        int32_t nd = 0, na = 0;
        int64_t units = 0;                    /* multiples of 2^-48 */
        for (int i = 0; i < R; ++i) {
            const float* c = conf + (size_t)i * gamma;
            int n = threshold_len(c, gamma, taus[k]);
            float s = 1.0f;
            for (int d = 0; d < n; ++d) {
                s = s * c[d];
                if (s >= tiny) units += (int64_t)ldexp((double)s, 48);
            }
            nd += n;
            if (ceiling) na += ceiling[i] < n ? ceiling[i] : n;
        }
        drafts[k] = nd;
        accepted[k] = ceiling ? na : -1;
        expected[k] = ldexp((double)units, -48);
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* RNN head ([DSpark notes] sec. 4, "RNN head": a memo that carries the */
/* whole draft so far, updated once per step from the previous memo,    */
/* the previous word and the current backbone state).  The update's    */
/* formula is not legible on the page; the reading taken here:          */
/*   m_0 = 0,  m_d = tanh(A m_{d-1} + U[y_{d-1}] + x_d)                 */
/*   z_d = L_d + bf16(m_d) . W                                          */
/* with U the Markov head's token table (the previous word's input),    */
/* x_d the backbone state at position d projected to the memo's size r  */
/* (an input), and the memo entering the vocabulary projection in bf16  */
/* like U does.  With A = 0 and x = 0 this is the Markov head on the    */
/* table bf16(tanh(U)).                                                 */
/* ------------------------------------------------------------------ */

/* IEEE round-to-nearest-even of a binary32 to its upper 16 bits. */
static uint16_t float_to_bf16(float f) {
    uint32_t b;
    memcpy(&b, &f, sizeof b);
    if ((b & 0x7F800000u) == 0x7F800000u && (b & 0x007FFFFFu)) return (uint16_t)((b >> 16) | 0x40u);   /* NaN */
    b += 0x7FFFu + ((b >> 16) & 1u);
    return (uint16_t)(b >> 16);
}

/* m_out = tanh(A m_prev + U[prev] + x), all in double; A is [r, r] row-major
 * (output index first). */
static void rnn_update(const uint16_t* A, const uint16_t* U, const uint16_t* x, int prev, int r,
                       const double* m_prev, double* m_out) {
    for (int j = 0; j < r; ++j) {
        double v = 0.0;
        for (int k = 0; k < r; ++k) v += (double)bf16_to_float(A[(size_t)j * r + (size_t)k]) * m_prev[k];
        v += (double)bf16_to_float(U[(size_t)prev * r + (size_t)j]) + (double)bf16_to_float(x[j]);
        m_out[j] = tanh(v);
    }
}

/* M[v] = sum_j bf16(m_j) W[j, v] in double. */
static void memo_times_w(const double* m, const uint16_t* W, int r, int V, double* M) {
    for (int v = 0; v < V; ++v) M[v] = 0.0;
    for (int j = 0; j < r; ++j) {
        double a = (double)bf16_to_float(float_to_bf16((float)m[j]));
        if (a == 0.0) continue;
        const uint16_t* wrow = W + (size_t)j * V;
        for (int v = 0; v < V; ++v) M[v] += a * (double)bf16_to_float(wrow[v]);
    }
}

/* The memo trajectory along a given token sequence: memo[i, d-1, :] = m_d
 * for d = 1..B (y_0 = anchor[i], y_d = tokens[i, d-1]). */
int orc_rnn_memo(const uint16_t* A, const uint16_t* U, const uint16_t* X, const int32_t* anchor,
                 const int32_t* tokens, int R, int B, int r, double* memo) {
    double* m = (double*)calloc((size_t)r, sizeof(double));
    for (int i = 0; i < R; ++i) {
        for (int j = 0; j < r; ++j) m[j] = 0.0;
        for (int d = 1; d <= B; ++d) {
            int prev = d == 1 ? anchor[i] : tokens[(size_t)i * B + (size_t)(d - 2)];
            double* out = memo + ((size_t)i * B + (size_t)(d - 1)) * r;
            rnn_update(A, U, X + ((size_t)i * B + (size_t)(d - 1)) * r, prev, r, m, out);
            memcpy(m, out, sizeof(double) * (size_t)r);
        }
    }
    free(m);
    return 0;
}

/* The chain draft with the RNN head: as orc_draft_chain, with z_d formed
 * from the memo.  X is [R, B, r] bf16, A [r, r] bf16. */
int orc_draft_chain_rnn(const void* L, int dtL, const uint16_t* U, const uint16_t* W, const uint16_t* A,
                        const uint16_t* X, const int32_t* anchor, const int32_t* req_ids, int R, int B, int V, int r,
                        int decode, double temperature, uint64_t seed, uint64_t cycle,
                        int32_t* tokens, double* logq, double* lse, double* margin) {
    double* M = (double*)malloc(sizeof(double) * (size_t)V);
    double* wts = (double*)malloc(sizeof(double) * (size_t)V);
    float* z = (float*)malloc(sizeof(float) * (size_t)V);
    double* m = (double*)malloc(sizeof(double) * (size_t)r);
    double* m_next = (double*)malloc(sizeof(double) * (size_t)r);
    double inv_t = 1.0 / temperature;
    for (int i = 0; i < R; ++i) {
        uint32_t gid = req_ids ? (uint32_t)req_ids[i] : (uint32_t)i;
        int prev = anchor[i];
        for (int j = 0; j < r; ++j) m[j] = 0.0;
        for (int d = 1; d <= B; ++d) {
            size_t o = (size_t)i * B + (size_t)(d - 1);
            rnn_update(A, U, X + o * (size_t)r, prev, r, m, m_next);
            memcpy(m, m_next, sizeof(double) * (size_t)r);
            memo_times_w(m, W, r, V, M);
            combine_logits(L, dtL, o * V, M, V, z);
            int y;
            double gap = 0.0;
            if (decode == ORC_GREEDY) {
                y = argmax_f32(z, V, &gap);
                if (logq) logq[o] = 0.0;
                if (lse) lse[o] = 0.0;
            } else {
                double zmax = -INFINITY;
                for (int v = 0; v < V; ++v)
                    if ((double)z[v] * inv_t > zmax) zmax = (double)z[v] * inv_t;
                for (int v = 0; v < V; ++v) wts[v] = exp((double)z[v] * inv_t - zmax);
                double u = orc_uniform(seed, cycle, ORC_STREAM_DRAFT, gid, (uint32_t)d, 0u);
                y = icdf_draw(wts, V, u, &gap);
                double l = logsumexp_scaled(z, V, inv_t);
                if (lse) lse[o] = l;
                if (logq) logq[o] = (double)z[y] * inv_t - l;
            }
            tokens[o] = y;
            if (margin) margin[o] = gap;
            prev = y;
        }
    }
    free(M);
    free(wts);
    free(z);
    free(m);
    free(m_next);
    return 0;
}

/* The RNN head's projection and decision at every position for a memo that
 * is given (fp32 [R, B, r], for instance the trajectory another
 * implementation formed): z_d = L_d + bf16(memo_d) . W with the memo rounded
 * to bf16 as in orc_draft_chain_rnn, then y_d, lse and logq exactly as there
 * (greedy argmax, or the inverse-CDF draw of softmax(z_d / T) with the
 * uniform of stream 0, row d).  Each position's decision depends on its own
 * memo row only, so margin[i, d-1] is the margin of that one decision. */
int orc_rnn_project(const void* L, int dtL, const uint16_t* W, const float* memo, const int32_t* req_ids,
                    int R, int B, int V, int r, int decode, double temperature, uint64_t seed, uint64_t cycle,
                    int32_t* tokens, double* logq, double* lse, double* margin) {
    double* M = (double*)malloc(sizeof(double) * (size_t)V);
    double* wts = (double*)malloc(sizeof(double) * (size_t)V);
    float* z = (float*)malloc(sizeof(float) * (size_t)V);
    double* m = (double*)malloc(sizeof(double) * (size_t)r);
    double inv_t = 1.0 / temperature;
    for (int i = 0; i < R; ++i) {
        uint32_t gid = req_ids ? (uint32_t)req_ids[i] : (uint32_t)i;
        for (int d = 1; d <= B; ++d) {
            size_t o = (size_t)i * B + (size_t)(d - 1);
            for (int j = 0; j < r; ++j) m[j] = (double)memo[o * (size_t)r + (size_t)j];
            memo_times_w(m, W, r, V, M);
            combine_logits(L, dtL, o * V, M, V, z);
            int y;
            double gap = 0.0;
            if (decode == ORC_GREEDY) {
                y = argmax_f32(z, V, &gap);
                if (logq) logq[o] = 0.0;
                if (lse) lse[o] = 0.0;
            } else {
                double zmax = -INFINITY;
                for (int v = 0; v < V; ++v)
                    if ((double)z[v] * inv_t > zmax) zmax = (double)z[v] * inv_t;
                for (int v = 0; v < V; ++v) wts[v] = exp((double)z[v] * inv_t - zmax);
                double u = orc_uniform(seed, cycle, ORC_STREAM_DRAFT, gid, (uint32_t)d, 0u);
                y = icdf_draw(wts, V, u, &gap);
                double l = logsumexp_scaled(z, V, inv_t);
                if (lse) lse[o] = l;
                if (logq) logq[o] = (double)z[y] * inv_t - l;
            }
            tokens[o] = y;
            if (margin) margin[o] = gap;
        }
    }
    free(M);
    free(wts);
    free(z);
    free(m);
    return 0;
}
