// markov_gemm.cu - the Markov-head projection on the 5th-generation tensor
// cores, with the vocab-wide reductions fused into the epilogue.
//
// One launch computes, for a set of GEMM rows m (requests, or PCTree
// (request, frontier slot) pairs), the logits
//     z[m, v] = L[row(m), v] + (U[tok(m)] . W)[v]          v in [0, V)
// and reduces them over the vocabulary without writing z anywhere:
//   MODE_CHAIN_GREEDY  argmax_v z                       (DSpark notes sec. 4)
//   MODE_CHAIN_SAMPLE  per 16-column block: max of z / T and the sum of
//                      exp(z / T - max) (the records an inverse-CDF draw
//                      walks; the draw itself is select.cu's)
//   MODE_TREE          the same block records of z (PCTree frontier rows;
//                      the top-k children come from select.cu)
//   MODE_RESID         per 16-column block: the sum of max(0, p - q) at a
//                      rejected position
//   MODE_ABSMAX        max_v |U[m] . W[:, v]| for m = 0..V-1, no L (the
//                      per-token bound of the pruned greedy chain)
//   MODE_QLSE          log-sum-exp of z / T of listed (request, position)
//                      rows, one partial (max, sum) per row, CTA and group
//   MODE_TVMIN         sum_v min(q_v, p_v) of listed rows (the soft label
//                      1 - TV, DSpark notes sec. 5.1), one partial sum per
//                      row, CTA and column group; MODE_TVMIN_B16 / _B32 are
//                      the same for bf16 L and bf16 / fp32 target rows with
//                      a tile's loads issued before its accumulator is read
//   MODE_TREE_LSE      PCTree level with the bound-pruned children: only the
//                      log-sum-exp of each frontier row, one partial (max,
//                      sum) per row and CTA (tree_pruned.cu scores the
//                      children)
//
// Data path (one CTA = 128 GEMM rows x a round-robin set of 128-wide vocab
// tiles, K = r):
//   * all threads gather the 128 rows U[tok(m)] (bf16, K-major) into shared
//     memory once, in the 128-byte swizzled layout tcgen05 reads;
//   * warp 0 streams W tiles [r x 128] as two 64-id boxes per 64-row K block
//     (MN-major, TMA 2-D, 128-byte swizzle, L2 evict_last) through a ring of
//     tile slots; warp 2 streams the matching L boxes [rows x 64] (TMA 3-D,
//     evict_first) through their own ring (modes that stage L);
//   * warp 1 first copies A into tensor memory (tcgen05.cp, r/16 blocks of
//     128 rows x 16 bf16), then issues r/16 tcgen05.mma per tile (M=128,
//     N=128 over the two boxes, K=16, bf16 -> fp32, A from tensor memory, B
//     from shared memory) into one of two 128-column TMEM accumulators, with
//     precomputed descriptors, and commits once per tile;
//   * warps 3-18 drain the accumulator with tcgen05.ld (thread = GEMM row of
//     its TMEM sub-partition; four warps per sub-partition, one per 16-column
//     group of each box), add L and run the mode's reduction in registers;
//     one result per row, CTA and column group is written at the end (the
//     sampling modes write one record per row and 16-column block instead).
// The grid is (vocab splits) x (M tiles), one CTA per SM; vocab tiles are
// dealt to the splits round-robin.
#include "device.cuh"
#include "internal.h"

namespace sdm {
namespace {

constexpr int kSmemLimit = 232448;   // 227 KB opt-in per block
constexpr uint32_t kWStageBytes = 64u * kTileN * 2u;   // 64 K rows x 128 ids bf16 = two 64 x 64 boxes
constexpr uint32_t kWBoxBytes = 64u * kBoxN * 2u;      // 8 KB
constexpr int kMaxWStages = 12;
constexpr int kMaxLStages = 6;
// Tensor memory: two 128-column fp32 accumulators, then A (128 rows x r
// bf16 per sub-tile, two per 32-bit column: r / 2 <= 128 columns each).
constexpr int kTmemA = 2 * kTileN;
constexpr int kTmemCols = 512;

// Shared memory: the W ring (stage = K block kb of 64 rows x the tile's two
// 64-id boxes), then the L ring (stage = one 64-id box of the tile's L rows),
// then the barriers.  A (128 rows x r, K-major, 128-byte swizzle) is gathered
// into the last r / 64 W stages and copied to tensor memory before those
// stages are first loaded.
struct SmemLayout {
    uint32_t a_off, l_off, l_box_bytes, l_stage_bytes, bar_off, tok_off, total;
};

__host__ __device__ inline SmemLayout make_layout(int r, int l_rows, int l_fp32, int w_stages, int l_stages,
                                                  int mode, int ms = 1) {
    SmemLayout s;
    const uint32_t w_bytes = static_cast<uint32_t>(w_stages) * kWStageBytes;
    // A fills the last ms tile slots (a slot is KB = r / 64 stages of 16 KB =
    // 128 x r x 2 bytes: one 128-row sub-tile of A)
    const int kb = r >> 6;
    s.a_off = static_cast<uint32_t>((w_stages / kb - ms) * kb) * kWStageBytes;
    s.l_off = w_bytes;
    s.l_box_bytes = (static_cast<uint32_t>(l_rows) * 128u + 1023u) & ~1023u;
    s.l_stage_bytes = mode_reads_l(mode) ? s.l_box_bytes * (l_fp32 ? 2u : 1u) : 0u;
    s.bar_off = s.l_off + static_cast<uint32_t>(l_stages) * s.l_stage_bytes;
    s.tok_off = s.bar_off + static_cast<uint32_t>(2 * w_stages + 2 * l_stages + 6) * 8u + 16u;   // the rows' tokens
    s.total = s.tok_off + static_cast<uint32_t>(kTileM * ms) * 4u + 1024u;
    return s;
}

__device__ __forceinline__ void fail_timeout(const GemmParams& p) { set_status(p.dev_status, SDM_DEV_TIMEOUT); }

// Token whose U row feeds GEMM row `grow`; -1 for an unused row.
template <int MODE>
__device__ __forceinline__ int gemm_row_token(const GemmParams& p, int grow) {
    int t = -1;
    if (MODE == MODE_CHAIN_GREEDY) {
        if (grow >= p.R) return -1;
        t = (p.d == 1) ? p.anchor[grow] : static_cast<int>(key_token(p.keys[static_cast<size_t>(p.d - 2) * p.R + grow]));
    } else if (MODE == MODE_CHAIN_SAMPLE) {
        if (grow >= p.R) return -1;
        t = (p.d == 1) ? p.anchor[grow] : p.tok_in[static_cast<size_t>(grow) * p.B + (p.d - 2)];
    } else if (mode_tree(MODE)) {
        if (grow >= p.rows) return -1;
        t = p.front_tok[grow];
        if (t < 0) return -1;
    } else if (MODE == MODE_ABSMAX) {
        return grow < p.rows ? grow : -1;
    } else if (mode_row_list(MODE)) {
        if (grow >= p.rows) return -1;
        t = p.res_tok[grow];
        if (t < 0) return -1;
    } else {
        if (grow >= p.R) return -1;
        t = p.res_tok[grow];
        if (t < 0) return -1;
    }
    if (t < 0 || t >= p.V) {
        set_status(p.dev_status, SDM_DEV_BAD_TOKEN);
        return -1;
    }
    return t;
}

__device__ __forceinline__ float bf_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf_hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

constexpr int C = kEpiCols;   // columns per epilogue thread and tile

// The C L values of column group g of the staged tile, box row lr (128-byte
// swizzle: 16-byte chunk c of a row sits at c ^ (lr & 7)).
__device__ __forceinline__ void load_l(const uint8_t* sl, uint32_t l_box_bytes, int l_fp32, int lr, int g,
                                       float (&out)[C]) {
    if (!l_fp32) {   // a constant where the kernel is instantiated per L dtype
        const uint8_t* rowp = sl + lr * 128;
#pragma unroll
        for (int c = 0; c < C / 8; ++c) {
            const int chunk = g * (C / 8) + c;
            const uint4 v = *reinterpret_cast<const uint4*>(rowp + ((chunk ^ (lr & 7)) << 4));
            out[c * 8 + 0] = bf_lo(v.x);
            out[c * 8 + 1] = bf_hi(v.x);
            out[c * 8 + 2] = bf_lo(v.y);
            out[c * 8 + 3] = bf_hi(v.y);
            out[c * 8 + 4] = bf_lo(v.z);
            out[c * 8 + 5] = bf_hi(v.z);
            out[c * 8 + 6] = bf_lo(v.w);
            out[c * 8 + 7] = bf_hi(v.w);
        }
    } else {   // two boxes of 32 fp32 columns
        const int col0 = g * C;
        const uint8_t* rowp = sl + (col0 >> 5) * l_box_bytes + lr * 128;
#pragma unroll
        for (int c = 0; c < C / 4; ++c) {
            const int chunk = ((col0 & 31) >> 2) + c;
            const float4 v = *reinterpret_cast<const float4*>(rowp + ((chunk ^ (lr & 7)) << 4));
            out[c * 4 + 0] = v.x;
            out[c * 4 + 1] = v.y;
            out[c * 4 + 2] = v.z;
            out[c * 4 + 3] = v.w;
        }
    }
}

// C consecutive elements of a global row (bf16 or fp32) starting at v0;
// entries at or past V read as 0 (callers mask them).
__device__ __forceinline__ void load_g(const void* base, int fp32, size_t off, int v0, int V, float (&out)[C]) {
    if (!fp32) {
        const uint16_t* p = static_cast<const uint16_t*>(base) + off;
#pragma unroll
        for (int c = 0; c < C / 8; ++c) {
            uint4 v = make_uint4(0, 0, 0, 0);
            if (v0 + c * 8 < V) v = __ldg(reinterpret_cast<const uint4*>(p + v0 + c * 8));
            out[c * 8 + 0] = bf_lo(v.x);
            out[c * 8 + 1] = bf_hi(v.x);
            out[c * 8 + 2] = bf_lo(v.y);
            out[c * 8 + 3] = bf_hi(v.y);
            out[c * 8 + 4] = bf_lo(v.z);
            out[c * 8 + 5] = bf_hi(v.z);
            out[c * 8 + 6] = bf_lo(v.w);
            out[c * 8 + 7] = bf_hi(v.w);
        }
    } else {
        const float* p = static_cast<const float*>(base) + off;
#pragma unroll
        for (int c = 0; c < C / 4; ++c) {
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (v0 + c * 4 < V) v = __ldg(reinterpret_cast<const float4*>(p + v0 + c * 4));
            out[c * 4 + 0] = v.x;
            out[c * 4 + 1] = v.y;
            out[c * 4 + 2] = v.z;
            out[c * 4 + 3] = v.w;
        }
    }
}

// C elements of a global row as raw 16-byte words (bf16: r[0..1], fp32:
// r[0..3]), issued now and unpacked when used; words at or past V read 0.
__device__ __forceinline__ void load_raw(const void* base, int fp32, size_t off, int v0, int V, uint4 (&r)[4]) {
    const int per = fp32 ? 4 : 8;
    const uint8_t* p = static_cast<const uint8_t*>(base) + (off + v0) * (fp32 ? 4 : 2);
#pragma unroll
    for (int c = 0; c < 4; ++c)
        r[c] = ((fp32 || c < 2) && v0 + c * per < V) ? __ldg(reinterpret_cast<const uint4*>(p + c * 16))
                                                      : make_uint4(0, 0, 0, 0);
}

__device__ __forceinline__ void unpack_raw(int fp32, const uint4 (&r)[4], float (&out)[C]) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const uint32_t w[4] = {r[c].x, r[c].y, r[c].z, r[c].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            if (fp32) {
                out[c * 4 + k] = __uint_as_float(w[k]);
            } else if (c < 2) {
                out[c * 8 + 2 * k] = bf_lo(w[k]);
                out[c * 8 + 2 * k + 1] = bf_hi(w[k]);
            }
        }
    }
}

// Per-row epilogue state of each mode.
template <int MODE>
struct Epi;

// Maximum of C values as a balanced tree (no serial dependency chain).
__device__ __forceinline__ float maxc(const float (&z)[C]) {
    float t[C / 2];
#pragma unroll
    for (int j = 0; j < C / 2; ++j) t[j] = fmaxf(z[j], z[j + C / 2]);
#pragma unroll
    for (int w = C / 4; w > 0; w >>= 1)
#pragma unroll
        for (int j = 0; j < w; ++j) t[j] = fmaxf(t[j], t[j + w]);
    return t[0];
}

// Lowest j with z[j] == m (m is one of the z).
__device__ __forceinline__ int first_index_of(const float (&z)[C], float m) {
    int jj = C - 1;
#pragma unroll
    for (int j = C - 1; j >= 0; --j)
        if (z[j] == m) jj = j;
    return jj;
}

__device__ __forceinline__ void mask_tail(float (&z)[C], int vbase, int V) {
    if (vbase + C > V) {
#pragma unroll
        for (int j = 0; j < C; ++j)
            if (vbase + j >= V) z[j] = -INFINITY;
    }
}

template <>
struct Epi<MODE_CHAIN_GREEDY> {
    bool valid;
    int group;
    float best;
    uint32_t best_v;
    __device__ __forceinline__ void init(const GemmParams& p, int grow) {
        valid = grow < p.R;
        best = -INFINITY;
        best_v = 0;
    }
    __device__ __forceinline__ void consume(const GemmParams& p, const uint8_t* sl, uint32_t lbb, int lf, int lrow,
                                            int vbase,
                                            int g, const uint32_t (&acc)[C]) {
        if (!valid) return;
        float z[C];
        load_l(sl, lbb, lf, lrow, g, z);
#pragma unroll
        for (int j = 0; j < C; ++j) z[j] = z[j] + __uint_as_float(acc[j]);   // fp32(L) + Markov, one rounding
        mask_tail(z, vbase, p.V);
        const float m = maxc(z);
        if (m > best) {   // strict: an earlier (lower) id keeps a tie
            best = m;
            best_v = static_cast<uint32_t>(vbase + first_index_of(z, m));
        }
    }
    __device__ __forceinline__ void flush(const GemmParams& p, int grow) {
        if (valid) atomicMax(&p.keys[static_cast<size_t>(p.d - 1) * p.R + grow], argmax_key(best, best_v));
    }
};

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Block record (m, s) of the 16 columns: m = max z / T, s = sum exp(z / T - m),
// formed in base 2 (x = z log2(e) / T, s = sum 2^(x - max x)).
template <>
struct Epi<MODE_CHAIN_SAMPLE> {
    bool valid;
    int group;
    float sc;      // log2(e) / T
    float2* rec;   // this row's records [nb]
    __device__ __forceinline__ void init(const GemmParams& p, int grow) {
        valid = grow < p.R;
        sc = p.inv_t * kLog2e;
        rec = p.blk + static_cast<size_t>(valid ? grow : 0) * p.nb;
    }
    __device__ __forceinline__ void consume(const GemmParams& p, const uint8_t* sl, uint32_t lbb, int lf, int lrow,
                                            int vbase,
                                            int g, const uint32_t (&acc)[C]) {
        if (!valid || vbase >= p.V) return;
        float z[C];
        load_l(sl, lbb, lf, lrow, g, z);
#pragma unroll
        for (int j = 0; j < C; ++j) z[j] = (z[j] + __uint_as_float(acc[j])) * sc;
        mask_tail(z, vbase, p.V);
        const float m = maxc(z);
        float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < C; ++j) ps[j & 3] += fast_exp2(z[j] - m);   // 2^-inf = 0 on the tail
        rec[vbase / C] = make_float2(m * kLn2, (ps[0] + ps[1]) + (ps[2] + ps[3]));
    }
    __device__ __forceinline__ void flush(const GemmParams&, int) {}
};

// Block record (m, s) of the 16 columns of a frontier row: m = max z,
// s = sum exp(z - m) (base 2 inside, as for sampling with T = 1).
template <>
struct Epi<MODE_TREE> {
    bool valid;
    int group;
    float2* rec;
    __device__ __forceinline__ void init(const GemmParams& p, int grow) {
        valid = grow < p.rows && p.front_tok[grow] >= 0;
        rec = p.blk + static_cast<size_t>(grow < p.rows ? grow : 0) * p.nb;
    }
    __device__ __forceinline__ void consume(const GemmParams& p, const uint8_t* sl, uint32_t lbb, int lf, int lrow,
                                            int vbase,
                                            int g, const uint32_t (&acc)[C]) {
        if (!valid || vbase >= p.V) return;
        float z[C];
        load_l(sl, lbb, lf, lrow, g, z);   // lrow: the request's L row
#pragma unroll
        for (int j = 0; j < C; ++j) z[j] = (z[j] + __uint_as_float(acc[j])) * kLog2e;
        mask_tail(z, vbase, p.V);
        const float m = maxc(z);
        float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < C; ++j) ps[j & 3] += fast_exp2(z[j] - m);
        rec[vbase / C] = make_float2(m * kLn2, (ps[0] + ps[1]) + (ps[2] + ps[3]));
    }
    __device__ __forceinline__ void flush(const GemmParams&, int) {}
};

// Block record (0, s) of the 16 columns: s = sum max(0, p_v - q_v) with
// p_v = exp(target / T - lse_p), q_v = exp(z / T - lse_q).
template <>
struct Epi<MODE_RESID> {
    bool valid;
    int group;
    size_t l_off, t_off;
    float lse_q, lse_p;
    float2* rec;
    __device__ __forceinline__ void init(const GemmParams& p, int grow) {
        valid = grow < p.R && p.res_tok[grow] >= 0;
        rec = p.blk + static_cast<size_t>(grow < p.R ? grow : 0) * p.nb;
        if (valid) {
            const int jpos = p.res_pos[grow];
            l_off = (static_cast<size_t>(grow) * p.gamma + jpos) * static_cast<size_t>(p.V);
            t_off = static_cast<size_t>(p.res_trow[grow]) * static_cast<size_t>(p.V);
            lse_q = p.lse_q[static_cast<size_t>(grow) * p.gamma + jpos];
            lse_p = p.res_lse_p[grow];
        }
    }
    __device__ __forceinline__ void consume(const GemmParams& p, const uint8_t*, uint32_t, int, int, int vbase, int,
                                            const uint32_t (&acc)[C]) {
        if (!valid || vbase >= p.V) return;
        float lv[C], tv[C];
        load_g(p.L, p.l_fp32, l_off, vbase, p.V, lv);
        load_g(p.target, p.t_fp32, t_off, vbase, p.V, tv);
        float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < C; ++j) {
            const float q = __expf((lv[j] + __uint_as_float(acc[j])) * p.inv_t - lse_q);
            const float pv = __expf(tv[j] * p.inv_t - lse_p);
            const float w = (vbase + j < p.V) ? fmaxf(pv - q, 0.f) : 0.f;
            ps[j & 3] += w;
        }
        rec[vbase / C] = make_float2(0.f, (ps[0] + ps[1]) + (ps[2] + ps[3]));
    }
    __device__ __forceinline__ void flush(const GemmParams&, int) {}
};

// Listed row g: window row res_pos[g] of request res_req[g], its L row at
// (request, position) and its target row res_trow[g].
__device__ __forceinline__ bool list_row(const GemmParams& p, int grow, size_t& l_off, size_t& t_off) {
    if (grow >= p.rows || p.res_tok[grow] < 0) return false;
    const size_t req = static_cast<size_t>(p.res_req[grow]);
    l_off = (req * p.gamma + static_cast<size_t>(p.res_pos[grow])) * static_cast<size_t>(p.V);
    t_off = static_cast<size_t>(p.res_trow[grow]) * static_cast<size_t>(p.V);
    return true;
}

__device__ __forceinline__ float2* part_slot(const GemmParams& p, int grow, int group) {
    return p.part + static_cast<size_t>(grow) * p.n_part + blockIdx.x * kColGroups + group;
}

// Two fp32 values in one 64-bit register, the operand of the f32x2
// instructions (sm_100 and later).
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ float2 f2_unpack(uint64_t x) {
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(x));
    return r;
}

// Two columns of the bounded tree step: z = fp32(L) + a for the bf16 pair in
// w (the mixed-precision add: the exact conversion and one rounding, as
// fp32(L) + a), then acc += 2^(z log2(e) - m log2(e)) lane-wise, the scaling
// one paired fma, the sum one paired add.
__device__ __forceinline__ void lse2_bf16(uint32_t w, uint32_t a0, uint32_t a1, uint64_t sc2, uint64_t mo2,
                                          uint64_t& acc) {
    asm("{\n\t.reg .b16 lo, hi;\n\t.reg .f32 z0, z1, e0, e1;\n\t.reg .b64 zz, xx, ee;\n\t"
        "mov.b32 {lo, hi}, %1;\n\t"
        "add.rn.f32.bf16 z0, lo, %2;\n\t"
        "add.rn.f32.bf16 z1, hi, %3;\n\t"
        "mov.b64 zz, {z0, z1};\n\t"
        "fma.rn.f32x2 xx, zz, %4, %5;\n\t"
        "mov.b64 {z0, z1}, xx;\n\t"
        "ex2.approx.ftz.f32 e0, z0;\n\t"
        "ex2.approx.ftz.f32 e1, z1;\n\t"
        "mov.b64 ee, {e0, e1};\n\t"
        "add.rn.f32x2 %0, %0, ee;\n\t}"
        : "+l"(acc)
        : "r"(w), "f"(__uint_as_float(a0)), "f"(__uint_as_float(a1)), "l"(sc2), "l"(mo2));
}

// (max, sum) of the logits z of a frontier row over every column this thread
// consumes, each exponential one fma and one ex2 (2^(z log2(e) - m log2(e))).
// The reference m is, where the prepared tables give it, the row's bound
// m = max_v L_v + c(y) >= every z (no maximum is tracked: the largest term is
// at least exp(-2 c(y)) and none exceeds 1; used while c(y) <= 16), else the
// running maximum.  A thread that consumed nothing leaves (-inf, 0).
template <>
struct Epi<MODE_TREE_LSE> {
    bool valid, bounded;
    int group;
    float m, s, mo;
    uint64_t pa, pb, sc2, mo2;   // bounded bf16 path: two paired sums, (log2 e, log2 e), (-mo, -mo)
    __device__ __forceinline__ void init(const GemmParams& p, int grow) {
        const int t = grow < p.rows ? p.front_tok[grow] : -1;
        valid = t >= 0 && t < p.V;
        m = -INFINITY;
        s = 0.f;
        bounded = false;
        if (valid && p.row_lmax && p.c_bound) {
            const float cy = p.c_bound[t];
            const float lmax = p.row_lmax[(grow / p.P) * p.B + (p.d - 1)];
            if (cy <= 16.f && lmax > -INFINITY && lmax < INFINITY) {
                bounded = true;
                m = lmax + cy;
            }
        }
        mo = m * kLog2e;
        pa = pb = 0;   // the bits of (0.f, 0.f)
        sc2 = f2_pack(kLog2e, kLog2e);
        mo2 = f2_pack(-mo, -mo);
    }
    __device__ __forceinline__ void consume(const GemmParams& p, const uint8_t* sl, uint32_t lbb, int lf, int lrow,
                                            int vbase, int g, const uint32_t (&acc)[C]) {
        if (!valid || vbase >= p.V) return;
        if (bounded && !lf && vbase + C <= p.V) {
            // the common case (fixed reference, bf16 L, no vocabulary tail):
            // the 16 L values of row lrow, column group g, two per 32-bit word
            const uint8_t* rowp = sl + lrow * 128;
#pragma unroll
            for (int c = 0; c < C / 8; ++c) {
                const uint4 v = *reinterpret_cast<const uint4*>(rowp + (((g * (C / 8) + c) ^ (lrow & 7)) << 4));
                lse2_bf16(v.x, acc[c * 8 + 0], acc[c * 8 + 1], sc2, mo2, pa);
                lse2_bf16(v.y, acc[c * 8 + 2], acc[c * 8 + 3], sc2, mo2, pb);
                lse2_bf16(v.z, acc[c * 8 + 4], acc[c * 8 + 5], sc2, mo2, pa);
                lse2_bf16(v.w, acc[c * 8 + 6], acc[c * 8 + 7], sc2, mo2, pb);
            }
            return;
        }
        float z[C];
        load_l(sl, lbb, lf, lrow, g, z);   // lrow: the request's L row
#pragma unroll
        for (int j = 0; j < C; ++j) z[j] = z[j] + __uint_as_float(acc[j]);   // fp32(L) + Markov, one rounding
        mask_tail(z, vbase, p.V);
        if (!bounded) {
            const float mb = maxc(z);   // finite: column vbase < V
            if (mb > m) {
                s *= fast_exp2((m - mb) * kLog2e);   // 0 while m = -inf
                m = mb;
                mo = m * kLog2e;
            }
        }
        float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < C; ++j) ps[j & 3] += fast_exp2(fmaf(z[j], kLog2e, -mo));   // 2^-inf = 0 on the tail
        s += (ps[0] + ps[1]) + (ps[2] + ps[3]);
    }
    // this thread's (m, s): (-inf, 0) when it consumed nothing (the paired
    // sums share the fixed reference m with s)
    __device__ __forceinline__ float2 partial() const {
        const float2 a = f2_unpack(pa), b = f2_unpack(pb);
        const float t = s + ((a.x + a.y) + (b.x + b.y));
        return make_float2(t > 0.f ? m : -INFINITY, t);
    }
    __device__ __forceinline__ void flush(const GemmParams& p, int grow) {
        if (valid) *part_slot(p, grow, group) = partial();
    }
};

// Online (max, sum) of x = z log2(e) / T over every column this thread
// consumes; the partial is (max x ln 2, sum 2^(x - max x)) = (max z / T, sum
// exp(z / T - max)).  A thread that consumed nothing writes (-inf, 0).
template <>
struct Epi<MODE_QLSE> {
    bool valid;
    int group;
    size_t l_off, t_off;
    float sc, m, s;
    uint4 lr[2][4];   // a tile's L words (bf16: [0..1] of each slice)
    __device__ __forceinline__ void init(const GemmParams& p, int grow) {
        valid = list_row(p, grow, l_off, t_off);
        sc = p.inv_t * kLog2e;
        m = -INFINITY;
        s = 0.f;
    }
    __device__ __forceinline__ void issue(const GemmParams& p, const int (&vbase)[2]) {
        if (!valid) return;
#pragma unroll
        for (int h = 0; h < 2; ++h) load_raw(p.L, p.l_fp32, l_off, vbase[h], p.V, lr[h]);
    }
    __device__ __forceinline__ void consume_slice(const GemmParams& p, int vbase, int h, const uint32_t (&acc)[C]) {
        if (!valid || vbase >= p.V) return;
        float z[C];
        unpack_raw(p.l_fp32, lr[h], z);
#pragma unroll
        for (int j = 0; j < C; ++j) z[j] = (z[j] + __uint_as_float(acc[j])) * sc;
        mask_tail(z, vbase, p.V);
        const float mb = maxc(z);   // finite: column vbase < V
        if (mb > m) {
            s *= fast_exp2(m - mb);
            m = mb;
        }
        float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < C; ++j) ps[j & 3] += fast_exp2(z[j] - m);
        s += (ps[0] + ps[1]) + (ps[2] + ps[3]);
    }
    __device__ __forceinline__ void flush(const GemmParams& p, int grow) {
        if (valid) *part_slot(p, grow, group) = make_float2(m * kLn2, s);
    }
};

// Partial sum of min(q_v, p_v), q_v = exp(z / T - lse_q), p_v = exp(target /
// T - lse_p), over every column this thread consumes.
template <>
struct Epi<MODE_TVMIN> {
    bool valid;
    int group;
    size_t l_off, t_off;
    float lse_q, lse_p, s;
    __device__ __forceinline__ void init(const GemmParams& p, int grow) {
        valid = list_row(p, grow, l_off, t_off);
        s = 0.f;
        if (valid) {
            lse_q = p.row_lse_q[grow];
            lse_p = p.res_lse_p[grow];
        }
    }
    __device__ __forceinline__ void consume(const GemmParams& p, const uint8_t*, uint32_t, int, int, int vbase, int,
                                            const uint32_t (&acc)[C]) {
        if (!valid || vbase >= p.V) return;
        float lv[C], tv[C];
        load_g(p.L, p.l_fp32, l_off, vbase, p.V, lv);
        load_g(p.target, p.t_fp32, t_off, vbase, p.V, tv);
        float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < C; ++j) {
            const float q = __expf((lv[j] + __uint_as_float(acc[j])) * p.inv_t - lse_q);
            const float pv = __expf(tv[j] * p.inv_t - lse_p);
            ps[j & 3] += (vbase + j < p.V) ? fminf(pv, q) : 0.f;
        }
        s += (ps[0] + ps[1]) + (ps[2] + ps[3]);
    }
    __device__ __forceinline__ void flush(const GemmParams& p, int grow) {
        if (valid) *part_slot(p, grow, group) = make_float2(0.f, s);
    }
};

// Typed soft-label pass (L bf16; target bf16 or fp32 by TF32): the loads of
// both 16-column slices of a tile are issued before the first is used, so a
// warp keeps a whole tile's rows in flight (the row-per-lane loads are
// latency-bound otherwise).
template <int TF32>
struct EpiTvTyped {
    static constexpr int kT = TF32 ? 4 : 2;   // 16-byte words of target per slice
    bool valid;
    int group;
    size_t l_off, t_off;
    float lse_q, lse_p, s;
    uint4 lr[2][2], tr[2][kT];
    __device__ __forceinline__ void init(const GemmParams& p, int grow) {
        valid = list_row(p, grow, l_off, t_off);
        s = 0.f;
        if (valid) {
            lse_q = p.row_lse_q[grow];
            lse_p = p.res_lse_p[grow];
        }
    }
    __device__ __forceinline__ void issue(const GemmParams& p, const int (&vbase)[2]) {
        if (!valid) return;
        const uint16_t* L = static_cast<const uint16_t*>(p.L) + l_off;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int c = 0; c < 2; ++c)
                lr[h][c] = vbase[h] + c * 8 < p.V ? __ldg(reinterpret_cast<const uint4*>(L + vbase[h] + c * 8))
                                                  : make_uint4(0, 0, 0, 0);
            if (TF32) {
                const float* T = static_cast<const float*>(p.target) + t_off;
#pragma unroll
                for (int c = 0; c < kT; ++c)
                    tr[h][c] = vbase[h] + c * 4 < p.V ? __ldg(reinterpret_cast<const uint4*>(T + vbase[h] + c * 4))
                                                      : make_uint4(0, 0, 0, 0);
            } else {
                const uint16_t* T = static_cast<const uint16_t*>(p.target) + t_off;
#pragma unroll
                for (int c = 0; c < kT; ++c)
                    tr[h][c] = vbase[h] + c * 8 < p.V ? __ldg(reinterpret_cast<const uint4*>(T + vbase[h] + c * 8))
                                                      : make_uint4(0, 0, 0, 0);
            }
        }
    }
    __device__ __forceinline__ void consume_slice(const GemmParams& p, int vbase, int h, const uint32_t (&acc)[C]) {
        if (!valid || vbase >= p.V) return;
        float lv[C], tv[C];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const uint32_t w[4] = {lr[h][c].x, lr[h][c].y, lr[h][c].z, lr[h][c].w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                lv[c * 8 + 2 * k] = bf_lo(w[k]);
                lv[c * 8 + 2 * k + 1] = bf_hi(w[k]);
            }
        }
#pragma unroll
        for (int c = 0; c < kT; ++c) {
            const uint32_t w[4] = {tr[h][c].x, tr[h][c].y, tr[h][c].z, tr[h][c].w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                if (TF32) {
                    tv[c * 4 + k] = __uint_as_float(w[k]);
                } else {
                    tv[c * 8 + 2 * k] = bf_lo(w[k]);
                    tv[c * 8 + 2 * k + 1] = bf_hi(w[k]);
                }
            }
        }
        float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < C; ++j) {
            const float q = __expf((lv[j] + __uint_as_float(acc[j])) * p.inv_t - lse_q);
            const float pv = __expf(tv[j] * p.inv_t - lse_p);
            ps[j & 3] += (vbase + j < p.V) ? fminf(pv, q) : 0.f;
        }
        s += (ps[0] + ps[1]) + (ps[2] + ps[3]);
    }
    __device__ __forceinline__ void flush(const GemmParams& p, int grow) {
        if (valid) *part_slot(p, grow, group) = make_float2(0.f, s);
    }
};

template <>
struct Epi<MODE_TVMIN_B16> : EpiTvTyped<0> {};
template <>
struct Epi<MODE_TVMIN_B32> : EpiTvTyped<1> {};

template <>
struct Epi<MODE_ABSMAX> {
    bool valid;
    int group;
    float best;
    __device__ __forceinline__ void init(const GemmParams& p, int grow) {
        valid = grow < p.rows;
        best = 0.f;
    }
    // Columns past V hold 0 (the W tile's out-of-range fill), which never
    // raises a maximum of absolute values.
    __device__ __forceinline__ void consume(const GemmParams&, const uint8_t*, uint32_t, int, int, int, int,
                                            const uint32_t (&acc)[C]) {
        float t[C / 2];
#pragma unroll
        for (int j = 0; j < C / 2; ++j)
            t[j] = fmaxf(fabsf(__uint_as_float(acc[j])), fabsf(__uint_as_float(acc[j + C / 2])));
#pragma unroll
        for (int w = C / 4; w > 0; w >>= 1)
#pragma unroll
            for (int j = 0; j < w; ++j) t[j] = fmaxf(t[j], t[j + w]);
        best = fmaxf(best, t[0]);
    }
    // the bits of non-negative floats order like their values
    __device__ __forceinline__ void flush(const GemmParams& p, int grow) {
        if (valid) atomicMax(&p.absmax_bits[grow], __float_as_uint(best));
    }
};

// W tile i (vocab ids from (blockIdx.x + i gridDim.x) 128) into tile slot
// `slot`: KB stages of [64 K rows x 128 ids], two 64-id boxes each.
__device__ __forceinline__ void issue_w_tile(const CUtensorMap& tmW, uint8_t* smem, uint64_t* wfull, int i, int slot,
                                             int KB, uint64_t pol) {
    const int v0 = (static_cast<int>(blockIdx.x) + i * static_cast<int>(gridDim.x)) * kTileN;
    for (int kb = 0; kb < KB; ++kb) {
        const int s = slot * KB + kb;
        uint8_t* st = smem + static_cast<uint32_t>(s) * kWStageBytes;
        mbar_arrive_expect_tx(&wfull[s], kWStageBytes);
        tma_load_2d(st, &tmW, &wfull[s], v0, kb * 64, pol);
        tma_load_2d(st + kWBoxBytes, &tmW, &wfull[s], v0 + kBoxN, kb * 64, pol);
    }
}

// L box bi (tile bi / 2, 64-id half bi % 2) of the CTA's L rows into stage t.
__device__ __forceinline__ void issue_l_box(const CUtensorMap& tmL, uint8_t* smem, const SmemLayout& lay,
                                            uint64_t* lfull, const GemmParams& p, int bi, int t, int mode, int ms,
                                            uint64_t pol) {
    const int lrow0 = mode_tree(mode) ? static_cast<int>(blockIdx.y) * (kTileM * ms / p.P)
                                      : static_cast<int>(blockIdx.y) * kTileM * ms;
    const int vb = (static_cast<int>(blockIdx.x) + (bi >> 1) * static_cast<int>(gridDim.x)) * kTileN + (bi & 1) * kBoxN;
    uint8_t* sl = smem + lay.l_off + static_cast<uint32_t>(t) * lay.l_stage_bytes;
    mbar_arrive_expect_tx(&lfull[t], static_cast<uint32_t>(p.l_rows) * 128u * (p.l_fp32 ? 2u : 1u));
    tma_load_3d(sl, &tmL, &lfull[t], vb, p.d - 1, lrow0, pol);
    if (p.l_fp32) tma_load_3d(sl + lay.l_box_bytes, &tmL, &lfull[t], vb + 32, p.d - 1, lrow0, pol);
}

// MS = 128-row sub-tiles of GEMM rows per CTA; LF = the L dtype (0 bf16, 1
// fp32) where the mode stages L in shared memory, -1 (read from p) otherwise.  MS = 2 (PCTree levels of
// more than 128 frontier rows): both sub-tiles' A rows sit in tensor memory
// and every W tile feeds both, one accumulator per sub-tile, the epilogue of
// one sub-tile overlapping the MMAs of the other; the W stream per row halves.
template <int MODE, int MS, int LF>
__global__ void __launch_bounds__(kGemmThreads, 1)
    markov_gemm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmL,
                       const GemmParams p) {
    static_assert(MS == 1 || (MS == 2 && mode_tree(MODE) && !mode_loads_first(MODE)), "two sub-tiles: PCTree modes");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int SW = p.w_stages, SL = p.l_stages;
    const SmemLayout lay = make_layout(p.r, p.l_rows, p.l_fp32, SW, SL, MODE, MS);
    uint8_t* sA = smem + lay.a_off;
    uint64_t* wfull = reinterpret_cast<uint64_t*>(smem + lay.bar_off);
    uint64_t* wdone = wfull + SW;   // per tile slot: the slot's last tile has completed
    uint64_t* lfull = wdone + SW;
    uint64_t* lempty = lfull + SL;
    constexpr int NACC = 2;   // accumulators: one per sub-tile, or two used in turn
    uint64_t* tfull = lempty + SL;
    uint64_t* tempty = tfull + NACC;
    uint64_t* a_done = tempty + NACC;
    uint64_t* drain = a_done + 1;   // the MMA warp's own tensor-core work, before tensor memory is freed
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    int* s_rowtok = reinterpret_cast<int*>(smem + lay.tok_off);   // [kTileM * MS]
    const uint64_t lim = p.wait_ns ? p.wait_ns : kWaitLimitNs;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int row0 = blockIdx.y * kTileM * MS;
    const int KB = p.r >> 6;   // K blocks of 64 per tile
    const int NTS = SW / KB;   // W tile slots: tile i takes stages (i % NTS) * KB .. + KB - 1
    // vocab tiles are dealt round-robin (tile = blockIdx.x + i * gridDim.x) so
    // that concurrently running CTAs read neighbouring segments of every W and
    // L row
    const int nt = (p.n_tiles - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) / static_cast<int>(gridDim.x);

    // set-up that reads nothing the previous kernel in the stream writes
    if (threadIdx.x == 0) {
        for (int s = 0; s < SW; ++s) {
            mbar_init(&wfull[s], 1);
            mbar_init(&wdone[s], 1);
        }
        for (int s = 0; s < SL; ++s) {
            mbar_init(&lfull[s], 1);
            mbar_init(&lempty[s], kEpiWarps);
        }
        for (int b = 0; b < NACC; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], kEpiWarps);
        }
        mbar_init(a_done, 1);
        mbar_init(drain, 1);
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmW);
        if (mode_reads_l(MODE)) tma_prefetch_desc(&tmL);
    }
    __syncthreads();   // the barriers are initialised for every warp

    // 0. loads that read nothing a previous kernel writes (W, and L, are
    //    inputs), issued before the wait on the previous kernel: the first W
    //    tiles (the slots that do not hold A) and the first L boxes
    const int w_pre = nt < NTS - MS ? nt : NTS - MS;
    const int l_pre = mode_reads_l(MODE) ? (2 * nt < SL ? 2 * nt : SL) : 0;
    if (warp == 0 && lane == 0 && !p.withhold_loads) {
        const uint64_t pol_w = policy_evict_last();
        for (int i = 0; i < w_pre; ++i) issue_w_tile(tmW, smem, wfull, i, i % NTS, KB, pol_w);
    }
    if (warp == 2 && lane == 0 && !p.withhold_loads) {
        const uint64_t pol_l = policy_evict_first();
        for (int bi = 0; bi < l_pre; ++bi) issue_l_box(tmL, smem, lay, lfull, p, bi, bi % SL, MODE, MS, pol_l);
    }
    pdl_wait();   // tokens (and every buffer this launch writes) belong to the previous kernel until here
    pdl_trigger();

    // 1. the rows' tokens, every load in flight at once, then A = U[tok(m)]
    //    for the 128 MS rows (K-major, 128-byte swizzle: 16-byte chunk c of
    //    row m in K block kb sits at chunk c ^ (m & 7)); sub-tile h occupies
    //    its own slot (128 x r x 2 bytes).
    for (int rr = threadIdx.x; rr < kTileM * MS; rr += kGemmThreads) s_rowtok[rr] = gemm_row_token<MODE>(p, row0 + rr);
    __syncthreads();
    const int kchunks = p.r >> 3;
    for (int rr = warp; rr < kTileM * MS; rr += kGemmThreads / 32) {
        const int tok = s_rowtok[rr];
        const uint16_t* src = (p.a_rows && tok >= 0) ? p.a_rows + static_cast<size_t>(row0 + rr) * p.r
                                                     : p.U + static_cast<size_t>(tok < 0 ? 0 : tok) * p.r;
        const int rm = rr & (kTileM - 1);
        uint8_t* sub = sA + (rr / kTileM) * (kTileM * p.r * 2);
        for (int q = lane; q < kchunks; q += 32) {
            uint8_t* dst = sub + (q >> 3) * (kTileM * 128) + rm * 128 + (((q & 7) ^ (rm & 7)) << 4);
            cp_async_16(dst, src + q * 8, tok < 0 ? 0u : 16u);
        }
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    cp_async_wait_all();
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // 2a. W producer: per tile, KB stages of [64 K rows x 128 ids] (two
        //     64 x 64 boxes) in the tile's slot.  A slot is free again once
        //     its last tile's MMAs have completed: the first epilogue warp
        //     arrives on wdone[slot] when it sees that tile's accumulator
        //     full, so the MMA warp commits once per tile (a commit waits for
        //     the MMA pipe to drain; one per stage would cost KB drains per
        //     tile).  The last slot holds A until it is in tensor memory.
        if (lane == 0 && nt > 0 && !p.withhold_loads) {
            const uint64_t pol_w = policy_evict_last();
            bool ok = true;
            int issued = w_pre;   // tiles whose W loads were issued (the first before the wait)
            for (int i = w_pre; i < nt && ok; ++i) {
                const int slot = i % NTS;
                if (i >= NTS) ok = mbar_wait(&wdone[slot], ((i / NTS) - 1) & 1, lim);
                else if (slot >= NTS - MS) ok = mbar_wait(a_done, 0, lim);
                if (!ok) break;
                issue_w_tile(tmW, smem, wfull, i, slot, KB, pol_w);
                issued = i + 1;
            }
            if (!ok) fail_timeout(p);
            // every copy issued has landed before the CTA may exit (a wait
            // elsewhere may have run out while they were in flight): slot sl
            // was armed by the tiles sl, sl + NTS, ... below `issued`
            for (int sl = 0; sl < NTS && sl < issued; ++sl) {
                const int arms = (issued - 1 - sl) / NTS + 1;
                for (int kb = 0; kb < KB; ++kb) mbar_wait(&wfull[sl * KB + kb], (arms - 1) & 1, lim);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // 3. MMA issuer: A into tensor memory once, then per tile
        //    D[128 x 128] = sum over K blocks of A_kb * W_kb, four K = 16
        //    steps per stage, N = 128 per instruction.  The whole warp runs
        //    the loop and waits; each tcgen05 instruction is issued by the
        //    lane elect.sync picks.
        const uint32_t idesc = idesc_bf16_f32(kTileM, kTileN, true);
        // Descriptors are formed once and advanced by adding the k-step's
        // offset to their 14-bit start-address field (address >> 4; every
        // shared address here is below 256 KB, so the field cannot carry):
        // A steps 32 bytes within a 128-byte swizzle row and 128 x 128
        // bytes per K block of 64; B steps 16 rows of 128 bytes, and its
        // second 64-id box (the MN-atom stride) is kWBoxBytes further.
        const int ksteps = p.r >> 4;
        for (int h = 0; h < MS; ++h) {   // sub-tile h's A at columns kTmemA + h r / 2
            const uint64_t a_desc0 = smem_desc_sw128(smem_u32(sA + h * (kTileM * p.r * 2)), 16, 1024);
            const uint32_t a_tmem = tmem_base + static_cast<uint32_t>(kTmemA + h * (p.r >> 1));
            for (int ks = 0; ks < ksteps; ++ks)
                tmem_cp_128x256b_warp(a_tmem + static_cast<uint32_t>(ks * 8),
                                      a_desc0 + static_cast<uint64_t>((ks >> 2) * ((kTileM * 128) >> 4) + (ks & 3) * 2));
        }
        mma_commit_warp(a_done);   // the A stages may be loaded once the copy has read them
        const uint64_t b_desc0 = smem_desc_sw128(smem_u32(smem), kWBoxBytes, 1024);
        bool ok = true;
        if constexpr (MS == 2) {
            // one 128 x 128 accumulator per sub-tile: each W stage feeds both
            // sub-tiles' MMAs, the epilogue of one sub-tile overlapping the
            // MMAs of the other (four 128 x 64 accumulators, which let the
            // MMAs run further ahead, measured slower)
            for (int i = 0; i < nt && ok; ++i) {
                const int slot = i % NTS;
                const uint32_t par = static_cast<uint32_t>(i / NTS) & 1u;
                for (int h = 0; h < MS && ok; ++h) {
                    if (i >= 1) ok = __all_sync(0xffffffffu, mbar_wait(&tempty[h], (i - 1) & 1, lim));
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(h * kTileN);
                    const uint32_t a_tmem = tmem_base + static_cast<uint32_t>(kTmemA + h * (p.r >> 1));
                    for (int kb = 0; kb < KB; ++kb) {
                        const int s = slot * KB + kb;
                        if (h == 0) {   // the second sub-tile reuses the stages the first waited for
                            ok = __all_sync(0xffffffffu, mbar_wait(&wfull[s], par, lim));
                            if (!ok) break;
                            tc_fence_after();
                        }
                        const uint64_t bd0 =
                            b_desc0 + static_cast<uint64_t>((static_cast<uint32_t>(s) * kWStageBytes) >> 4);
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            mma_bf16_ts_warp(d_tmem, a_tmem + static_cast<uint32_t>((kb * 4 + j) * 8),
                                             bd0 + static_cast<uint64_t>(j * (2048 >> 4)), idesc, (kb | j) ? 1u : 0u);
                    }
                    if (ok) mma_commit_warp(&tfull[h]);
                }
            }
        } else {
            // two 128 x 128 accumulators, used in turn
            for (int i = 0; i < nt && ok; ++i) {
                const int slot = i % NTS;
                const uint32_t par = static_cast<uint32_t>(i / NTS) & 1u;
                const int b = i & 1, use = i >> 1;
                if (use >= 1) ok = __all_sync(0xffffffffu, mbar_wait(&tempty[b], (use - 1) & 1, lim));
                if (!ok) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(b * kTileN);
                const uint32_t a_tmem = tmem_base + static_cast<uint32_t>(kTmemA);
                for (int kb = 0; kb < KB; ++kb) {
                    const int s = slot * KB + kb;
                    ok = __all_sync(0xffffffffu, mbar_wait(&wfull[s], par, lim));
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t bd0 = b_desc0 + static_cast<uint64_t>((static_cast<uint32_t>(s) * kWStageBytes) >> 4);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        mma_bf16_ts_warp(d_tmem, a_tmem + static_cast<uint32_t>((kb * 4 + j) * 8),
                                         bd0 + static_cast<uint64_t>(j * (2048 >> 4)), idesc, (kb | j) ? 1u : 0u);
                }
                if (ok) mma_commit_warp(&tfull[b]);
            }
        }
        if (!ok && lane == 0) fail_timeout(p);
        // every tensor-core operation this warp issued (the A copy, the
        // MMAs) completes before tensor memory is freed, whether or not the
        // epilogue waited for it
        mma_commit_warp(drain);
        mbar_wait(drain, 0, lim);
        __syncwarp();
    } else if (warp == 2) {
        // 2b. L producer: the tile's two 64-id boxes of L rows, one stage each
        if (mode_reads_l(MODE) && lane == 0 && nt > 0 && !p.withhold_loads) {
            const uint64_t pol_l = policy_evict_first();
            bool ok = true;
            int issued = l_pre;   // boxes issued (the first before the wait)
            for (int bi = l_pre; bi < 2 * nt; ++bi) {   // box bi = (tile bi / 2, half bi % 2) in stage bi % SL
                const int t = bi % SL, lap = bi / SL;
                if (lap > 0 && !mbar_wait(&lempty[t], (lap - 1) & 1, lim)) {
                    ok = false;
                    break;
                }
                issue_l_box(tmL, smem, lay, lfull, p, bi, t, MODE, MS, pol_l);
                ++issued;
            }
            if (!ok) fail_timeout(p);
            // every box issued has landed before the CTA may exit: stage t
            // was armed by the boxes t, t + SL, ... below `issued`
            for (int st = 0; st < SL && st < issued; ++st) mbar_wait(&lfull[st], ((issued - 1 - st) / SL) & 1, lim);
        }
        __syncwarp();
    } else {
        // 4. epilogue: thread = GEMM row (TMEM lane of its sub-partition
        //    warp % 4); column group g = (warp - 3) / 4 takes columns
        //    [16 g, 16 g + 16) of both 64-id boxes of every tile
        const int q = warp & 3;
        const int g = (warp - 3) >> 2;
        const int lrow = q * 32 + lane;
        const int grow = row0 + lrow;
        Epi<MODE> sts[MS];   // one row of each sub-tile
#pragma unroll
        for (int h = 0; h < MS; ++h) {
            sts[h].init(p, grow + h * kTileM);
            sts[h].group = g;
        }
        Epi<MODE>& st = sts[0];
        // the L row of each sub-tile's row in the staged L boxes (PCTree: one
        // per request, shared by its P frontier rows) and the L dtype
        int lr[MS];
#pragma unroll
        for (int h = 0; h < MS; ++h) lr[h] = mode_tree(MODE) ? (lrow + h * kTileM) / p.P : lrow + h * kTileM;
        const int lf = LF >= 0 ? LF : p.l_fp32;
        const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
        int t = 0, lap = 0;   // L ring slot and wraps
        for (int i = 0; i < nt; ++i) {
            const int b = i & 1;
            if constexpr (mode_loads_first(MODE)) {
                // the tile's L and target loads first (they do not wait on
                // the MMA), then one accumulator slice at a time
                const int v0 = (static_cast<int>(blockIdx.x) + i * static_cast<int>(gridDim.x)) * kTileN;
                const int vb[2] = {v0 + g * C, v0 + kBoxN + g * C};
                st.issue(p, vb);
                bool ok = mbar_wait(&tfull[b], (i >> 1) & 1, lim);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) {
                    if (lane == 0) fail_timeout(p);
                    break;
                }
                if (warp == 3 && lane == 0) mbar_arrive(&wdone[i % NTS]);
                tc_fence_after();
                uint32_t acc[C];
                tmem_ld16(lane_addr + static_cast<uint32_t>(b * kTileN + g * C), acc);
                tmem_ld_wait();
                st.consume_slice(p, vb[0], 0, acc);
                tmem_ld16(lane_addr + static_cast<uint32_t>(b * kTileN + kBoxN + g * C), acc);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tempty[b]);
                st.consume_slice(p, vb[1], 1, acc);
                continue;
            } else {
            // the tile's two L stages (one per 64-id box), shared by the sub-tiles
            const int t0 = t, lap0 = lap;
            const int t1 = (t0 + 1 == SL) ? 0 : t0 + 1, lap1 = (t0 + 1 == SL) ? lap0 + 1 : lap0;
            const int ts[2] = {t0, t1}, laps[2] = {lap0, lap1};
            const int v0 = (static_cast<int>(blockIdx.x) + i * static_cast<int>(gridDim.x)) * kTileN;
            bool ok = true;
            if constexpr (MS == 2) {
                // sub-tile h's accumulator: both 16-column slices into
                // registers, handed back to the MMA warp before the arithmetic
#pragma unroll
                for (int h = 0; h < MS; ++h) {
                    ok = __all_sync(0xffffffffu, mbar_wait(&tfull[h], i & 1, lim));
                    if (!ok) break;
                    // the tile's W stages are free once its last sub-tile's MMAs are done
                    if (h == MS - 1 && warp == 3 && lane == 0) mbar_arrive(&wdone[i % NTS]);
                    tc_fence_after();
                    uint32_t acc[2][C];
                    tmem_ld16(lane_addr + static_cast<uint32_t>(h * kTileN + g * C), acc[0]);
                    tmem_ld16(lane_addr + static_cast<uint32_t>(h * kTileN + kBoxN + g * C), acc[1]);
                    tmem_ld_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&tempty[h]);
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        if (mode_reads_l(MODE) && h == 0) {
                            ok = __all_sync(0xffffffffu, mbar_wait(&lfull[ts[hh]], laps[hh] & 1, lim));
                            if (!ok) break;
                        }
                        const uint8_t* sl = smem + lay.l_off + static_cast<uint32_t>(ts[hh]) * lay.l_stage_bytes;
                        sts[h].consume(p, sl, lay.l_box_bytes, lf, lr[h], v0 + hh * kBoxN + g * C, g, acc[hh]);
                        if (mode_reads_l(MODE) && h == MS - 1) {
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&lempty[ts[hh]]);
                        }
                    }
                    if (!ok) break;
                }
            } else {
                ok = __all_sync(0xffffffffu, mbar_wait(&tfull[b], (i >> 1) & 1, lim));
                if (ok) {
                    // the tile's W stages are free once its MMAs are done
                    if (warp == 3 && lane == 0) mbar_arrive(&wdone[i % NTS]);
                    tc_fence_after();
                    // both 16-column slices of the tile into registers, then
                    // the accumulator goes back to the MMA warp before any
                    // arithmetic
                    uint32_t acc[2][C];
                    tmem_ld16(lane_addr + static_cast<uint32_t>(b * kTileN + g * C), acc[0]);
                    tmem_ld16(lane_addr + static_cast<uint32_t>(b * kTileN + kBoxN + g * C), acc[1]);
                    tmem_ld_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&tempty[b]);
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        if (mode_reads_l(MODE)) {
                            ok = __all_sync(0xffffffffu, mbar_wait(&lfull[ts[hh]], laps[hh] & 1, lim));
                            if (!ok) break;
                        }
                        const uint8_t* sl = smem + lay.l_off + static_cast<uint32_t>(ts[hh]) * lay.l_stage_bytes;
                        st.consume(p, sl, lay.l_box_bytes, lf, lr[0], v0 + hh * kBoxN + g * C, g, acc[hh]);
                        if (mode_reads_l(MODE)) {
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&lempty[ts[hh]]);
                        }
                    }
                }
            }
            if (mode_reads_l(MODE)) {
                t = (t1 + 1 == SL) ? 0 : t1 + 1;
                lap = (t1 + 1 == SL) ? lap1 + 1 : lap1;
            }
            if (!ok) {
                if (lane == 0) fail_timeout(p);
                break;
            }
            }
        }
        if constexpr (MODE == MODE_TREE_LSE) {
            // one partial per row and CTA: the column groups' pairs meet in
            // shared memory (the rings are idle once every epilogue warp has
            // consumed its last tile), the first group merges and writes them
            float2* cmb = reinterpret_cast<float2*>(smem);   // [kColGroups][MS][kTileM]
#pragma unroll
            for (int h = 0; h < MS; ++h) cmb[(g * MS + h) * kTileM + lrow] = sts[h].partial();
            asm volatile("bar.sync 1, %0;" ::"r"(kEpiWarps * 32) : "memory");
            if (g == 0) {
#pragma unroll
                for (int h = 0; h < MS; ++h) {
                    float mm = -INFINITY;
#pragma unroll
                    for (int gg = 0; gg < kColGroups; ++gg) mm = fmaxf(mm, cmb[(gg * MS + h) * kTileM + lrow].x);
                    float ss = 0.f;
#pragma unroll
                    for (int gg = 0; gg < kColGroups; ++gg) {
                        const float2 x = cmb[(gg * MS + h) * kTileM + lrow];
                        if (x.y > 0.f) ss += x.y * fast_exp2((x.x - mm) * kLog2e);
                    }
                    if (sts[h].valid)
                        p.part[static_cast<size_t>(grow + h * kTileM) * p.n_part + blockIdx.x] =
                            make_float2(ss > 0.f ? mm : -INFINITY, ss);
                }
            }
        } else {
#pragma unroll
            for (int h = 0; h < MS; ++h) sts[h].flush(p, grow + h * kTileM);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

template <int MODE, int MS = 1, int LF = -1>
cudaError_t launch_mode(const CUtensorMap& tmW, const CUtensorMap& tmL, const GemmParams& p, int gx, int gy,
                        cudaStream_t s) {
    const SmemLayout lay = make_layout(p.r, p.l_rows, p.l_fp32, p.w_stages, p.l_stages, MODE, MS);
    // every sub-tile's A needs a W slot of its own, and the ring at least two
    if (lay.total > static_cast<uint32_t>(kSmemLimit) || p.w_stages < 2 * (p.r >> 6)) return cudaErrorInvalidValue;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(markov_gemm_kernel<MODE, MS, LF>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    return launch_pdl(markov_gemm_kernel<MODE, MS, LF>, dim3(gx, gy), dim3(kGemmThreads), lay.total, s, tmW, tmL, p);
}

}  // namespace

void gemm_pick_stages(GemmParams& p, int mode) {
    // W in whole tile slots (r / 64 stages each), at least two; then as many
    // L boxes as fit up to kMaxLStages (three tiles ahead: L comes from HBM
    // in scattered rows); then more W slots with what is left.
    const int kb = p.r >> 6;
    const int ms = p.m_sub > 1 ? p.m_sub : 1;
    const auto fits = [&](int ws, int ls) {
        return make_layout(p.r, p.l_rows, p.l_fp32, ws, ls, mode, ms).total <= static_cast<uint32_t>(kSmemLimit);
    };
    int ws = 2 * kb, ls = 0;
    if (mode_reads_l(mode))
        for (ls = kMaxLStages; ls > 2 && !fits(ws, ls); --ls) {
        }
    while (ws + kb <= kMaxWStages && fits(ws + kb, ls)) ws += kb;
    p.w_stages = ws;
    p.l_stages = ls;
}

cudaError_t launch_markov_gemm(int mode, const CUtensorMap& tmW, const CUtensorMap& tmL, const GemmParams& p,
                               int grid_x, int grid_y, cudaStream_t s) {
    switch (mode) {
        // the modes that stage L in shared memory: one kernel per L dtype
        case MODE_CHAIN_GREEDY:
            return p.l_fp32 ? launch_mode<MODE_CHAIN_GREEDY, 1, 1>(tmW, tmL, p, grid_x, grid_y, s)
                            : launch_mode<MODE_CHAIN_GREEDY, 1, 0>(tmW, tmL, p, grid_x, grid_y, s);
        case MODE_CHAIN_SAMPLE:
            return p.l_fp32 ? launch_mode<MODE_CHAIN_SAMPLE, 1, 1>(tmW, tmL, p, grid_x, grid_y, s)
                            : launch_mode<MODE_CHAIN_SAMPLE, 1, 0>(tmW, tmL, p, grid_x, grid_y, s);
        case MODE_TREE:
            return p.l_fp32 ? launch_mode<MODE_TREE, 1, 1>(tmW, tmL, p, grid_x, grid_y, s)
                            : launch_mode<MODE_TREE, 1, 0>(tmW, tmL, p, grid_x, grid_y, s);
        case MODE_RESID: return launch_mode<MODE_RESID>(tmW, tmL, p, grid_x, grid_y, s);
        case MODE_ABSMAX: return launch_mode<MODE_ABSMAX>(tmW, tmL, p, grid_x, grid_y, s);
        case MODE_QLSE: return launch_mode<MODE_QLSE>(tmW, tmL, p, grid_x, grid_y, s);
        case MODE_TVMIN: return launch_mode<MODE_TVMIN>(tmW, tmL, p, grid_x, grid_y, s);
        case MODE_TVMIN_B16: return launch_mode<MODE_TVMIN_B16>(tmW, tmL, p, grid_x, grid_y, s);
        case MODE_TVMIN_B32: return launch_mode<MODE_TVMIN_B32>(tmW, tmL, p, grid_x, grid_y, s);
        case MODE_TREE_LSE:
            if (p.m_sub == 2)
                return p.l_fp32 ? launch_mode<MODE_TREE_LSE, 2, 1>(tmW, tmL, p, grid_x, grid_y, s)
                                : launch_mode<MODE_TREE_LSE, 2, 0>(tmW, tmL, p, grid_x, grid_y, s);
            return p.l_fp32 ? launch_mode<MODE_TREE_LSE, 1, 1>(tmW, tmL, p, grid_x, grid_y, s)
                            : launch_mode<MODE_TREE_LSE, 1, 0>(tmW, tmL, p, grid_x, grid_y, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace sdm
