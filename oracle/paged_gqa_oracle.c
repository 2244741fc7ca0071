/*
 * paged_gqa_oracle.c -- plain, slow FP64 CPU oracle for paged grouped-query
 * attention over a block-table KV cache holding FP16 or FP8-E4M3 keys/values.
 *
 * TEST INFRASTRUCTURE ONLY.  The product path never includes, links or calls
 * this file: only the test suite, the package smoke check and the benchmark's
 * CPU-baseline leg load it.  It shares no code, header, table or helper with
 * the CUDA library.
 *
 * What it computes, and the passages it follows (1Cat-vLLM pull requests):
 *
 *   [D] "[Kernel][SM70] Scale NVFP4 E4M3 decode batches" (#282), Purpose:
 *       batched paged decode, FP8-E4M3 KV, GQA-6 (six query heads share one
 *       KV head), head dim 256, over a paged-KV layout.
 *   [P] "[Kernel][SM70] Accelerate Qwen3.8 QSA paged prefill" (#378), Changes:
 *       selected-sparse prefill, Hq6/Hkv1/D256 FP16, each query row attending
 *       to its selected four-token blocks with its own causal partial block
 *       last; block tables in physical-page units; contiguous or interleaved
 *       K/V strides; padded or stale positions clamped to the live length and
 *       invalid requests made inert.
 *   [D] also lists, as the decode step's second operator, the combined
 *       top-k/top-p masking of B8/B16 x 248,320 logits (Purpose; run with
 *       top-k 20, top-p 0.95 in the Performance contract; compared bitwise
 *       against its rollback in Test plan and result).
 *   [S] "[Kernel][SM70] Accelerate exact Qwen3.8 decode" (#415),
 *       Implementation and Focused tests: QSA's block selection, a radix
 *       selection over the block scores whose ties at the pivot go to the
 *       lower block index, checked for GPU exactness; its output is the
 *       selected-block list that [P] consumes.
 *
 * The method is exact softmax attention over a defined token set, so this
 * oracle is that definition written out in FP64:
 *     x_t = s * sum_d q[d] * K_t[d]
 *     w_t = exp(x_t - max_u x_u) / sum_u exp(x_u - max_u x_u)
 *     o   = sum_t w_t * V_t          then rounded once to FP16 (nearest-even).
 * K_t and V_t are the exact values of the stored codes: FP16 -> FP64 exactly,
 * or E4M3 code -> E(c) * kv_scale in FP64 (exact: a 4-bit significand times a
 * 24-bit one fits in 53 bits).
 *
 * Readings taken where the pages are silent:
 *   - query head h uses KV head floor(h / G), G = Hq / Hkv (consecutive groups);
 *   - one kv_scale per call multiplies both K and V codes; unused for FP16;
 *   - E4M3 is the OCP E4M3FN variant: no infinities, codes 0x7F/0xFF are NaN,
 *     largest finite magnitude 448;
 *   - a decode query attends to all seq_len tokens of its sequence;
 *   - inert rules: seq_len <= 0 gives a zero output row; seq_len above
 *     max_seq_len is clamped to max_seq_len; a token whose block-table entry is
 *     outside [0, num_pages) is skipped; a row with no attendable token is zero;
 *   - sparse prefill: q_pos < 0 gives a zero row; q_pos >= kv_len is clamped to
 *     kv_len - 1; the tail is tokens 4*floor(p/4) .. p; a selected block b is
 *     used only if 0 <= b < floor(p/4) (negative entries are padding, entries at
 *     or after the tail block are skipped as non-causal); duplicates count twice.
 *
 * Status flags (ORed into *flags when flags != NULL) use their own constants
 * below; the tests compare them with the library's documented bit values.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_FLAG_BAD_PAGE     1  /* a block-table entry outside [0, num_pages)  */
#define ORC_FLAG_SEQ_CLAMPED  2  /* seq_len > max_seq_len, clamped               */
#define ORC_FLAG_EMPTY_ROW    4  /* seq_len <= 0 or q_pos < 0: zero output row   */
#define ORC_FLAG_QPOS_CLAMPED 8  /* q_pos >= kv_len, clamped to kv_len - 1       */
#define ORC_FLAG_BAD_SEL     16  /* selected block at/after the tail block       */
#define ORC_FLAG_SCORES_SHORT 32  /* a row's candidates exceed the scores given   */

/* ------------------------------------------------------------------------- */
/* Number formats                                                              */
/* ------------------------------------------------------------------------- */

/* IEEE 754 binary16 -> double, from the format definition:
 * sign bit 15, 5-bit exponent (bias 15), 10-bit fraction. */
double orc_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int f = h & 0x3FF;
    double mag;
    if (e == 0)
        mag = ldexp((double)f, -24);                 /* subnormal: f * 2^-24  */
    else if (e == 31)
        mag = (f == 0) ? INFINITY : NAN;
    else
        mag = ldexp(1.0 + (double)f / 1024.0, e - 15);
    return sign ? -mag : mag;
}

/* double -> binary16, round to nearest, ties to even; overflow to infinity. */
uint16_t orc_f64_to_f16(double x)
{
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (isnan(x))
        return 0x7E00;
    if (a >= 65520.0)                      /* halfway above 65504 rounds up   */
        return sign | 0x7C00;
    if (a < ldexp(1.0, -14)) {             /* subnormal range: units of 2^-24 */
        double q = nearbyint(ldexp(a, 24)); /* default mode: nearest-even     */
        return sign | (uint16_t)q;         /* q == 1024 is the smallest normal */
    }
    int E;
    double m = frexp(a, &E);               /* a = m * 2^E, m in [0.5, 1)       */
    int e = E - 1;                         /* a = (2m) * 2^e, 2m in [1, 2)     */
    double q = nearbyint(ldexp(m, 11));    /* significand in units of 2^-10   */
    if (q >= 2048.0) { q = 1024.0; e += 1; }
    if (e > 15)
        return sign | 0x7C00;
    return sign | (uint16_t)((e + 15) << 10) | (uint16_t)((int)q - 1024);
}

/* OCP FP8 E4M3FN code -> double, from the format definition:
 * sign bit 7, 4-bit exponent (bias 7), 3-bit mantissa; exponent field 0 is
 * subnormal (f * 2^-9); exponent 15 with mantissa 7 is NaN; no infinities. */
double orc_e4m3_to_f64(uint8_t c)
{
    int sign = (c >> 7) & 1;
    int e = (c >> 3) & 0xF;
    int f = c & 0x7;
    double mag;
    if (e == 15 && f == 7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)f, -9);
    else
        mag = ldexp(1.0 + (double)f / 8.0, e - 7);
    return sign ? -mag : mag;
}

/* ------------------------------------------------------------------------- */
/* KV cache access                                                            */
/* ------------------------------------------------------------------------- */

typedef struct {
    const void* base;        /* K or V pool                                   */
    int is_e4m3;             /* 1: uint8 E4M3 codes, 0: binary16 bits         */
    int64_t page_stride;     /* in elements of the stored type                */
    int64_t token_stride;
    int64_t head_stride;
    double scale;            /* kv_scale for E4M3, 1 for FP16                 */
} orc_pool;

/* Value of element d of the row stored at (page, slot, head). */
static double pool_value(const orc_pool* p, int64_t page, int64_t slot, int64_t head, int64_t d)
{
    int64_t off = page * p->page_stride + slot * p->token_stride + head * p->head_stride + d;
    if (p->is_e4m3)
        return orc_e4m3_to_f64(((const uint8_t*)p->base)[off]) * p->scale;
    return orc_f16_to_f64(((const uint16_t*)p->base)[off]);
}

/* Logical token t of a sequence whose block-table row is bt_row: the physical
 * page is bt_row[t / page_size] and the slot in it t mod page_size.
 * Returns the page, or -1 if the entry is outside [0, num_pages). */
static int64_t token_page(const int32_t* bt_row, int64_t t, int page_size, int num_pages)
{
    int64_t page = bt_row[t / page_size];
    if (page < 0 || page >= num_pages)
        return -1;
    return page;
}

/* ------------------------------------------------------------------------- */
/* Softmax attention of one query head over an explicit token list            */
/* ------------------------------------------------------------------------- */

/* tokens[n] are logical token indices (all with valid pages).  Writes D values
 * of the FP64 output; an empty list gives zeros. */
static void attend(const double* q, int D, const orc_pool* K, const orc_pool* V,
                   const int32_t* bt_row, int page_size, int num_pages, int kv_head,
                   const int64_t* tokens, int64_t n, double softmax_scale,
                   double* x /* scratch [n] */, double* o /* [D] out */)
{
    for (int d = 0; d < D; ++d)
        o[d] = 0.0;
    if (n == 0)
        return;
    double m = -INFINITY;
    for (int64_t i = 0; i < n; ++i) {
        int64_t t = tokens[i];
        int64_t page = token_page(bt_row, t, page_size, num_pages);
        int64_t slot = t % page_size;
        double dot = 0.0;
        for (int d = 0; d < D; ++d)
            dot += q[d] * pool_value(K, page, slot, kv_head, d);
        x[i] = softmax_scale * dot;
        if (x[i] > m)
            m = x[i];
    }
    double l = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        x[i] = exp(x[i] - m);
        l += x[i];
    }
    for (int64_t i = 0; i < n; ++i) {
        int64_t t = tokens[i];
        int64_t page = token_page(bt_row, t, page_size, num_pages);
        int64_t slot = t % page_size;
        double w = x[i] / l;
        for (int d = 0; d < D; ++d)
            o[d] += w * pool_value(V, page, slot, kv_head, d);
    }
}

static void or_flag(int* flags, int bit)
{
    if (flags) {
#pragma omp atomic
        *flags |= bit;
    }
}

/* ------------------------------------------------------------------------- */
/* Batched paged decode  ([D])                                                */
/* ------------------------------------------------------------------------- */

/*
 * q        [B, Hq, D] binary16 bits, contiguous.
 * k, v     pools (uint8 E4M3 codes or binary16 bits), element (page, slot,
 *          head, d) at page*page_stride + slot*token_stride + head*head_stride + d.
 * block_table  row b at block_table + b*bt_row_stride, >= ceil(max_seq_len /
 *          page_size) entries used.
 * pairs    optional list of n_pairs (b, h) pairs (2 ints each) to compute; NULL
 *          computes every (b, h).  Rows not computed are left untouched.
 * out_f16  [B, Hq, D] binary16 bits (nearest-even of the FP64 result); may be NULL.
 * out_f64  [B, Hq, D] FP64 result before rounding; may be NULL.
 * Returns 0, or -1 on a shape the oracle does not accept.
 */
int orc_decode(const uint16_t* q, const void* k, const void* v, int kv_is_e4m3,
               int64_t page_stride, int64_t token_stride, int64_t head_stride,
               const int32_t* block_table, int64_t bt_row_stride, const int32_t* seq_lens,
               int B, int Hq, int Hkv, int D, int page_size, int num_pages, int max_seq_len,
               double kv_scale, double softmax_scale,
               const int32_t* pairs, int n_pairs,
               uint16_t* out_f16, double* out_f64, int* flags, int n_threads)
{
    if (B < 0 || Hkv < 1 || Hq < Hkv || Hq % Hkv != 0 || D < 1 || page_size < 1 ||
        max_seq_len < 0)
        return -1;
    int G = Hq / Hkv;
    orc_pool K = {k, kv_is_e4m3, page_stride, token_stride, head_stride, kv_is_e4m3 ? kv_scale : 1.0};
    orc_pool V = {v, kv_is_e4m3, page_stride, token_stride, head_stride, kv_is_e4m3 ? kv_scale : 1.0};
    int64_t total = pairs ? n_pairs : (int64_t)B * Hq;

#pragma omp parallel for schedule(dynamic, 1) num_threads(n_threads > 0 ? n_threads : 1)
    for (int64_t it = 0; it < total; ++it) {
        int b = pairs ? pairs[2 * it] : (int)(it / Hq);
        int h = pairs ? pairs[2 * it + 1] : (int)(it % Hq);
        int j = h / G;
        const int32_t* bt_row = block_table + (int64_t)b * bt_row_stride;
        int64_t L = seq_lens[b];
        if (L > max_seq_len) {
            or_flag(flags, ORC_FLAG_SEQ_CLAMPED);
            L = max_seq_len;
        }
        if (L <= 0) {
            or_flag(flags, ORC_FLAG_EMPTY_ROW);
            L = 0;
        }
        int64_t* tokens = (int64_t*)malloc(sizeof(int64_t) * (size_t)(L > 0 ? L : 1));
        double* x = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
        double* qd = (double*)malloc(sizeof(double) * (size_t)D);
        double* o = (double*)malloc(sizeof(double) * (size_t)D);
        int64_t n = 0;
        for (int64_t t = 0; t < L; ++t) {
            if (token_page(bt_row, t, page_size, num_pages) < 0) {
                or_flag(flags, ORC_FLAG_BAD_PAGE);
                continue;
            }
            tokens[n++] = t;
        }
        const uint16_t* qrow = q + ((int64_t)b * Hq + h) * D;
        for (int d = 0; d < D; ++d)
            qd[d] = orc_f16_to_f64(qrow[d]);
        attend(qd, D, &K, &V, bt_row, page_size, num_pages, j, tokens, n, softmax_scale, x, o);
        int64_t ob = ((int64_t)b * Hq + h) * D;
        for (int d = 0; d < D; ++d) {
            if (out_f16) out_f16[ob + d] = orc_f64_to_f16(o[d]);
            if (out_f64) out_f64[ob + d] = o[d];
        }
        free(tokens); free(x); free(qd); free(o);
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Selected-sparse prefill over four-token blocks  ([P])                      */
/* ------------------------------------------------------------------------- */

/*
 * One sequence of kv_len tokens whose block table is block_table[0 ..].
 * q        [R, Hq, D] binary16 bits.
 * sel_idx  [R, n_sel] four-token block ids (block b = tokens 4b .. 4b+3).
 * q_pos    [R] position of each query row.
 * rows     optional list of n_rows row indices to compute (NULL: all R).
 * Token list of row r with p = q_pos[r] (after the inert rules above):
 *     { 4b + i : b in sel_idx[r], 0 <= b < floor(p/4), i = 0..3 }
 *  ++ { 4*floor(p/4), ..., p }                      (causal partial block last)
 * then the decode formula with KV head floor(h / G).
 */
int orc_sparse_prefill(const uint16_t* q, const void* k, const void* v, int kv_is_e4m3,
                       int64_t page_stride, int64_t token_stride, int64_t head_stride,
                       const int32_t* block_table, int num_pages, int kv_len,
                       const int32_t* sel_idx, int n_sel, const int32_t* q_pos,
                       int R, int Hq, int Hkv, int D, int page_size,
                       double kv_scale, double softmax_scale,
                       const int32_t* rows, int n_rows,
                       uint16_t* out_f16, double* out_f64, int* flags, int n_threads)
{
    if (R < 0 || n_sel < 0 || Hkv < 1 || Hq < Hkv || Hq % Hkv != 0 || D < 1 ||
        page_size < 1 || page_size % 4 != 0)
        return -1;
    int G = Hq / Hkv;
    orc_pool K = {k, kv_is_e4m3, page_stride, token_stride, head_stride, kv_is_e4m3 ? kv_scale : 1.0};
    orc_pool V = {v, kv_is_e4m3, page_stride, token_stride, head_stride, kv_is_e4m3 ? kv_scale : 1.0};
    int64_t total = (int64_t)(rows ? n_rows : R) * Hq;

#pragma omp parallel for schedule(dynamic, 1) num_threads(n_threads > 0 ? n_threads : 1)
    for (int64_t it = 0; it < total; ++it) {
        int r = rows ? rows[it / Hq] : (int)(it / Hq);
        int h = (int)(it % Hq);
        int j = h / G;
        int64_t cap = 4 * (int64_t)n_sel + 4;
        int64_t* tokens = (int64_t*)malloc(sizeof(int64_t) * (size_t)cap);
        double* x = (double*)malloc(sizeof(double) * (size_t)cap);
        double* qd = (double*)malloc(sizeof(double) * (size_t)D);
        double* o = (double*)malloc(sizeof(double) * (size_t)D);
        int64_t n = 0;
        int64_t p = q_pos[r];
        if (p < 0 || kv_len <= 0) {
            or_flag(flags, ORC_FLAG_EMPTY_ROW);
        } else {
            if (p >= kv_len) {
                or_flag(flags, ORC_FLAG_QPOS_CLAMPED);
                p = kv_len - 1;
            }
            int64_t own = p / 4;                       /* the tail's block   */
            for (int i = 0; i < n_sel; ++i) {
                int64_t b = sel_idx[(int64_t)r * n_sel + i];
                if (b < 0)
                    continue;                          /* padding           */
                if (b >= own) {
                    or_flag(flags, ORC_FLAG_BAD_SEL);  /* not before the tail */
                    continue;
                }
                for (int64_t t = 4 * b; t < 4 * b + 4; ++t) {
                    if (token_page(block_table, t, page_size, num_pages) < 0) {
                        or_flag(flags, ORC_FLAG_BAD_PAGE);
                        continue;
                    }
                    tokens[n++] = t;
                }
            }
            for (int64_t t = 4 * own; t <= p; ++t) {   /* causal tail, last  */
                if (token_page(block_table, t, page_size, num_pages) < 0) {
                    or_flag(flags, ORC_FLAG_BAD_PAGE);
                    continue;
                }
                tokens[n++] = t;
            }
        }
        const uint16_t* qrow = q + ((int64_t)r * Hq + h) * D;
        for (int d = 0; d < D; ++d)
            qd[d] = orc_f16_to_f64(qrow[d]);
        attend(qd, D, &K, &V, block_table, page_size, num_pages, j, tokens, n, softmax_scale, x, o);
        int64_t ob = ((int64_t)r * Hq + h) * D;
        for (int d = 0; d < D; ++d) {
            if (out_f16) out_f16[ob + d] = orc_f64_to_f16(o[d]);
            if (out_f64) out_f64[ob + d] = o[d];
        }
        free(tokens); free(x); free(qd); free(o);
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Gathered, dequantised rows (for the bit-exact gather comparison)           */
/* ------------------------------------------------------------------------- */

/*
 * out [B, T, Hkv, D] float: for t < min(seq_len, max_seq_len) with a valid
 * page, the stored row's values (E(c) * kv_scale rounded once to float, or
 * the FP16 value); every other entry is 0.
 */
int orc_gather_rows(const void* cache, int is_e4m3,
                    int64_t page_stride, int64_t token_stride, int64_t head_stride,
                    const int32_t* block_table, int64_t bt_row_stride, const int32_t* seq_lens,
                    int B, int T, int Hkv, int D, int page_size, int num_pages, int max_seq_len,
                    double kv_scale, float* out, int n_threads)
{
    if (B < 0 || T < 0 || Hkv < 1 || D < 1 || page_size < 1)
        return -1;
    orc_pool P = {cache, is_e4m3, page_stride, token_stride, head_stride, is_e4m3 ? kv_scale : 1.0};
#pragma omp parallel for schedule(static) num_threads(n_threads > 0 ? n_threads : 1)
    for (int64_t bt = 0; bt < (int64_t)B * T; ++bt) {
        int b = (int)(bt / T);
        int64_t t = bt % T;
        int64_t L = seq_lens[b];
        if (L > max_seq_len) L = max_seq_len;
        const int32_t* bt_row = block_table + (int64_t)b * bt_row_stride;
        int64_t page = (t < L) ? token_page(bt_row, t, page_size, num_pages) : -1;
        for (int j = 0; j < Hkv; ++j) {
            float* dst = out + ((bt * Hkv) + j) * D;
            for (int d = 0; d < D; ++d)
                dst[d] = (page < 0) ? 0.0f : (float)pool_value(&P, page, t % page_size, j, d);
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* The token list of one sparse-prefill row (for the bit-exact index check)   */
/* ------------------------------------------------------------------------- */

/*
 * Writes the logical tokens row r attends to, in the order used above
 * (selected blocks in sel_idx order, then the causal tail), skipping tokens
 * whose page is invalid.  Returns the count, or -1 if cap is too small.
 */
int64_t orc_sparse_row_tokens(const int32_t* block_table, int num_pages, int kv_len,
                              const int32_t* sel_row, int n_sel, int32_t q_pos,
                              int page_size, int64_t* tokens, int64_t cap)
{
    int64_t n = 0;
    int64_t p = q_pos;
    if (p < 0 || kv_len <= 0)
        return 0;
    if (p >= kv_len)
        p = kv_len - 1;
    int64_t own = p / 4;
    for (int i = 0; i < n_sel; ++i) {
        int64_t b = sel_row[i];
        if (b < 0 || b >= own)
            continue;
        for (int64_t t = 4 * b; t < 4 * b + 4; ++t) {
            if (token_page(block_table, t, page_size, num_pages) < 0)
                continue;
            if (n >= cap)
                return -1;
            tokens[n++] = t;
        }
    }
    for (int64_t t = 4 * own; t <= p; ++t) {
        if (token_page(block_table, t, page_size, num_pages) < 0)
            continue;
        if (n >= cap)
            return -1;
        tokens[n++] = t;
    }
    return n;
}

/* ------------------------------------------------------------------------- */
/* QSA block selection [S]                                                     */
/* ------------------------------------------------------------------------- */
/*
 * The result the radix selection of [S] reaches is a plain top-k, so the
 * oracle is that definition written out: sort a row's candidate blocks best
 * first (greater score first, equal scores by increasing block index), keep
 * the first min(k, n), and list them by increasing block index, padded with
 * -1 to k entries.
 *
 * Readings taken where the pages are silent:
 *   - the candidates of a row at position p are the blocks strictly before its
 *     own block, 0 .. floor(p / 4) - 1, the blocks [P] accepts in a selection;
 *     p is q_pos clamped to kv_len - 1 as in [P] (ORC_FLAG_QPOS_CLAMPED);
 *   - q_pos < 0 or kv_len <= 0 gives a row of -1 (ORC_FLAG_EMPTY_ROW);
 *   - only the n_blocks scores a row provides can be candidates
 *     (ORC_FLAG_SCORES_SHORT when floor(p / 4) > n_blocks);
 *   - scores are binary32 compared by IEEE 754 totalOrder, which orders every
 *     bit pattern: -NaN < -inf < negatives < -0 < +0 < positives < +inf < +NaN.
 */

/* totalOrder of two binary32 values given by their bit patterns: a value
 * with the sign bit set is below one without; among values without it, a
 * larger encoding (greater magnitude, then infinity, then NaN payloads) is
 * greater, and among values with it the larger encoding is smaller.
 * Returns -1 (a below b), 0 (same pattern) or 1. */
static int orc_total_order_cmp(uint32_t a, uint32_t b)
{
    const int neg_a = (int)(a >> 31), neg_b = (int)(b >> 31);
    if (neg_a != neg_b)
        return neg_a ? -1 : 1;
    if (a == b)
        return 0;
    if (!neg_a)
        return a < b ? -1 : 1;
    return a > b ? -1 : 1;
}

typedef struct {
    uint32_t bits;   /* the score's bit pattern */
    int32_t idx;     /* its block index */
} orc_cand;

/* qsort order of candidates: best first; equal scores by increasing index. */
static int orc_cand_best_first(const void* x, const void* y)
{
    const orc_cand* a = (const orc_cand*)x;
    const orc_cand* b = (const orc_cand*)y;
    const int c = orc_total_order_cmp(a->bits, b->bits);
    if (c != 0)
        return -c;
    return (a->idx > b->idx) - (a->idx < b->idx);
}

static int orc_int32_ascending(const void* x, const void* y)
{
    const int32_t a = *(const int32_t*)x, b = *(const int32_t*)y;
    return (a > b) - (a < b);
}

/* scores: R rows of score_stride floats, the first n_blocks of each used;
 * q_pos int32 [R]; sel_out int32 [R, k].  Returns 0, -1 on bad shapes or -2
 * when memory runs out. */
int orc_select_blocks(const float* scores, int64_t score_stride, int n_blocks,
                      const int32_t* q_pos, int R, int kv_len, int k, int32_t* sel_out,
                      int* flags, int n_threads)
{
    if (R < 0 || k < 0 || n_blocks < 0 || score_stride < n_blocks)
        return -1;
    int fl = 0, oom = 0;
#pragma omp parallel for num_threads(n_threads) schedule(dynamic, 8) reduction(|:fl, oom)
    for (int r = 0; r < R; ++r) {
        int32_t* out = sel_out + (int64_t)r * k;
        for (int i = 0; i < k; ++i)
            out[i] = -1;
        int64_t p = q_pos[r];
        if (p < 0 || kv_len <= 0) {
            fl |= ORC_FLAG_EMPTY_ROW;
            continue;
        }
        if (p >= kv_len) {
            fl |= ORC_FLAG_QPOS_CLAMPED;
            p = kv_len - 1;
        }
        int64_t n = p / 4;                      /* blocks strictly before its own */
        if (n > n_blocks) {
            fl |= ORC_FLAG_SCORES_SHORT;
            n = n_blocks;
        }
        if (n == 0 || k == 0)
            continue;
        orc_cand* cand = (orc_cand*)malloc((size_t)n * sizeof(orc_cand));
        int32_t* pick = (int32_t*)malloc((size_t)n * sizeof(int32_t));
        if (cand == NULL || pick == NULL) {
            free(cand);
            free(pick);
            oom = 1;
            continue;
        }
        const float* row = scores + (int64_t)r * score_stride;
        for (int64_t i = 0; i < n; ++i) {
            memcpy(&cand[i].bits, &row[i], sizeof(uint32_t));
            cand[i].idx = (int32_t)i;
        }
        qsort(cand, (size_t)n, sizeof(orc_cand), orc_cand_best_first);
        const int64_t m = n < k ? n : k;
        for (int64_t i = 0; i < m; ++i)
            pick[i] = cand[i].idx;
        qsort(pick, (size_t)m, sizeof(int32_t), orc_int32_ascending);
        memcpy(out, pick, (size_t)m * sizeof(int32_t));
        free(cand);
        free(pick);
    }
    if (flags != NULL)
        *flags |= fl;
    return oom ? -2 : 0;
}

/* ------------------------------------------------------------------------- */
/* Combined top-k / top-p masking [D]                                          */
/* ------------------------------------------------------------------------- */
/*
 * For each row of V logits: top-k keeps the min(k, V) largest logits (equal
 * logits: the lower index first, the tie rule of [S]); top-p then keeps, of
 * those in that order, the shortest leading run whose probability mass
 * reaches p, the probabilities being the softmax over the top-k logits; every
 * logit not kept becomes -infinity, kept logits pass through unchanged.
 *
 * Readings taken where the pages are silent:
 *   - top-k keeps exactly min(k, V) logits, ties to the lower index;
 *   - the top-p mass is computed in FP64: e_j = exp(x_j - x_0) over the
 *     top-k list in order (x_0 its largest), suffix sums S_j = e_j + S_{j+1}
 *     accumulated from the end of the list, Z = S_0; logit j is kept iff
 *     S_j > (1 - p) Z, i.e. iff the mass of the logits before it is < p Z;
 *   - a row whose largest logit is -infinity keeps its top-k list as is;
 *   - logits are finite or -infinity (NaN and +infinity are outside the
 *     contract and rejected here).
 * margin (optional, [B]) receives min_j |S_j - (1 - p) Z| / Z: how far the
 * row's top-p decisions are from their threshold.
 */

typedef struct {
    float x;
    int32_t idx;
} orc_logit;

/* Descending value, equal values by increasing index. */
static int orc_logit_desc(const void* a_, const void* b_)
{
    const orc_logit* a = (const orc_logit*)a_;
    const orc_logit* b = (const orc_logit*)b_;
    if (a->x != b->x)
        return a->x > b->x ? -1 : 1;
    return (a->idx > b->idx) - (a->idx < b->idx);
}

/* Returns 0, -1 on bad arguments, -2 when memory runs out, -3 on a NaN or
 * +infinity logit. */
int orc_topk_topp_mask(const float* logits, int64_t stride, int B, int V, int k, double p,
                       float* out, int64_t out_stride, double* margin, int n_threads)
{
    if (B < 0 || V < 1 || k < 1 || stride < V || out_stride < V || !(p > 0.0 && p <= 1.0))
        return -1;
    int bad = 0;
#pragma omp parallel for num_threads(n_threads) schedule(dynamic, 1) reduction(|:bad)
    for (int b = 0; b < B; ++b) {
        const float* x = logits + (int64_t)b * stride;
        float* o = out + (int64_t)b * out_stride;
        orc_logit* l = (orc_logit*)malloc((size_t)V * sizeof(orc_logit));
        if (l == NULL) {
            bad |= 2;
            continue;
        }
        int finite = 1;
        for (int i = 0; i < V; ++i) {
            if (isnan(x[i]) || (isinf(x[i]) && x[i] > 0))
                finite = 0;
            l[i].x = x[i];
            l[i].idx = i;
        }
        if (!finite) {
            free(l);
            bad |= 4;
            continue;
        }
        qsort(l, (size_t)V, sizeof(orc_logit), orc_logit_desc);
        const int K = k < V ? k : V;
        int m = K;
        double mg = INFINITY;
        if (l[0].x != -INFINITY) {
            double* S = (double*)malloc((size_t)(K + 1) * sizeof(double));
            if (S == NULL) {
                free(l);
                bad |= 2;
                continue;
            }
            const double x0 = (double)l[0].x;
            S[K] = 0.0;
            for (int j = K - 1; j >= 0; --j)
                S[j] = exp((double)l[j].x - x0) + S[j + 1];
            const double Z = S[0], cut = (1.0 - p) * Z;
            m = 0;
            for (int j = 0; j < K; ++j) {
                if (S[j] > cut)
                    m = j + 1;
                const double d = fabs(S[j] - cut) / Z;
                if (d < mg)
                    mg = d;
            }
            free(S);
        }
        for (int i = 0; i < V; ++i)
            o[i] = -INFINITY;
        for (int j = 0; j < m; ++j)
            o[l[j].idx] = l[j].x;
        if (margin != NULL)
            margin[b] = mg;
        free(l);
    }
    if (bad & 2)
        return -2;
    if (bad & 4)
        return -3;
    return 0;
}
