/*
 * paged_gqa.h -- C ABI of the GB300 (sm_103a) paged grouped-query attention
 * library: batched decode and selected-sparse prefill over a block-table KV
 * cache holding FP16 or FP8-E4M3 keys and values.
 *
 * The operations follow two 1Cat-vLLM pull requests:
 *   - "[Kernel][SM70] Scale NVFP4 E4M3 decode batches" (#282), Purpose:
 *     FP8-E4M3, GQA-6, head dim 256 paged decode for batches of 1..16, with
 *     wide KV loads, a packed E4M3 converter and long-context routes;
 *   - "[Kernel][SM70] Accelerate Qwen3.8 QSA paged prefill" (#378), Changes:
 *     selected-sparse prefill (Hq6/Hkv1/D256) where each query row attends to
 *     its selected four-token blocks, read in place from the page-16 cache,
 *     with its own causal partial block last; contiguous or interleaved K/V
 *     strides; block tables in physical-page units; stale positions clamped
 *     and invalid requests inert.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  * Pointers named as device data point to memory on the current CUDA
 *    device, owned by the caller.  The library never allocates device or host
 *    memory and never frees caller memory.  Between calls it keeps only a
 *    per-device cache of the SM count and kernel occupancy, so concurrent
 *    calls from several host threads are safe.
 *  * Every call is asynchronous on `stream` (a cudaStream_t; NULL means the
 *    legacy default stream) and never synchronises the host, so calls can be
 *    captured into CUDA graphs.
 *  * Return value: PAGED_GQA_OK (0) or a negative paged_gqa_status.  Argument
 *    errors are detected on the host before anything is launched.  A launch
 *    failure returns PAGED_GQA_ERR_CUDA.
 *  * Invalid data found on the device is inert rather than fatal (see the
 *    PAGED_GQA_FLAG_* bits): it never faults, never traps, and is reported
 *    by atomically ORing a bit into the optional device int `err_flag`.
 *  * FP16 means IEEE binary16; E4M3 means OCP FP8 E4M3FN (bias 7, no
 *    infinities, codes 0x7F/0xFF are NaN, largest finite 448).  An E4M3 KV
 *    value is code_value * kv_scale; FP16 KV ignores kv_scale.
 *  * KV layout: element d of the row of (page, slot, kv_head) lives at
 *        cache + page*page_stride + slot*token_stride + kv_head*head_stride + d
 *    (strides in elements of the KV type).  K and V share one layout, which
 *    covers separate contiguous pools and one interleaved buffer.
 *  * Logical token t of a sequence lives on page block_table_row[t / page_size]
 *    at slot t % page_size.  Block-table entries are physical page ids into the
 *    pool; ids outside [0, num_pages) are skipped.
 *  * Query head h reads KV head h / (Hq / Hkv) (consecutive groups).
 *  * Only head dim D = 256 and groups Hq / Hkv <= 8 are built.
 */
#ifndef PAGED_GQA_H
#define PAGED_GQA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PAGED_GQA_VERSION 1

/* Host-side status codes. */
typedef enum {
    PAGED_GQA_OK = 0,
    PAGED_GQA_ERR_NULL_POINTER = -1,  /* a required pointer is NULL              */
    PAGED_GQA_ERR_ALIGNMENT = -2,     /* a pointer or stride is not 16-byte aligned */
    PAGED_GQA_ERR_SHAPE = -3,         /* inconsistent or out-of-range sizes      */
    PAGED_GQA_ERR_UNSUPPORTED = -4,   /* D != 256, group > 8, unknown dtype ...  */
    PAGED_GQA_ERR_WORKSPACE = -5,     /* workspace too small or misaligned        */
    PAGED_GQA_ERR_CUDA = -6           /* a CUDA runtime call or launch failed     */
} paged_gqa_status;

/* Bits ORed into *err_flag by the kernels when they meet invalid data. */
#define PAGED_GQA_FLAG_BAD_PAGE     1  /* block-table entry outside [0, num_pages): its tokens skipped */
#define PAGED_GQA_FLAG_SEQ_CLAMPED  2  /* seq_len > max_seq_len: clamped to max_seq_len             */
#define PAGED_GQA_FLAG_EMPTY_ROW    4  /* seq_len <= 0 or q_pos < 0: that output row is zero         */
#define PAGED_GQA_FLAG_QPOS_CLAMPED 8  /* q_pos >= kv_len: clamped to kv_len - 1                     */
#define PAGED_GQA_FLAG_BAD_SEL     16  /* selected block at or after the row's own block: skipped   */
#define PAGED_GQA_FLAG_SCORES_SHORT 32  /* a selection row has more causal blocks than scores given  */
#define PAGED_GQA_FLAG_BAD_LOGIT   64  /* a masking row's largest logit is NaN or +inf: top-p skipped */
#define PAGED_GQA_FLAG_TIMEOUT    128  /* a kernel's bounded wait ran out (never expected); output invalid */

typedef enum {
    PAGED_GQA_KV_FP16 = 0,            /* binary16 K/V                            */
    PAGED_GQA_KV_E4M3 = 1             /* uint8 E4M3FN codes, times kv_scale      */
} paged_gqa_kv_dtype;

/* Strides of the K/V pools in elements of the KV type; the head-dim stride is
 * 1.  Each stride times the element size must be a multiple of 16 bytes. */
typedef struct {
    int64_t page_stride;
    int64_t token_stride;
    int64_t head_stride;
} paged_gqa_kv_layout;

/* Caller-owned scratch for split-KV decode.
 *  ptr/bytes     device buffer of at least paged_gqa_decode_workspace_size()
 *                bytes, 256-byte aligned.  ptr == NULL selects the unsplit
 *                route (one CTA per (sequence, KV head), no merge kernel).
 *  force_splits  0 = automatic; > 0 forces that many split CTAs (tests use it
 *                to check that the result does not depend on the split).
 *  err_flag      optional device int receiving PAGED_GQA_FLAG_* bits.
 *  split_events  optional pair of cudaEvent_t; when both are non-NULL the
 *                library records [0] before and [1] after the split kernel on
 *                `stream` (for timing that kernel alone). */
typedef struct {
    void* ptr;
    size_t bytes;
    int force_splits;
    int* err_flag;
    void* split_events[2];
} paged_gqa_workspace;

/*
 * Bytes of workspace paged_gqa_decode needs for this shape on the current
 * CUDA device (the split count depends on its SM count).  Returns 0 for
 * invalid shapes.  Pure host function: launches nothing.
 */
size_t paged_gqa_decode_workspace_size(int B, int Hq, int Hkv, int D, int max_seq_len);

/*
 * Bytes of workspace needed when paged_gqa_workspace.force_splits = splits
 * (splits > 0).  Returns 0 for invalid shapes.  Pure host function.
 */
size_t paged_gqa_decode_workspace_size_splits(int B, int Hq, int Hkv, int D, int splits);

/*
 * Batched paged decode ("[Kernel][SM70] Scale NVFP4 E4M3 decode batches",
 * Purpose).  For every sequence b and query head h, with L = min(seq_lens[b],
 * max_seq_len) and j = h / (Hq / Hkv):
 *     out[b, h, :] = sum_{t < L} softmax_t(softmax_scale * <q[b,h,:], K_t>) V_t
 * over the tokens t whose page is valid, K_t and V_t being rows of KV head j.
 *
 *  q            device, binary16 [B, Hq, D] contiguous, 16-byte aligned.
 *  k_cache,     device, K and V pools in `kv_layout`, of kv_dtype, 16-byte
 *  v_cache      aligned; num_pages pages of page_size tokens.
 *  block_table  device int32, row b at block_table + b * bt_row_stride, with at
 *               least ceil(max_seq_len / page_size) entries per row.
 *  seq_lens     device int32 [B].
 *  max_seq_len  host upper bound of seq_lens used to size the split; longer
 *               sequences are clamped (PAGED_GQA_FLAG_SEQ_CLAMPED).
 *  out          device, binary16 [B, Hq, D] contiguous, 16-byte aligned; fully
 *               written (zero rows for empty sequences).
 *  ws           see paged_gqa_workspace; NULL selects the unsplit route.
 * Two kernels are launched on the split route (split, then merge), one on
 * the unsplit route.  Results are deterministic for a given device, shape and
 * force_splits: no floating-point atomics are used.
 */
int paged_gqa_decode(const void* q, const void* k_cache, const void* v_cache,
                     paged_gqa_kv_layout kv_layout, int kv_dtype,
                     const int32_t* block_table, int64_t bt_row_stride,
                     const int32_t* seq_lens,
                     int B, int Hq, int Hkv, int D, int page_size, int num_pages,
                     int max_seq_len, float kv_scale, float softmax_scale,
                     void* out, const paged_gqa_workspace* ws, void* stream);

/*
 * paged_gqa_decode for callers that cannot allocate device memory.  The
 * pages have no counterpart of this entry point; it exists for users of this
 * library whose code runs where a cudaMalloc is forbidden or unwanted (an
 * execute hook of a host framework that owns all device memory, a
 * latency-critical path where an allocation could synchronise the device, a
 * process whose memory another allocator already holds).
 *
 * Same arguments and results as paged_gqa_decode with the split route, except
 * that there is no workspace argument: the split scratch lives in a 16 MiB
 * static device array inside this library (held on every GPU where the
 * library's device code is loaded, until the process exits) and the call
 * allocates nothing.  err_flag is the optional device int of
 * PAGED_GQA_FLAG_* bits.
 *  * Shapes whose split scratch for the given kv_dtype exceeds 16 MiB (the
 *    workspace paged_gqa_decode would need with its automatic split count
 *    for that dtype; never more than paged_gqa_decode_workspace_size()) are
 *    refused with PAGED_GQA_ERR_WORKSPACE before anything is launched.
 *    Batches above 4096 take the unsplit route and need no scratch.
 *  * The first call on each device looks up the array's device address with
 *    that device current.  Under the CUDA runtime's lazy module loading (its
 *    default) that lookup loads the library's device code on that device,
 *    which is when the 16 MiB is reserved: the first call can fail for lack
 *    of memory and can synchronise.  Make one warm-up call per device at
 *    initialisation, before any stream capture and outside any hook where
 *    allocation is not allowed; later calls allocate nothing.
 *  * Every call shares the array: calls whose kernels may overlap on the GPU
 *    (e.g. on unordered streams) race and give wrong results; calls ordered
 *    on one stream are safe.  No scratch value needs to start at zero.
 */
int paged_gqa_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                             paged_gqa_kv_layout kv_layout, int kv_dtype,
                             const int32_t* block_table, int64_t bt_row_stride,
                             const int32_t* seq_lens,
                             int B, int Hq, int Hkv, int D, int page_size, int num_pages,
                             int max_seq_len, float kv_scale, float softmax_scale,
                             void* out, int* err_flag, void* stream);

/*
 * Selected-sparse prefill over four-token blocks of one sequence ("[Kernel]
 * [SM70] Accelerate Qwen3.8 QSA paged prefill", Changes).  For query row r
 * with p = min(q_pos[r], kv_len - 1) and own = p / 4, the row attends to
 *     { 4b .. 4b+3 : b in sel_idx[r, :], 0 <= b < own }   (selected blocks)
 *  ++ { 4*own .. p }                                      (causal tail, last)
 * read in place from the page_size-token pages through block_table, and
 *     out[r, h, :] = sum_t softmax_t(softmax_scale * <q[r,h,:], K_t>) V_t.
 *
 *  q            device, binary16 [R, Hq, D] contiguous.
 *  k_cache,     device pools as for decode (FP16 or E4M3).
 *  v_cache
 *  block_table  device int32 [>= ceil(kv_len / page_size)], this sequence's pages.
 *  sel_idx      device int32 [R, n_sel]; entries < 0 are padding; entries >=
 *               own are skipped (PAGED_GQA_FLAG_BAD_SEL).  Order is free.
 *  q_pos        device int32 [R]; q_pos < 0 gives a zero row
 *               (PAGED_GQA_FLAG_EMPTY_ROW); q_pos >= kv_len is clamped
 *               (PAGED_GQA_FLAG_QPOS_CLAMPED).
 *  page_size    a multiple of 4, so a four-token block never straddles pages.
 *  out          device, binary16 [R, Hq, D] contiguous; fully written.
 * One kernel is launched; no workspace is needed.  The kernel route is the
 * automatic one of paged_gqa_sparse_prefill_route below.
 */
int paged_gqa_sparse_prefill(const void* q, const void* k_cache, const void* v_cache,
                             paged_gqa_kv_layout kv_layout, int kv_dtype,
                             const int32_t* block_table, int num_pages, int kv_len,
                             const int32_t* sel_idx, int n_sel, const int32_t* q_pos,
                             int R, int Hq, int Hkv, int D, int page_size,
                             float kv_scale, float softmax_scale,
                             void* out, int* err_flag, void* stream);

/*
 * paged_gqa_sparse_prefill with the kernel route chosen by the caller: the
 * same operation ("[Kernel][SM70] Accelerate Qwen3.8 QSA paged prefill",
 * Changes), arguments, layouts, inert rules and flags, computed by one of
 * two designs whose results agree within rounding:
 *  route = PAGED_GQA_PREFILL_AUTO     grouped when kv_len <= 131072 and,
 *                                     with C = R * Hkv: FP16, 64 * n_sel >=
 *                                     kv_len, or C >= 1024 and 2048 * n_sel
 *                                     >= kv_len; E4M3, C >= 1024 and
 *                                     36 * n_sel >= kv_len (enough rows and
 *                                     selections that row-group unions pay
 *                                     for the grouped route's fixed cost);
 *                                     per-row otherwise;
 *          PAGED_GQA_PREFILL_ROWWISE  one CTA per (row, KV head): each row's
 *                                     blocks are gathered for that row alone;
 *          PAGED_GQA_PREFILL_GROUPED  a pair of CTAs per group of consecutive
 *                                     rows of one KV head (128 query-head
 *                                     slots at most): the union of the
 *                                     group's blocks is gathered once into
 *                                     shared memory (half of it by each CTA)
 *                                     and each row masks the tokens it attends;
 *                                     tcgen05 tensor cores, TMEM accumulators
 *                                     (E4M3 rows are converted to binary16 as
 *                                     they are gathered).  kv_len <= 131072
 *                                     only (else PAGED_GQA_ERR_UNSUPPORTED).
 *  rows_per_group  grouped route: rows of one group, 1 .. 128 / (Hq / Hkv);
 *                  0 = sized to fill whole waves of the co-resident
 *                  pairs of CTAs (one CTA per SM, two per unit).
 * A listed block counts once per listing on both routes (duplicates are a
 * caller error; the grouped route recounts such rows on a slow path).
 */

#define PAGED_GQA_PREFILL_AUTO     0
#define PAGED_GQA_PREFILL_ROWWISE  1
#define PAGED_GQA_PREFILL_GROUPED  2
int paged_gqa_sparse_prefill_route(const void* q, const void* k_cache, const void* v_cache,
                                   paged_gqa_kv_layout kv_layout, int kv_dtype,
                                   const int32_t* block_table, int num_pages, int kv_len,
                                   const int32_t* sel_idx, int n_sel, const int32_t* q_pos,
                                   int R, int Hq, int Hkv, int D, int page_size,
                                   float kv_scale, float softmax_scale,
                                   void* out, int* err_flag, void* stream,
                                   int route, int rows_per_group);

/*
 * The kernel route PAGED_GQA_PREFILL_AUTO takes for this shape:
 * PAGED_GQA_PREFILL_ROWWISE or PAGED_GQA_PREFILL_GROUPED (the rule above,
 * for kv_dtype PAGED_GQA_KV_FP16 or PAGED_GQA_KV_E4M3), or a negative
 * status for invalid arguments.  Host only; launches nothing.  The pages
 * have no counterpart of this helper: it tells a caller which design its
 * calls run (for benchmarks and reports).
 */
int paged_gqa_sparse_prefill_auto_route(int R, int Hq, int Hkv, int kv_len, int n_sel,
                                        int kv_dtype);

/*
 * Test hook of the grouped route's failure path; the pages have no
 * counterpart of it.  Runs paged_gqa_sparse_prefill_route with route =
 * PAGED_GQA_PREFILL_GROUPED and rows_per_group = 0, except that every bounded
 * wait of the kernel gives up after spin_limit polls (0 = the library's
 * default of 2^20; at most 2^30) and, when stall_stage >= 0, that each CTA
 * leaves its ring stage number stall_stage (counted from the CTA's start)
 * unpublished, so the waits for it run out.  A CTA whose wait ran out skips
 * its remaining waits, lets the tensor-core work it issued complete, frees
 * its tensor memory and sets PAGED_GQA_FLAG_TIMEOUT in *err_flag; the output
 * is then undefined.  No fault, trap or endless wait is involved, and later
 * calls are unaffected.  Only tests of that path should call it.
 * Returns PAGED_GQA_ERR_SHAPE for spin_limit outside [0, 2^30] or
 * stall_stage < -1, else as paged_gqa_sparse_prefill_route.
 */
int paged_gqa_debug_grouped_prefill_stall(const void* q, const void* k_cache, const void* v_cache,
                                          paged_gqa_kv_layout kv_layout, int kv_dtype,
                                          const int32_t* block_table, int num_pages, int kv_len,
                                          const int32_t* sel_idx, int n_sel, const int32_t* q_pos,
                                          int R, int Hq, int Hkv, int D, int page_size,
                                          float kv_scale, float softmax_scale, void* out,
                                          int* err_flag, void* stream, long long spin_limit,
                                          int stall_stage);

/*
 * Rows per group of the grouped route for R query rows of Hq / Hkv heads on
 * the current device, given rows_per_group as passed to
 * paged_gqa_sparse_prefill_route (0 = automatic: groups sized so the units
 * fill whole waves of the co-resident CTA pairs, each pair one unit).
 * Returns the count, or a negative status: PAGED_GQA_ERR_SHAPE (R < 1,
 * Hq % Hkv != 0, rows_per_group out of range), PAGED_GQA_ERR_UNSUPPORTED
 * (more than 8 query heads per KV head),
 * PAGED_GQA_ERR_CUDA (no device to query).  Host only; launches nothing.
 * The pages have no counterpart of this helper: it tells a caller how the
 * grouped route partitions its rows (for sizing benchmarks and reports).
 */
int paged_gqa_sparse_prefill_group_rows(int R, int Hq, int Hkv, int rows_per_group);

/*
 * QSA block selection ("[Kernel][SM70] Accelerate exact Qwen3.8 decode",
 * Implementation: radix selection over the block scores, ties at the pivot
 * taken by increasing block index), producing the sel_idx rows that
 * paged_gqa_sparse_prefill consumes.  For query row r with
 * p = min(q_pos[r], kv_len - 1), the candidates are the blocks before the
 * row's own block, i = 0 .. n - 1 with n = min(p / 4, n_blocks), scored
 * scores[r * score_stride + i].  The row's output is the min(k, n) best
 * candidates -- greater score first under IEEE 754 totalOrder (-NaN < -inf
 * < ... < -0 < +0 < ... < +inf < +NaN), equal scores by increasing index --
 * listed in increasing index order, then -1 up to k entries.  The result is
 * exact (integer work on the scores' bit patterns) and deterministic.
 *
 *  scores        device float32; row r starts at scores + r * score_stride
 *                (score_stride >= n_blocks, in elements).
 *  n_blocks      scores per row; a row with p / 4 > n_blocks uses the first
 *                n_blocks (PAGED_GQA_FLAG_SCORES_SHORT).
 *  q_pos         device int32 [R]; q_pos < 0 (or kv_len <= 0) gives a row of
 *                -1 (PAGED_GQA_FLAG_EMPTY_ROW); q_pos >= kv_len is clamped
 *                (PAGED_GQA_FLAG_QPOS_CLAMPED).
 *  k             selected blocks per row (>= 0).
 *  sel_out       device int32 [R, k]; fully written.
 *  err_flag      optional device int receiving PAGED_GQA_FLAG_* bits.
 * One kernel is launched; nothing is allocated.
 */
int paged_gqa_select_blocks(const float* scores, int64_t score_stride, int n_blocks,
                            const int32_t* q_pos, int R, int kv_len, int k,
                            int32_t* sel_out, int* err_flag, void* stream);

/*
 * Combined top-k/top-p masking of the decode step's logits ("[Kernel][SM70]
 * Scale NVFP4 E4M3 decode batches", Purpose: B8/B16 x 248,320 logits, run at
 * top-k 20, top-p 0.95).  For each row of V logits: top-k keeps the min(k, V)
 * largest (equal logits: the lower index first); top-p keeps, of those in
 * that order, the shortest leading run whose probability mass reaches p, the
 * probabilities being the softmax over the top-k logits, computed in FP64:
 * e_j = exp(x_j - x_0), S_j = e_j + e_{j+1} + ... (the suffix sums of the
 * list, added in FP64 by a parallel scan: they may differ from a serial sum
 * from the end by a few units in the last place), logit j kept iff
 * S_j > (1 - p) S_0.  out = the kept logits, bit for bit, and -infinity
 * everywhere else.
 *
 *  logits        device float32; row b starts at logits + b * logits_stride
 *                (>= V, in elements).  Finite or -inf values; a row whose
 *                largest logit is NaN or +inf keeps its top-k list
 *                (PAGED_GQA_FLAG_BAD_LOGIT), a row of -inf stays -inf.
 *  out           device float32, row stride out_stride (>= V); fully written.
 *                out == logits (with equal strides) masks in place; any other
 *                overlap is not allowed.
 *  k             1 .. 128.
 *  p             0 < p <= 1 (p = 1: top-k alone).
 *  V             1 .. 327680.
 *  B             0 .. 2^27 rows (8 CTAs each).
 *  err_flag      optional device int receiving PAGED_GQA_FLAG_* bits.
 * One kernel is launched: a cluster of 8 CTAs per row; nothing is allocated.
 */
int paged_gqa_topk_topp_mask(const float* logits, int64_t logits_stride, float* out,
                             int64_t out_stride, int B, int V, int k, float p, int* err_flag,
                             void* stream);

/*
 * Inspection: the rows the decode kernels gather, dequantised.  For every
 * b < B, t < T and KV head j writes out[b, t, j, :] (float32, device,
 * [B, T, Hkv, D]) = the stored row of logical token t of sequence b as a
 * float (E4M3 code value times kv_scale, rounded once; FP16 exactly), or
 * zeros when t >= min(seq_lens[b], max_seq_len) or its page is invalid.  Uses
 * the decode kernels' own address arithmetic and E4M3 converter, so tests can
 * compare the gather and the dequantisation bit for bit.
 */
int paged_gqa_gather_dequant(const void* cache, paged_gqa_kv_layout kv_layout, int kv_dtype,
                             const int32_t* block_table, int64_t bt_row_stride,
                             const int32_t* seq_lens, int B, int T, int Hkv, int D,
                             int page_size, int num_pages, int max_seq_len, float kv_scale,
                             float* out, void* stream);

/*
 * Inspection: the token list the sparse-prefill kernel builds for each row.
 * out is device int32 [R, 4 * (n_sel + 1)]: slot 4*i + u holds the logical
 * token of lane u of block entry i (entries 0..n_sel-1 are sel_idx[r, i],
 * entry n_sel is the row's causal tail block), or -1 when that slot is not
 * attended.  Uses the prefill kernel's own index arithmetic.
 */
int paged_gqa_sparse_prefill_tokens(const int32_t* block_table, int num_pages, int kv_len,
                                    const int32_t* sel_idx, int n_sel, const int32_t* q_pos,
                                    int R, int page_size, int32_t* out, void* stream);

/*
 * Measurement helper; the pages have no counterpart of it.  Runs the gather
 * of the per-row sparse-prefill kernel (PAGED_GQA_PREFILL_ROWWISE) alone:
 * every row's selected four-token blocks and causal tail, K and V rows,
 * copied through the same shared-memory rings with the same launch shape,
 * entry table and inert rules, and each copied row read once from shared
 * memory, with no attention arithmetic.  Its time is the ceiling of that
 * gather on the device, the bound the per-row route is measured against.
 *  arguments    as for paged_gqa_sparse_prefill (no q, no softmax scales).
 *  out          device uint32 [R, Hkv]: the XOR of every 32-bit word of the
 *               K and V rows row r attends through KV head j (0 for a row
 *               that attends nothing), so tests can check the gather exactly.
 * One kernel is launched; nothing is allocated.
 */
int paged_gqa_sparse_gather_probe(const void* k_cache, const void* v_cache,
                                  paged_gqa_kv_layout kv_layout, int kv_dtype,
                                  const int32_t* block_table, int num_pages, int kv_len,
                                  const int32_t* sel_idx, int n_sel, const int32_t* q_pos, int R,
                                  int Hkv, int D, int page_size, uint32_t* out, void* stream);

/* Human-readable name of a status code (static string). */
const char* paged_gqa_status_string(int status);

/* PAGED_GQA_VERSION of the loaded library. */
int paged_gqa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGED_GQA_H */
