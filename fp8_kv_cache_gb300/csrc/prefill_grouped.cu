// prefill_grouped.cu -- selected-sparse paged prefill with grouped query rows
// on the fifth-generation tensor cores (FP16 or E4M3 KV; the tensor cores see
// binary16 tiles either way).
//
// Operation: "[Kernel][SM70] Accelerate Qwen3.8 QSA paged prefill"
// (1Cat-vLLM #378), Changes: query row r with p = min(q_pos[r], kv_len - 1)
// attends to its selected four-token blocks strictly before its own block,
// then to its own block up to p, read in place from the paged cache;
// padding, non-causal selections and invalid pages are inert.
//
// Design (ours, GB300-first).  The per-row kernel of prefill.cu reads each
// row's ~2050 tokens on its own: at 4096 rows that is 8.6 GB pulled from L2
// for a 32 MiB cache, and the gather, not the arithmetic, bounds it.  Nearby
// rows select many of the same blocks, so here a unit -- a group of
// consecutive rows of one KV head, up to 128 query-head slots, the M of one
// tcgen05 MMA -- streams the UNION of its rows' blocks once.  Persistent CTAs,
// one per SM, run in clusters of two: both CTAs of a pair take the same unit,
// each half of its 64-token half-tiles, and combine their results at the end.
//   * setup: the unit's selection rows, its Q rows and (when it fits) the
//     block table are staged in the idle ring by cp.async; the rows' valid
//     entries are OR-ed into a bitmap over the sequence's blocks; a prefix
//     popcount ranks the union; each row gets a 16-bit mask per 64-token
//     stage saying which of the stage's 16 blocks it attends (its own block
//     limited to positions <= p); Q goes to TMEM.
//   * 5 producer warps take turns over a 6-stage ring, gathering whole
//     stages (K and V of 64 tokens, in the order K0 K1 V0 K2 V1 ...) into the
//     128-byte-swizzled K-major tile (see tc_device.cuh): FP16 rows by 16-byte
//     cp.async, E4M3 codes by cp.async into the slot and converted in place.
//   * two threads in two warps issue S = Q K^T (M = 128 slots, N = 64
//     tokens, K = 256; Q from TMEM, K from the stage), one for the even and
//     one for the odd stages, each into its own TMEM score buffer as soon as
//     that buffer is free, and a thread of a third warp issues O += P V
//     (M = 128, N = 256, K = 64; P from TMEM, V from the stage bytes read as
//     an MN-major operand) into a 256-column TMEM accumulator, its first two
//     K steps once the first half of a stage's probabilities is written and
//     the last two once all are, so Q K^T runs ahead of the softmax without
//     waiting behind P V.  Each issuer counts its own phases of every
//     ring slot (K barriers per parity, a V barrier per slot), so no waiter
//     ever runs two phases ahead of a barrier.
//   * 8 softmax warps in two warpgroups that take alternate stages (A the
//     even ones, B the odd ones), so one group's exponentials and stores
//     overlap the other's score reads.  A thread owns one slot (its TMEM
//     lane) and all 64 score columns of its group's stage: it reads the
//     scores, masks them, and takes the running reference maximum from the
//     other group's previous stage (a named-barrier handoff per lane
//     quarter, the only link between the groups).  The reference grows only
//     when a stage's maximum exceeds it by more than 2^8, and then O is
//     rescaled in TMEM; each group keeps its own sum under the reference it
//     last saw, so the result is exact up to rounding.  The FP16
//     probabilities go back into TMEM over the first 32 columns of the
//     stage's score buffer (its scores are in registers by then), so no
//     shared memory holds P and the ring has a sixth slot; a score buffer is
//     reused by Q K^T once P V has read the P in it.
//   * the pair: each CTA sends its partner the unnormalised O of the
//     dimensions the partner writes, with its (m, l), through distributed
//     shared memory; each combines the two halves of its 128 dimensions.
// Masked-out (slot, token) pairs cost tensor-core work but no memory traffic;
// on the 4096-row workload (18-row units) the union is 0.52 of the per-row
// gather.  Units are sized to fill whole waves of the co-resident CTA pairs
// and are dealt in snake order (later rows have longer prefixes).
//
// Duplicated selections (a caller error) keep their meaning -- a block listed
// c times counts c times -- through a slow per-row recount.
#include <algorithm>
#include <atomic>

#include "pgqa_internal.h"
#include "tc_device.cuh"

namespace pgqa {
namespace grp {

constexpr int kM = kGroupSlots;               // query-head slots of a group (MMA M)
constexpr int kStageTokens = 64;             // tokens per stage: 16 four-token blocks
constexpr int kStageBlocks = 16;
constexpr int kNS = 6;                       // ring stages
constexpr int kRegionBytes = kStageTokens * 128;      // 64 head-dim columns of a stage
constexpr int kStageBytes = kStageTokens * kD * 2;    // 32 KB
constexpr int kMaskWords = 4096;             // 16 KB of per-row stage masks
constexpr int kSoftWarps = 8, kMmaWarp = 8, kProdWarps = 5, kProdWarp0 = 9;
constexpr int kPvWarp = kProdWarp0 + kProdWarps;   // issues P V
constexpr int kQkWarp1 = kPvWarp + 1;               // with kMmaWarp: Q K^T of odd / even stages
constexpr int kThreads = 32 * (kSoftWarps + 1 + kProdWarps + 2);
constexpr int kGroupThreads = kSoftWarps / 2 * 32;   // one softmax warpgroup
constexpr float kRescaleSlack = 8.f;         // log2-domain growth tolerated before rescaling O
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemQ = 0;               // Q: 128 columns of f16 pairs
constexpr uint32_t kTmemS = 128;             // S buffers at 128 and 192 (64 columns each);
                                             // P of a stage overwrites its first 32 columns
constexpr uint32_t kTmemO = 256;             // O: 256 f32 columns

struct Smem {
    unsigned char ring[kNS][kStageBytes];
    uint32_t bitmap[kGroupMaxWords];         // union of the group's blocks
    int rank[kGroupMaxWords];                // exclusive prefix popcount of bitmap
    uint32_t masks[kMaskWords];              // [row][stage / 2]: two 16-bit stage masks per word
    int row_p[kM], row_own[kM], row_rank_own[kM], row_dup[kM];
    float mref[kM];                          // [slot]: reference maximum handed between the groups
    float xl[2][kM];                         // [group][slot]: final sums exchanged
    float xml[kM][2];                        // [slot]: the partner CTA's final reference and sum
    // K stage loaded (by the parity of its half-tile in the unit), V stage
    // loaded, slot free.
    uint64_t full_k[2][kNS], full_v[kNS], empty[kNS];
    // Stages taken so far from each ring slot by each MMA thread ([0], [1]:
    // the Q K^T threads of even and odd half-tiles, [2]: P V).  Each kind of
    // stage publishes on its own barrier, so every consumer waits for every
    // phase of its barriers in order: a parity wait is only unambiguous
    // while its barrier is at most one phase behind.
    uint32_t taken[3][kNS];
    // Uses of each ring slot published so far.  Consecutive uses of a slot
    // come from different producer warps (stage it: warp it % kProdWarps,
    // slot it % kNS), so the producer of use u first waits until use u - 1
    // is published: its producer had waited for use u - 2 to be consumed,
    // which keeps the slot's empty barrier at most one phase behind the
    // parity this producer waits for.
    uint32_t slot_pub[kNS];
    // S written; P's first 32 tokens written (p_half) and all of P (p_full);
    // P V done reading P.
    uint64_t s_full[2], p_half[2], p_full[2], p_free[2], done;
    uint32_t tmem_base;
    int flags, n_union, abort;
    long spin_limit;
};

constexpr size_t kSmemBytes = sizeof(Smem) + 1024;   // + alignment of the tiles
static_assert(kSmemBytes <= 232448, "shared memory above the per-CTA opt-in limit");

// Where a unit's loop stands; every role walks the same sequence, so the
// global counters agree between roles without communication.
struct Cursor {
    uint32_t it = 0;    // ring stage counter
    uint32_t g = 0;     // half-tile (S/P buffer) counter
};



// Bounded wait; after any wait of the CTA has timed out, waits are skipped
// (every role keeps its control flow, so all barriers are still reached and
// the kernel ends; the result is then garbage and PAGED_GQA_FLAG_TIMEOUT set).
__device__ __forceinline__ void wait_or_abort(Smem& sm, uint64_t* bar, uint32_t par)
{
    volatile int* ab = &sm.abort;
    if (*ab)
        return;
    if (!tc::mbar_wait(bar, par, sm.spin_limit))
        *ab = 1;
}

// Bounded wait until `uses` uses of ring slot s are published (a counter
// other producer warps of this CTA write); skipped, like the mbarrier waits,
// once any wait of the CTA has timed out.
__device__ __forceinline__ void wait_published(Smem& sm, int s, uint32_t uses)
{
    volatile int* ab = &sm.abort;
    const volatile uint32_t* pub = &sm.slot_pub[s];
    for (long n = 0; !*ab && *pub < uses; ++n) {
        if (n >= sm.spin_limit) {
            *ab = 1;
            return;
        }
        __nanosleep(64);
    }
}

__device__ __forceinline__ bool page_valid_block(const KVGeom& g, const int32_t* bt, int b,
                                                 int& page, int& slot)
{
    int pi;
    page_and_slot(g, 4 * b, pi, slot);
    page = __ldg(bt + pi);
    return page >= 0 && page < g.num_pages;
}

// Block of entry e of group row rl (selected blocks, then the own block), or
// -1 when the entry is not attended.  Setup has built the union bitmap and
// taken the blocks with invalid pages out of it (raising their flag then),
// so the bitmap stands in for the page-table check.
__device__ __forceinline__ int entry_block_in_union(const GroupArgs& ga, const Smem& sm, int r0,
                                                    int rl, int e)
{
    const PrefillArgs& a = ga.a;
    const int own = sm.row_own[rl];
    if (own < 0)
        return -1;
    int b = own;
    if (e < a.n_sel) {
        b = __ldg(a.sel + (size_t)(r0 + rl) * a.n_sel + e);
        if (b < 0 || b >= own)
            return -1;
    }
    return (sm.bitmap[b >> 5] >> (b & 31)) & 1u ? b : -1;
}

__device__ __forceinline__ int rank_of_block(const Smem& sm, int b)
{
    const int w = b >> 5;
    return sm.rank[w] + __popc(sm.bitmap[w] & ((1u << (b & 31)) - 1u));
}

// The union block of rank k (k < n_union).
__device__ __forceinline__ int block_of_rank(const Smem& sm, int nbw, int k)
{
    int lo = 0, hi = nbw - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (sm.rank[mid] <= k)
            lo = mid;
        else
            hi = mid - 1;
    }
    return 32 * lo + (int)__fns(sm.bitmap[lo], 0, k - sm.rank[lo] + 1);
}

// Stage masks of the half-tiles (64-token tiles: one K and one V stage each)
// [ht0, ht0 + cap) for every row of the group, built by the 256 softmax
// threads (named barrier 1).  A block already present in a row's mask is a
// duplicated selection: the row is marked.
__device__ void build_masks(const GroupArgs& ga, Smem& sm, int r0, int Rg, int ht0, int cap,
                            int words_per_row)
{
    const int t = threadIdx.x;
    asm volatile("bar.sync 1, %0;" ::"n"(kSoftWarps * 32) : "memory");   // old masks read
    for (int i = t; i < Rg * words_per_row; i += kSoftWarps * 32)
        sm.masks[i] = 0u;
    asm volatile("bar.sync 1, %0;" ::"n"(kSoftWarps * 32) : "memory");
    const int n_ent = ga.a.n_sel + 1;
#pragma unroll 4
    for (int idx = t; idx < Rg * n_ent; idx += kSoftWarps * 32) {
        const int rl = idx / n_ent, e = idx - rl * n_ent;
        const int b = entry_block_in_union(ga, sm, r0, rl, e);
        if (b < 0)
            continue;
        const int k = rank_of_block(sm, b), ht = (k >> 4) - ht0;
        if (ht < 0 || ht >= cap)
            continue;
        const uint32_t bit = 1u << (((ht & 1) << 4) + (k & 15));
        const uint32_t old = atomicOr(&sm.masks[rl * words_per_row + (ht >> 1)], bit);
        if (old & bit)
            sm.row_dup[rl] = 1;
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kSoftWarps * 32) : "memory");
}

// Setup stages its inputs in the ring, idle between units: the Q rows of
// the unit's slots in the first 64 KB (slot s's 32 chunks of 16 bytes at
// 512 s + 16 (c ^ (s & 31)), so a warp reading one chunk of 32 slots is free
// of bank conflicts), the sequence's block table when it has at most
// kBtStage entries, then its selection entries (row-major, as in memory), at
// most kSelStage at a time.
constexpr int kStageQBytes = kM * kD * 2;
constexpr int kBtStage = 4096;
constexpr int kSelOffset = kStageQBytes + 4 * kBtStage;
constexpr int kSelStage = (kNS * kStageBytes - kSelOffset) / 4 - 4;

// cp.async of entries [c0, c0 + n) of the unit's selection rows into the
// ring; the staged copy keeps the source's offset modulo 16 bytes.  Returns
// where entry c0 lands.
__device__ __forceinline__ const int32_t* stage_sel(const PrefillArgs& a, Smem& sm, int r0, int c0,
                                                    int n)
{
    const int32_t* src = a.sel + (size_t)r0 * a.n_sel + c0;
    unsigned char* dst = &sm.ring[0][0] + kSelOffset + (reinterpret_cast<uintptr_t>(src) & 15u);
    const uint32_t d0 = tc::smem_addr(dst);
    for (int i = threadIdx.x; i < n; i += kThreads)
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(d0 + 4u * i), "l"(src + i)
                     : "memory");
    return reinterpret_cast<const int32_t*>(dst);
}

// A thread's share of entries [0, n) of the unit's selection rows, flattened
// row-major: a contiguous run, so consecutive entries of a (usually sorted)
// row let it gather its bitmap and mask bits per word before one atomic.
struct EntryRun {
    int i, i1, rl, e;
    __device__ EntryRun(const PrefillArgs& a, int c0, int n)
    {
        const int per = (n + kThreads - 1) / kThreads;
        i = min(n, (int)threadIdx.x * per);
        i1 = min(n, i + per);
        rl = (c0 + i) / max(a.n_sel, 1);
        e = (c0 + i) - rl * a.n_sel;
    }
    __device__ void next(const PrefillArgs& a)
    {
        ++i;
        if (++e == a.n_sel) {
            e = 0;
            ++rl;
        }
    }
};

// Whether block b's page is valid, from the staged block table.
__device__ __forceinline__ bool staged_page_ok(const PrefillArgs& a, const int32_t* btab, int b)
{
    int pi, slot;
    page_and_slot(a.kv, 4 * b, pi, slot);
    const int page = btab[pi];
    return page >= 0 && page < a.kv.num_pages;
}

// Selected entries [c0, c0 + n) of the unit, staged at st, OR-ed into the
// union bitmap (padding and rows without a position skipped; a block at or
// after its row's own block is flagged and skipped; with the block table
// staged at btab, so is a block whose page is invalid).
__device__ __forceinline__ void union_entries(const PrefillArgs& a, Smem& sm, const int32_t* st,
                                              int c0, int n, int& flags, const int32_t* btab)
{
#pragma unroll 4
    for (int i = threadIdx.x; i < n; i += kThreads) {
        const int rl = (c0 + i) / a.n_sel;
        const int own = sm.row_own[rl], b = st[i];
        if (own < 0 || b < 0)
            continue;
        if (b >= own) {
            flags |= PAGED_GQA_FLAG_BAD_SEL;
            continue;
        }
        if (btab != nullptr && !staged_page_ok(a, btab, b)) {
            flags |= PAGED_GQA_FLAG_BAD_PAGE;
            continue;
        }
        atomicOr(&sm.bitmap[b >> 5], 1u << (b & 31));
    }
}

// Stage masks of half-tiles [ht0, ht0 + cap) from the staged entries of a
// unit whose entries all fit in one staging (the masks are zero): the same
// masks as build_masks, built by all threads, each over a run of entries
// with one atomic per mask word it touches.
__device__ void staged_masks(const PrefillArgs& a, Smem& sm, const int32_t* st, int Rg, int ht0,
                             int cap, int words_per_row)
{
    const int n_all = Rg * a.n_sel;
    EntryRun r(a, 0, n_all);
    int cw = -1, crl = 0;                    // the mask word being gathered, its row, its bits
    uint32_t cb = 0u;
    const auto flush = [&]() {
        if (cb) {
            const uint32_t old = atomicOr(&sm.masks[cw], cb);
            if (old & cb)
                sm.row_dup[crl] = 1;
        }
    };
    for (int own = r.i < r.i1 ? sm.row_own[r.rl] : -1; r.i < r.i1;) {
        const int b = st[r.i];
        if (own >= 0 && b >= 0 && b < own && ((sm.bitmap[b >> 5] >> (b & 31)) & 1u)) {
            const int k = rank_of_block(sm, b), ht = (k >> 4) - ht0;
            if (ht >= 0 && ht < cap) {
                const int wi = r.rl * words_per_row + (ht >> 1);
                const uint32_t bit = 1u << (((ht & 1) << 4) + (k & 15));
                if (wi != cw) {
                    flush();
                    cw = wi;
                    crl = r.rl;
                    cb = 0u;
                }
                if (cb & bit)                // listed twice in this run
                    sm.row_dup[r.rl] = 1;
                cb |= bit;
            }
        }
        const int rl = r.rl;
        r.next(a);
        if (r.rl != rl && r.i < r.i1)
            own = sm.row_own[r.rl];
    }
    flush();
    if (threadIdx.x < Rg) {                  // the own blocks (their pages were checked)
        const int rl = threadIdx.x, b = sm.row_own[rl];
        if (b >= 0 && ((sm.bitmap[b >> 5] >> (b & 31)) & 1u)) {
            const int k = rank_of_block(sm, b), ht = (k >> 4) - ht0;
            if (ht >= 0 && ht < cap) {
                const uint32_t bit = 1u << (((ht & 1) << 4) + (k & 15));
                const uint32_t old = atomicOr(&sm.masks[rl * words_per_row + (ht >> 1)], bit);
                if (old & bit)
                    sm.row_dup[rl] = 1;
            }
        }
    }
}

// Everything a unit needs before its first stage: row positions, the union
// bitmap and its ranks, the Q tile, the first window of masks.  All threads.
// The selection entries, Q and (when it fits) the block table are fetched by
// cp.async in one round trip.
__device__ void unit_setup(const GroupArgs& ga, Smem& sm, int r0, int Rg, int j, int nbw,
                           int words_per_row, int cap, uint32_t crank)
{
    const PrefillArgs& a = ga.a;
    const int tid = threadIdx.x;
    const int n_all = Rg * a.n_sel;
    const int n_chunks = (n_all + kSelStage - 1) / kSelStage;
    if (tid == 0) {
        sm.flags = 0;
        sm.n_union = 0;
    }
    for (int w = tid; w < nbw; w += kThreads)
        sm.bitmap[w] = 0u;
    for (int i = tid; i < Rg * words_per_row; i += kThreads)
        sm.masks[i] = 0u;
    {                                        // Q rows: the G heads of KV head j are contiguous
        const uint32_t q0 = tc::smem_addr(&sm.ring[0][0]);
        for (int i = tid; i < Rg * a.G * 32; i += kThreads) {
            const int slot = i >> 5, c = i & 31, rl = slot / a.G, h = slot - rl * a.G;
            cp_async16(q0 + 512u * slot + 16u * (c ^ (slot & 31)),
                       reinterpret_cast<const unsigned char*>(
                           a.q + ((size_t)(r0 + rl) * a.Hq + (size_t)j * a.G + h) * kD + 8 * c));
        }
    }
    const int32_t* st = stage_sel(a, sm, r0, 0, min(n_all, kSelStage));
    // the block table, for the page checks, when it fits
    const int n_bt = a.kv_len > 0 ? (int)(((int64_t)a.kv_len + a.kv.page_size - 1) / a.kv.page_size) : 0;
    const bool bt_staged = n_bt <= kBtStage;
    const int32_t* btab = reinterpret_cast<const int32_t*>(&sm.ring[0][0] + kStageQBytes);
    if (bt_staged) {
        const uint32_t d0 = tc::smem_addr(&sm.ring[0][0] + kStageQBytes);
        for (int i = tid; i < n_bt; i += kThreads)
            asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(d0 + 4u * i), "l"(a.bt + i)
                         : "memory");
    }
    cp_async_commit();
    if (tid < Rg) {
        int p = __ldg(a.q_pos + r0 + tid), fl = 0, own = -1;
        if (p < 0 || a.kv_len <= 0) {
            fl |= PAGED_GQA_FLAG_EMPTY_ROW;
        } else {
            if (p >= a.kv_len) {
                p = a.kv_len - 1;
                fl |= PAGED_GQA_FLAG_QPOS_CLAMPED;
            }
            own = p >> 2;
        }
        sm.row_p[tid] = p;
        sm.row_own[tid] = own;
        sm.row_rank_own[tid] = -1;
        sm.row_dup[tid] = 0;
        if (fl)
            atomicOr(&sm.flags, fl);
    }
    cp_async_wait<0>();
    __syncthreads();

    // The union; with the block table staged, each entry's page is checked
    // as it joins, else each union block's page once afterwards (an invalid
    // one leaves the union and raises BAD_PAGE, as its entries would have).
    int flags = 0;
    const int32_t* bt_s = bt_staged ? btab : nullptr;
    if (tid < Rg && sm.row_own[tid] >= 0) {      // the own block
        const int b = sm.row_own[tid];
        if (bt_s == nullptr || staged_page_ok(a, bt_s, b))
            atomicOr(&sm.bitmap[b >> 5], 1u << (b & 31));
        else
            flags |= PAGED_GQA_FLAG_BAD_PAGE;
    }
    union_entries(a, sm, st, 0, min(n_all, kSelStage), flags, bt_s);
    for (int c = 1; c < n_chunks; ++c) {         // entries beyond one staging
        __syncthreads();
        const int c0 = c * kSelStage, n = min(n_all - c0, kSelStage);
        st = stage_sel(a, sm, r0, c0, n);
        cp_async_commit();
        cp_async_wait<0>();
        __syncthreads();
        union_entries(a, sm, st, c0, n, flags, bt_s);
    }
    if (!bt_staged) {                        // one page check per union block
        __syncthreads();
        const int nb = 32 * nbw;
        for (int b0 = tid; b0 < nb; b0 += 8 * kThreads) {
            int page[8];
            uint32_t in = 0u;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int b = b0 + k * kThreads;
                page[k] = 0;
                if (b < nb && ((sm.bitmap[b >> 5] >> (b & 31)) & 1u)) {
                    int pi, slot;
                    page_and_slot(a.kv, 4 * b, pi, slot);
                    page[k] = __ldg(a.bt + pi);
                    in |= 1u << k;
                }
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int b = b0 + k * kThreads;
                if (((in >> k) & 1u) && (page[k] < 0 || page[k] >= a.kv.num_pages)) {
                    atomicAnd(&sm.bitmap[b >> 5], ~(1u << (b & 31)));
                    flags |= PAGED_GQA_FLAG_BAD_PAGE;
                }
            }
        }
    }
    if (flags)
        atomicOr(&sm.flags, flags);
    __syncthreads();

    if (tid < 32) {                          // exclusive scan of the word popcounts
        const int per = (nbw + 31) >> 5, w0 = tid * per, w1 = min(nbw, w0 + per);
        int sum = 0;
        for (int w = w0; w < w1; ++w)
            sum += __popc(sm.bitmap[w]);
        int inc = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, inc, o);
            if (tid >= o)
                inc += v;
        }
        int run = inc - sum;
        for (int w = w0; w < w1; ++w) {
            sm.rank[w] = run;
            run += __popc(sm.bitmap[w]);
        }
        if (tid == 31)
            sm.n_union = inc;
    }
    __syncthreads();

    if (tid < Rg) {
        const int own = sm.row_own[tid];
        if (own >= 0 && ((sm.bitmap[own >> 5] >> (own & 31)) & 1u))
            sm.row_rank_own[tid] = rank_of_block(sm, own);
    }
    if (tid < kSoftWarps * 32) {             // Q into TMEM: lane = slot = (row slot / G, head slot % G)
        // The softmax takes its scores in units of |score scale|: a negative
        // scale is folded into Q by negating it, a zero scale by a zero Q
        // (both exact), so that the kernel's score scale is positive.
        const uint32_t q_xor = a.scale_log2 < 0.f ? 0x80008000u : 0u;
        const uint32_t q_and = a.scale_log2 == 0.f ? 0u : 0xFFFFFFFFu;
        const int slot = tid & (kM - 1), half = tid >> 7;         // two threads per slot
        const int rl = slot / a.G;
        const bool live = rl < Rg && sm.row_own[rl] >= 0;
        const uint32_t qs = tc::smem_addr(&sm.ring[0][0]) + 512u * slot;
        const uint32_t tl = sm.tmem_base + ((uint32_t)(32 * ((tid >> 5) & 3)) << 16);
#pragma unroll 1
        for (int part = 0; part < 2; ++part) {   // 8 chunks of 16 bytes = 32 columns of f16 pairs
            uint32_t w[32];
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const int chunk = 16 * half + 8 * part + c;
                const uint4 v = live ? lds128(qs + 16u * (chunk ^ (slot & 31)))
                                     : make_uint4(0u, 0u, 0u, 0u);
                w[4 * c] = (v.x ^ q_xor) & q_and;
                w[4 * c + 1] = (v.y ^ q_xor) & q_and;
                w[4 * c + 2] = (v.z ^ q_xor) & q_and;
                w[4 * c + 3] = (v.w ^ q_xor) & q_and;
            }
            tc::tmem_st32(tl + kTmemQ + 64 * half + 32 * part, w);
        }
        tc::tmem_wait_st();
    }
    const int nt = (sm.n_union + kStageBlocks - 1) / kStageBlocks;
    const int ht0 = crank ? nt / 2 : 0;
    if (n_chunks <= 1)
        staged_masks(a, sm, st, Rg, ht0, cap, words_per_row);
    else if (tid < kSoftWarps * 32)
        build_masks(ga, sm, r0, Rg, ht0, cap, words_per_row);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
}

// Stage q of a unit with nt half-tiles, in ring order: the K stages of the
// first kKLead half-tiles, then V0, K(kKLead), V1, K(kKLead + 1), ..., and
// the last V stages.  Q K^T of half-tile h runs once the softmax has read
// the scores of h - 2 (two score buffers), so K stages loaded further ahead
// only wait in the ring; leads of 2 to 5 half-tiles measured within 3 % of
// each other on the 4096-row workload, 2 the fastest.
constexpr int kKLead = 2;

__device__ __forceinline__ void stage_of(int q, int nt, bool& is_v, int& ht)
{
    const int lead = nt < kKLead ? nt : kKLead;
    if (q < lead) {
        is_v = false;
        ht = q;
        return;
    }
    const int r = q - lead, pairs = 2 * (nt - lead);
    if (r < pairs) {
        is_v = (r & 1) == 0;
        ht = is_v ? r >> 1 : (r >> 1) + kKLead;
    } else {
        is_v = true;
        ht = r - pairs + (nt - lead);
    }
}

// Byte offset (K and V share it) of the first row of block lane (lanes
// 0 .. 15) of the stage of half-tile ht, or -1 past the union or on other
// lanes.
__device__ __forceinline__ int64_t stage_block_offset(const GroupArgs& ga, const Smem& sm, int j,
                                                      int nbw, int n_union, int ht, int lane)
{
    int64_t off = -1;
    if (lane < kStageBlocks) {
        const int k = kStageBlocks * ht + lane;
        if (k < n_union) {
            const int b = block_of_rank(sm, nbw, k);
            int page, slot;
            page_valid_block(ga.a.kv, ga.a.bt, b, page, slot);
            off = row_offset(ga.a.kv, page, slot, j);
        }
    }
    return off;
}

// Producer warps: warp pw fills the stages it = pw, pw + kProdWarps, ... of
// the ring (slot it % kNS; the warp waits until the slot's previous use is
// published, then consumed): lanes 0..15 resolve the
// stage's 16 blocks (rank -> block -> page) in parallel, for the warp's next
// stage while the current one's copies are in flight.  FP16 rows: each lane
// copies its 16-byte chunk of all 64 rows with cp.async and waits for its
// own copies.  E4M3 rows (256 codes, half the bytes): the codes go by
// cp.async into the upper half of the slot, all in flight at once; the warp
// then holds codes 128..255 in registers, converts codes 0..127 exactly to
// binary16 (hardware converter) into the lower half of the tile layout, and
// after a warp barrier writes the held half over the raw codes.  The warp then
// fences its writes for the tensor cores and publishes the stage on the
// barrier of its kind; stages of different warps are in flight together.
template <bool kE4M3>
__device__ void produce(const GroupArgs& ga, Smem& sm, Cursor& cur, int j, int nbw, int nt,
                        int h0, int n_union)
{
    const PrefillArgs& a = ga.a;
    const int lane = threadIdx.x & 31, pw = (threadIdx.x >> 5) - kProdWarp0;
    const uint32_t it0 = cur.it;
    const int n = 2 * nt;
    int q = (pw - (int)(it0 % kProdWarps) + kProdWarps) % kProdWarps;
    bool is_v = false;
    int ht = 0;
    int64_t off = -1;
    if (q < n) {
        stage_of(q, nt, is_v, ht);
        off = stage_block_offset(ga, sm, j, nbw, n_union, h0 + ht, lane);
    }
    for (; q < n; q += kProdWarps) {
        const uint32_t it = it0 + q;
        const int s = (int)(it % kNS);
        const uint32_t use = it / kNS;       // this stage is use `use` of slot s
        if (use > 0) {
            wait_published(sm, s, use);      // use - 1 is in the slot (or was)
            wait_or_abort(sm, &sm.empty[s], (use - 1) & 1);
        }
        const unsigned char* base = is_v ? a.kv.v : a.kv.k;
        const int qn = q + kProdWarps;
        bool nv = false;
        int nh = 0;
        if (qn < n)
            stage_of(qn, nt, nv, nh);
        int64_t off_next = -1;
        if (kE4M3) {
            // The stage's raw codes (64 rows x 256 bytes) go by cp.async into
            // the upper half of the slot, linearly (row t at 16 KB + 256 t), all
            // in flight at once.  Chunk idx = lane + 32 i: row idx / 16, codes
            // 16 (idx % 16) .. + 15.
            const uint32_t st = tc::smem_addr(sm.ring[s]);
            const uint32_t raw = st + kStageBytes / 2;
#pragma unroll 8
            for (int i = 0; i < 32; ++i) {
                const int idx = lane + 32 * i, row = idx >> 4;
                const int64_t o = __shfl_sync(0xffffffffu, off, row >> 2);
                const unsigned char* src =
                    base + (o < 0 ? 0 : o + (row & 3) * a.kv.token_b + 16 * (idx & 15));
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(raw + 16 * idx),
                             "l"(src), "r"(o < 0 ? 0 : 16)
                             : "memory");
            }
            cp_async_commit();
            if (qn < n)                          // the next stage's rows, while these copies fly
                off_next = stage_block_offset(ga, sm, j, nbw, n_union, h0 + nh, lane);
            cp_async_wait<0>();
            __syncwarp();
            // codes 128..255 of every row into registers (chunk idx = lane +
            // 32 i: row idx / 8, codes 128 + 16 (idx % 8) .. + 15), so the
            // f16 tiles of dimensions 128..255 may overwrite the raw half
            uint4 hi[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int idx = lane + 32 * i;
                asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                             : "=r"(hi[i].x), "=r"(hi[i].y), "=r"(hi[i].z), "=r"(hi[i].w)
                             : "r"(raw + 256 * (idx >> 3) + 128 + 16 * (idx & 7)));
            }
            // 16 codes (chunk c16 of row `row`) -> two 16-byte f16 chunks of the
            // 128-byte-swizzled K-major tile
            auto put = [&](const uint4& r4, int row, int c16) {
                uint32_t h[8];
                e4m3x4_to_f16x2x2(r4.x, h[0], h[1]);
                e4m3x4_to_f16x2x2(r4.y, h[2], h[3]);
                e4m3x4_to_f16x2x2(r4.z, h[4], h[5]);
                e4m3x4_to_f16x2x2(r4.w, h[6], h[7]);
                const uint32_t rb = st + (c16 >> 2) * kRegionBytes + row * 128;
                const uint32_t x0 = 2 * (c16 & 3);
                asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(rb + ((x0 ^ (row & 7)) << 4)),
                             "r"(h[0]), "r"(h[1]), "r"(h[2]), "r"(h[3]) : "memory");
                asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(rb + (((x0 + 1) ^ (row & 7)) << 4)),
                             "r"(h[4]), "r"(h[5]), "r"(h[6]), "r"(h[7]) : "memory");
            };
            // dimensions 0..127 into the lower half, read from the raw half
#pragma unroll 4
            for (int i = 0; i < 16; ++i) {
                const int idx = lane + 32 * i, row = idx >> 3, c16 = idx & 7;
                uint4 r4;
                asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                             : "=r"(r4.x), "=r"(r4.y), "=r"(r4.z), "=r"(r4.w)
                             : "r"(raw + 256 * row + 16 * c16));
                put(r4, row, c16);
            }
            __syncwarp();                        // every lane is done with the raw half
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int idx = lane + 32 * i;
                put(hi[i], idx >> 3, 8 + (idx & 7));
            }
        } else {
            const uint32_t st = tc::smem_addr(sm.ring[s]) + (lane >> 3) * kRegionBytes;
            const uint32_t x = lane & 7;
#pragma unroll 4
            for (int blk = 0; blk < kStageBlocks; ++blk) {
                const int64_t o = __shfl_sync(0xffffffffu, off, blk);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int row = 4 * blk + u;
                    const uint32_t dst = st + row * 128 + ((x ^ (row & 7)) << 4);
                    const unsigned char* src = base + (o < 0 ? 0 : o + u * a.kv.token_b + 16 * lane);
                    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                                 "r"(o < 0 ? 0 : 16)
                                 : "memory");
                }
            }
            cp_async_commit();
            if (qn < n)                          // the next stage's rows, while these copies fly
                off_next = stage_block_offset(ga, sm, j, nbw, n_union, h0 + nh, lane);
            cp_async_wait<0>();
        }
        tc::fence_async_shared();
        if ((int)it != ga.stall_stage) {     // test hook: a stage left unpublished
            tc::mbar_arrive(is_v ? &sm.full_v[s] : &sm.full_k[ht & 1][s]);
            __syncwarp();
            if (lane == 0)
                *reinterpret_cast<volatile uint32_t*>(&sm.slot_pub[s]) = use + 1;
        }
        off = off_next;
        is_v = nv;
        ht = nh;
    }
    cur.it = it0 + n;
}

// The two MMA issuer threads walk the unit's stages in ring order and each
// acts on its own kind: Q K^T of a stage goes out as soon as its K stage is
// full and its score buffer free (the softmax has read the scores two
// stages back), independently of P V, which waits for the stage's
// probabilities.  Both kinds share the tensor pipe; they touch disjoint TMEM
// columns and shared-memory stages.
__device__ void issue_qk(Smem& sm, Cursor& cur, int nt, int par)
{
    constexpr uint32_t kIdQK = tc::f16_idesc(kM, kStageTokens, false, false);
    const uint32_t tm = sm.tmem_base;
    const uint32_t g0 = cur.g;
    for (int q = 0; q < 2 * nt; ++q, ++cur.it) {
        bool is_v;
        int ht;
        stage_of(q, nt, is_v, ht);
        if (is_v || (ht & 1) != par)
            continue;
        const uint32_t g = g0 + ht, buf = g & 1, s = cur.it % kNS;
        const uint32_t st = tc::smem_addr(sm.ring[s]);
        wait_or_abort(sm, &sm.full_k[par][s], sm.taken[par][s]++ & 1);
        if (g >= 2)                          // P V of stage g - 2 has read P (and so S) there
            wait_or_abort(sm, &sm.p_free[buf], ((g >> 1) - 1) & 1);
        tc::fence_after_sync();
        // descriptors advance by their 16-byte address field: K steps of
        // 16 elements are 32 bytes inside a row, every 4th a new region
        const uint64_t db0 = tc::sw128_desc(st, 16, 1024);
        const uint32_t d = tm + kTmemS + 64 * buf;
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk)
            tc::mma_ts(d, tm + kTmemQ + 8 * kk,
                       db0 + (uint64_t)(((kk >> 2) * kRegionBytes + (kk & 3) * 32) >> 4), kIdQK,
                       kk > 0);
        tc::mma_commit(&sm.empty[s]);
        tc::mma_commit(&sm.s_full[buf]);
    }
    cur.g = g0 + nt;
}

__device__ void issue_pv(Smem& sm, Cursor& cur, int nt)
{
    constexpr uint32_t kIdPV = tc::f16_idesc(kM, kD, false, true);
    const uint32_t tm = sm.tmem_base;
    const uint32_t g0 = cur.g;
    for (int q = 0; q < 2 * nt; ++q, ++cur.it) {
        bool is_v;
        int ht;
        stage_of(q, nt, is_v, ht);
        if (!is_v)
            continue;
        const uint32_t g = g0 + ht, buf = g & 1, s = cur.it % kNS;
        const uint32_t st = tc::smem_addr(sm.ring[s]);
        wait_or_abort(sm, &sm.full_v[s], sm.taken[2][s]++ & 1);
        const uint64_t db0 = tc::sw128_desc(st, kRegionBytes, 1024);
        const uint32_t acc0 = ht > 0;
        // P (128 slots x 64 tokens, f16 pairs) from the first 32 columns of
        // the stage's score buffer; 16 tokens per K step = 8 columns.  The
        // first two K steps go as soon as their half of P is written.
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            wait_or_abort(sm, half ? &sm.p_full[buf] : &sm.p_half[buf], (g >> 1) & 1);
            tc::fence_after_sync();
#pragma unroll
            for (int kk = 2 * half; kk < 2 * half + 2; ++kk)
                tc::mma_ts(tm + kTmemO, tm + kTmemS + 64 * buf + 8 * kk,
                           db0 + (uint64_t)(kk * 128), kIdPV, kk > 0 ? 1u : acc0);
        }
        tc::mma_commit(&sm.empty[s]);
        tc::mma_commit(&sm.p_free[buf]);
    }
    cur.g = g0 + nt;
}

// How many times block b is listed in the selection row (duplicates are a
// caller error that still counts per listing); the own block counts once.
__device__ int listed_count(const int32_t* sel, int n_sel, int r, int b, int own)
{
    if (b == own)
        return 1;
    const int32_t* row = sel + (size_t)r * n_sel;
    int c = 0;
    for (int e = 0; e < n_sel; ++e)
        c += __ldg(row + e) == b;
    return c;
}

// Slow path of a row with duplicated selections: the probabilities of each
// attended block of the stage (first union rank k0) in the slot's P row are
// multiplied by the number of times the row lists the block; returns the
// probability mass this adds to the row's sum.
// Duplicated selections (a caller error) keep their meaning -- a block
// listed c times counts c times: the probabilities of this thread's slot in
// the stage's P (32 TMEM columns of f16 pairs at taddr, just stored) are
// multiplied by their blocks' listing counts; returns the mass added.
// Warp-collective (TMEM loads and stores are): lanes without duplicates
// write their row back unchanged.  (The selection comes by value: no
// address of the kernel's parameters escapes into this out-of-line call.)
__device__ __noinline__ float scale_listed(const int32_t* sel, int n_sel, const Smem& sm,
                                           uint32_t taddr, bool dup, int r, int own, int nbw,
                                           int k0, uint32_t live16)
{
    uint32_t pk[32];
    tc::tmem_wait_st();                        // the stores just issued, before reading them
    tc::tmem_ld32(taddr, pk);
    tc::tmem_wait_ld();
    float added = 0.f;
#pragma unroll
    for (int kb = 0; kb < kStageBlocks; ++kb) {
        if (!dup || !((live16 >> kb) & 1u))
            continue;
        const int cnt = listed_count(sel, n_sel, r, block_of_rank(sm, nbw, k0 + kb), own);
        if (cnt == 1)
            continue;
        for (int e = 0; e < 2; ++e) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&pk[2 * kb + e]));
            const float p0 = f.x * (float)cnt, p1 = f.y * (float)cnt;
            added += (p0 + p1) - (f.x + f.y);
            pk[2 * kb + e] = pack_half2(p0, p1);
        }
    }
    tc::tmem_st32(taddr, pk);
    return added;
}

// Named barriers of the softmax warps (0 is __syncthreads, 1 the mask
// rebuild of all softmax warps).  Per TMEM lane quarter wq: the reference
// handoff from warpgroup A to B (2 + wq) and from B to A (6 + wq), and the
// exchange of the sums at the end of a unit (10 + wq).
__device__ __forceinline__ void named_sync(int id)
{
    asm volatile("bar.sync %0, 64;" ::"r"(id) : "memory");
}

__device__ __forceinline__ void named_arrive(int id)
{
    asm volatile("bar.arrive %0, 64;" ::"r"(id) : "memory");
}

// Softmax warps.  Warpgroup wg = t >> 7 takes the unit's stages i = wg,
// wg + 2, ...; slot = t & 127 (row slot / G, head slot % G) is the thread's
// TMEM lane, and the thread handles all 64 score columns of its stage.  Per
// stage:
//   1. the scores (two 32-column TMEM loads), masked to the blocks the
//      slot's row attends, and their maximum;
//   2. the reference m after the previous stage, from the other group
//      (named barrier); m grows to this stage's maximum only when that
//      exceeds it by more than 2^8 -- O (holding every earlier stage under
//      the old m) is then rescaled in TMEM once P V of the previous stage is
//      done -- and goes on to the other group;
//   3. P = 2^(x - m) as FP16 over the first 32 columns of the score buffer
//      for P V (the first 32 tokens published on their own), and the
//      group's running sum (kept under the reference the group last used
//      and brought to the newer one whenever it changes).
// The scores arrive in units of the kernel's score scale sl2 > 0 (its sign
// was folded into Q), so a masked score of -inf gives P = 0 directly.
// At the end of the unit both groups bring their sums to the final reference,
// add them, and split the output columns (group wg writes 128 wg ... + 127).
__device__ float2 softmax_unit(const GroupArgs& ga, Smem& sm, Cursor& cur, int r0, int Rg,
                               int nt, int h0, int nbw, int cap, int words_per_row, float sl2)
{
    const PrefillArgs& a = ga.a;
    const int t = threadIdx.x, wg = t >> 7, slot = t & (kM - 1), wq = (t >> 5) & 3;
    const int rl = slot / a.G;
    const bool slot_ok = rl < Rg;
    const int own = slot_ok ? sm.row_own[rl] : -1;
    const int rank_own = slot_ok ? sm.row_rank_own[rl] : -1;
    const int tail_n = own >= 0 ? sm.row_p[rl] - 4 * own + 1 : 0;
    const bool dup = own >= 0 && sm.row_dup[rl] != 0;
    const uint32_t tl = sm.tmem_base + ((uint32_t)(32 * wq) << 16);
    const int bar_in = (wg ? 2 : 6) + wq;      // the other group's reference arrives here
    const int bar_out = (wg ? 6 : 2) + wq;     // this group's reference leaves here
    float m_used = -INFINITY, l = 0.f;
    const uint32_t g0 = cur.g;
    int win = 0;                               // mask window of this group's latest stage
    for (int i = wg; i < nt; i += 2) {
        const uint32_t g = g0 + i, buf = g & 1;
        const int wi = i / cap;
        while (win < wi) {                     // both groups rebuild every window once
            ++win;
            build_masks(ga, sm, r0, Rg, h0 + win * cap, cap, words_per_row);
        }
        uint32_t live16 = 0u;                  // blocks of the stage the slot attends
        if (own >= 0) {
            const int li = i - wi * cap;
            live16 = (sm.masks[rl * words_per_row + (li >> 1)] >> ((li & 1) << 4)) & 0xFFFFu;
        }

        wait_or_abort(sm, &sm.s_full[buf], (g >> 1) & 1);
        tc::fence_after_sync();
        uint32_t sv[64];
        tc::tmem_ld32(tl + kTmemS + 64 * buf, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
        tc::tmem_ld32(tl + kTmemS + 64 * buf + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
        tc::tmem_wait_ld();

        float x[64];
#pragma unroll
        for (int kb = 0; kb < kStageBlocks; ++kb) {
            const bool pb = (live16 >> kb) & 1u;
#pragma unroll
            for (int u = 0; u < 4; ++u)
                x[4 * kb + u] = pb ? __uint_as_float(sv[4 * kb + u]) : -INFINITY;
        }
        if (rank_own >= 0 && (rank_own >> 4) == h0 + i) {   // the row's own block: tokens <= p
            const int ko = rank_own & 15;
#pragma unroll
            for (int kb = 0; kb < kStageBlocks; ++kb)
                if (kb == ko) {
#pragma unroll
                    for (int u = 1; u < 4; ++u)
                        if (u >= tail_n)
                            x[4 * kb + u] = -INFINITY;
                }
        }
        float mx[16];
#pragma unroll
        for (int c = 0; c < 16; ++c)
            mx[c] = fmaxf(fmaxf(x[c], x[c + 16]), fmaxf(x[c + 32], x[c + 48]));
#pragma unroll
        for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
            for (int c = 0; c < w; ++c)
                mx[c] = fmaxf(mx[c], mx[c + w]);
        const float mt = mx[0] * sl2;

        // ---- the reference after this stage
        float m_prev = -INFINITY;
        if (i > 0) {
            named_sync(bar_in);
            m_prev = sm.mref[slot];
        }
        const float m_new = mt > m_prev + kRescaleSlack ? mt : m_prev;
        sm.mref[slot] = m_new;
        __threadfence_block();                 // the store is visible before the arrival
        named_arrive(bar_out);
        if (m_new != m_used) {                 // 0 while nothing was attended yet
            l *= ex2(m_used - m_new);
            m_used = m_new;
        }
        // ---- a grown reference: O holds stages < i under m_prev once P V of
        // stage i - 1 is done (P V completes in issue order); scale the
        // lane's O row in place before any of P(g) is published (P V of
        // stage g adds to the scaled O)
        const bool resc = m_new != m_prev && m_prev != -INFINITY;
        if (__any_sync(0xffffffffu, resc)) {
            wait_or_abort(sm, &sm.p_free[(g - 1) & 1], ((g - 1) >> 1) & 1);
            tc::fence_after_sync();
            const float f = resc ? ex2(m_prev - m_new) : 1.f;
#pragma unroll 1
            for (int c = 0; c < kD / 16; ++c) {    // 16 columns a step: the scores stay in registers
                uint32_t o[16];
                const uint32_t col = kTmemO + 16 * c;
                tc::tmem_ld16(tl + col, o);
                tc::tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
                tc::tmem_st16(tl + col, o);
            }
        }
        // ---- P(g) into the first 32 columns of the stage's score buffer (its
        // scores are in registers; Q K^T of stage g waited for P V of stage
        // g - 2, the buffer's previous user): every column unconditionally
        // (masked ones give 0), straight-line so the exponentials overlap.
        // The first 32 tokens are published on their own, so P V starts on
        // them while the rest are computed; a warp with duplicated
        // selections rescales P in place first and publishes both at the end.
        const float m_off = m_new == -INFINITY ? 0.f : -m_new;
        const bool wdup = __any_sync(0xffffffffu, dup);
        float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            uint32_t pk[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const float p0 = ex2(fmaf(x[32 * half + 2 * c], sl2, m_off));
                const float p1 = ex2(fmaf(x[32 * half + 2 * c + 1], sl2, m_off));
                ls[c & 3] += p0 + p1;
                pk[c] = pack_half2(p0, p1);
            }
            tc::tmem_st16(tl + kTmemS + 64 * buf + 16 * half, pk);
            if (half == 0 && !wdup) {
                tc::tmem_wait_st();
                tc::fence_before_sync();
                tc::mbar_arrive(&sm.p_half[buf]);
            }
        }
        l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
        if (wdup)                              // duplicated selections: count per listing
            l += scale_listed(a.sel, a.n_sel, sm, tl + kTmemS + 64 * buf, dup, r0 + rl, own, nbw,
                              kStageBlocks * (h0 + i), live16);

        tc::tmem_wait_st();                    // P and any O rescale stores
        tc::fence_before_sync();
        if (wdup)
            tc::mbar_arrive(&sm.p_half[buf]);
        tc::mbar_arrive(&sm.p_full[buf]);
    }

    // ---- epilogue
    const int last_win = nt > 0 ? (nt - 1) / cap : 0;
    while (win < last_win) {                   // rebuilds the other group still makes
        ++win;
        build_masks(ga, sm, r0, Rg, h0 + win * cap, cap, words_per_row);
    }
    float m_fin = m_used;
    if (nt > 0 && wg != ((nt - 1) & 1)) {      // the other group ran the last stage
        named_sync(bar_in);
        m_fin = sm.mref[slot];
    }
    if (m_fin != m_used)
        l *= ex2(m_used - m_fin);
    sm.xl[wg][slot] = l;
    named_sync(10 + wq);
    const float lt = l + sm.xl[wg ^ 1][slot];
    if (nt > 0) {                              // the last P V is done
        const uint32_t g_last = g0 + nt - 1;
        wait_or_abort(sm, &sm.p_free[g_last & 1], (g_last >> 1) & 1);
        tc::fence_after_sync();
    }
    tc::fence_before_sync();
    cur.g = g0 + nt;
    return make_float2(nt > 0 ? m_fin : -INFINITY, nt > 0 ? lt : 0.f);
}

__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Barrier of every thread of both CTAs of the cluster; the writes before it
// (shared memory of either CTA) are visible after it.
__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The two CTAs of a cluster each ran half of a unit's stages (rank 0 the
// first half) into their own TMEM accumulators, each with its own final
// reference m and sum l per slot.  CTA rank c writes output dimensions
// 128 c .. 128 c + 127; each softmax thread (slot, warpgroup wg) owns 64 of
// them.  Step 1 (between the two cluster barriers): send the partner the
// thread's accumulator over the partner's 64 dimensions, and (wg 0) m and l,
// into the partner's shared memory (the first two ring slots: the ring is
// idle between units).  Step 2: combine the two halves,
//   out = (2^(m_a - M) O_a + 2^(m_b - M) O_b) / (2^(m_a - M) l_a + 2^(m_b - M) l_b)
// (M = max(m_a, m_b); a half with l = 0 adds nothing), and write FP16.
// Exchange buffer (the first two ring slots): the sending warp (warpgroup
// wg, lane quarter wq) and the combining warp of the partner are the same
// (slot, wg) threads, so each warp has an 8 KB block, chunk-major: chunk c
// (16 bytes, c = 0..15) of lane l at 16 (32 c + l).  For one chunk the 32
// lanes write 512 contiguous bytes to the partner and read them back free of
// bank conflicts.
__device__ __forceinline__ uint32_t xchg_offset(int wg, int wq, int lane, int chunk)
{
    return (uint32_t)(8192 * (4 * wg + wq) + 16 * (32 * chunk + lane));
}

__device__ void pair_send(Smem& sm, uint32_t crank, float2 ml)
{
    const int t = threadIdx.x, wg = t >> 7, slot = t & (kM - 1), wq = (t >> 5) & 3;
    const uint32_t tl = sm.tmem_base + ((uint32_t)(32 * wq) << 16);
    const uint32_t peer = crank ^ 1u;
    uint32_t rb;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rb) : "r"(tc::smem_addr(sm.ring[0])), "r"(peer));
    const bool have = ml.y > 0.f;
    uint32_t o[64];                          // all 64 columns in flight at once
    tc::tmem_ld32(tl + kTmemO + 128 * peer + 64 * wg, *reinterpret_cast<uint32_t(*)[32]>(&o[0]));
    tc::tmem_ld32(tl + kTmemO + 128 * peer + 64 * wg + 32,
                  *reinterpret_cast<uint32_t(*)[32]>(&o[32]));
    tc::tmem_wait_ld();
#pragma unroll
    for (int e = 0; e < 16; ++e)
        asm volatile("st.shared::cluster.v4.u32 [%0], {%1,%2,%3,%4};"
                     ::"r"(rb + xchg_offset(wg, wq, t & 31, e)),
                     "r"(have ? o[4 * e] : 0u), "r"(have ? o[4 * e + 1] : 0u),
                     "r"(have ? o[4 * e + 2] : 0u), "r"(have ? o[4 * e + 3] : 0u)
                     : "memory");
    if (wg == 0) {
        uint32_t rm;
        asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rm) : "r"(tc::smem_addr(&sm.xml[slot][0])), "r"(peer));
        asm volatile("st.shared::cluster.v2.f32 [%0], {%1,%2};" ::"r"(rm), "f"(ml.x), "f"(ml.y) : "memory");
    }
}

__device__ void pair_combine(const GroupArgs& ga, Smem& sm, int r0, int Rg, int j, uint32_t crank,
                             float2 ml)
{
    const PrefillArgs& a = ga.a;
    const int t = threadIdx.x, wg = t >> 7, slot = t & (kM - 1), wq = (t >> 5) & 3;
    const int rl = slot / a.G, h = slot - rl * a.G;
    const uint32_t tl = sm.tmem_base + ((uint32_t)(32 * wq) << 16);
    const float m_a = ml.x, l_a = ml.y, m_b = sm.xml[slot][0], l_b = sm.xml[slot][1];
    const float M = fmaxf(m_a, m_b);
    const float w_a = l_a > 0.f ? ex2(m_a - M) : 0.f, w_b = l_b > 0.f ? ex2(m_b - M) : 0.f;
    const float den = w_a * l_a + w_b * l_b;
    const float inv = den > 0.f ? a.v_scale / den : 0.f;     // E4M3: the per-tensor scale of V
    const unsigned char* xb = sm.ring[0];
    uint4* dst = rl < Rg ? reinterpret_cast<uint4*>(a.out + ((size_t)(r0 + rl) * a.Hq +
                                                             (size_t)j * a.G + h) * kD +
                                                    128 * crank + 64 * wg)
                         : nullptr;
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
        uint32_t o[16];
        tc::tmem_ld16(tl + kTmemO + 128 * crank + 64 * wg + 16 * c, o);
        float pb[16];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float4 v = *reinterpret_cast<const float4*>(xb + xchg_offset(wg, wq, t & 31, 4 * c + e));
            pb[4 * e] = v.x;
            pb[4 * e + 1] = v.y;
            pb[4 * e + 2] = v.z;
            pb[4 * e + 3] = v.w;
        }
        tc::tmem_wait_ld();
        if (dst != nullptr) {
            uint32_t hv[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                float v[2];
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const float oa = l_a > 0.f ? __uint_as_float(o[2 * e + k]) * w_a : 0.f;
                    const float ob = l_b > 0.f ? pb[2 * e + k] * w_b : 0.f;
                    v[k] = (oa + ob) * inv;
                }
                hv[e] = pack_half2(v[0], v[1]);
            }
            dst[2 * c] = make_uint4(hv[0], hv[1], hv[2], hv[3]);
            dst[2 * c + 1] = make_uint4(hv[4], hv[5], hv[6], hv[7]);
        }
    }
}

template <bool kE4M3>
__global__ void __launch_bounds__(kThreads, 1) sparse_prefill_grouped_kernel(const GroupArgs ga)
{
    extern __shared__ unsigned char smem_raw[];
    Smem& sm = *reinterpret_cast<Smem*>(
        smem_raw + ((1024u - (tc::smem_addr(smem_raw) & 1023u)) & 1023u));
    const PrefillArgs& a = ga.a;
    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < kNS; ++s) {
            tc::mbar_init(&sm.full_k[0][s], 32);
            tc::mbar_init(&sm.full_k[1][s], 32);
            tc::mbar_init(&sm.full_v[s], 32);
            tc::mbar_init(&sm.empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(&sm.s_full[b], 1);
            tc::mbar_init(&sm.p_half[b], kGroupThreads);   // and writes P(g)
            tc::mbar_init(&sm.p_full[b], kGroupThreads);
            tc::mbar_init(&sm.p_free[b], 1);
        }
        tc::mbar_init(&sm.done, 3);                         // all three MMA issuers commit
        for (int s = 0; s < kNS; ++s) {
            sm.taken[0][s] = sm.taken[1][s] = sm.taken[2][s] = 0u;
            sm.slot_pub[s] = 0u;
        }
        sm.abort = 0;
        sm.spin_limit = ga.spin_limit > 0 ? ga.spin_limit : tc::kSpinLimit;
        tc::mbar_init_fence();
    }
    if (w == kMmaWarp)
        tc::tmem_alloc(&sm.tmem_base, kTmemCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();

    Cursor cur;
    // Clusters of two CTAs: both take the same unit, rank 0 the first half of
    // its half-tiles, rank 1 the rest; units go to the clusters in snake order.
    const uint32_t crank = cluster_ctarank();
    const int C = gridDim.x / 2, ci = (int)blockIdx.x / 2;
    for (int wave = 0; wave * C < ga.n_units; ++wave) {
        const int u = wave * C + ((wave & 1) ? C - 1 - ci : ci);
        if (u >= ga.n_units)
            continue;                            // both CTAs of the cluster alike
        const int gi = u / a.Hkv, j = u - gi * a.Hkv;
        const int r0 = gi * ga.Rg, Rg = min(ga.Rg, a.R - r0);
        const int words_per_row = kMaskWords / Rg, cap = 2 * words_per_row;
        unit_setup(ga, sm, r0, Rg, j, ga.nbw, words_per_row, cap, crank);
        const int nt_all = (sm.n_union + kStageBlocks - 1) / kStageBlocks;
        const int h0 = crank ? nt_all / 2 : 0;
        const int nt = crank ? nt_all - nt_all / 2 : nt_all / 2;
        float2 ml = make_float2(-INFINITY, 0.f);
        if (w >= kProdWarp0 && w < kProdWarp0 + kProdWarps)
            produce<kE4M3>(ga, sm, cur, j, ga.nbw, nt, h0, sm.n_union);
        else if (w == kMmaWarp && lane == 0)
            issue_qk(sm, cur, nt, 0);
        else if (w == kQkWarp1 && lane == 0)
            issue_qk(sm, cur, nt, 1);
        else if (w == kPvWarp && lane == 0)
            issue_pv(sm, cur, nt);
        else if (w < kSoftWarps)
            ml = softmax_unit(ga, sm, cur, r0, Rg, nt, h0, ga.nbw, cap, words_per_row,
                              a.scale_log2 == 0.f ? 1.f : fabsf(a.scale_log2));
        if (tid == 0 && sm.flags)
            raise_flag(a.err, sm.flags);
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
        // ---- the two halves: exchange across the cluster, combine, write
        cluster_sync_all();                      // both rings idle, both accumulators final
        if (w < kSoftWarps)
            pair_send(sm, crank, ml);
        cluster_sync_all();
        if (w < kSoftWarps)
            pair_combine(ga, sm, r0, Rg, j, crank, ml);
        tc::fence_before_sync();
        __syncthreads();                         // the exchange buffer and TMEM read
        tc::fence_after_sync();
    }
    if ((w == kMmaWarp || w == kPvWarp || w == kQkWarp1) && lane == 0)
        tc::mma_commit(&sm.done);            // arrives once this issuer's MMAs are done
    if (w == kMmaWarp && lane == 0) {        // every MMA done before TMEM is released
        // (waited for even after a time-out: the MMAs issued complete on
        // their own, and TMEM must not be freed under them)
        if (!tc::mbar_wait(&sm.done, 0, sm.spin_limit))
            sm.abort = 1;
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (tid == 0 && sm.abort)
        raise_flag(a.err, PAGED_GQA_FLAG_TIMEOUT);
    if (w == kMmaWarp)
        tc::tmem_dealloc(sm.tmem_base, kTmemCols);
}

}  // namespace grp

bool grouped_prefill_supported(const PrefillArgs& a)
{
    return a.G >= 1 && a.G <= grp::kM &&
           (int64_t)a.kv_len <= (int64_t)4 * 32 * kGroupMaxWords;
}

int grouped_prefill_rows(const PrefillArgs& a, int clusters, int rows_per_group)
{
    const int rg_max = grp::kM / a.G;
    if (rows_per_group > 0)
        return min(rows_per_group, rg_max);
    // Fill whole waves of co-resident CTA pairs with units as large as that
    // allows.
    const int64_t units_min = (int64_t)((a.R + rg_max - 1) / rg_max) * a.Hkv;
    const int64_t waves = (units_min + clusters - 1) / clusters;
    const int64_t groups = std::max<int64_t>(1, waves * clusters / a.Hkv);
    return (int)std::min<int64_t>(rg_max, (a.R + groups - 1) / groups);
}

namespace {

// The kernel's launch shape: clusters of two CTAs, one CTA per SM.
cudaLaunchConfig_t grouped_config(int clusters, cudaStream_t s, cudaLaunchAttribute* attr)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * clusters));
    cfg.blockDim = dim3(grp::kThreads);
    cfg.dynamicSmemBytes = grp::kSmemBytes;
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

}  // namespace

// CTA pairs of the grouped kernel that the current device holds at once
// (cached per device; the kernels' shared-memory attribute is set here).
cudaError_t grouped_prefill_clusters(int& clusters)
{
    static std::atomic<int> cached[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    clusters = cached[dev].load(std::memory_order_acquire);
    if (clusters > 0)
        return cudaSuccess;
    for (int k = 0; k < 2; ++k) {
        e = k ? cudaFuncSetAttribute(grp::sparse_prefill_grouped_kernel<true>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)grp::kSmemBytes)
              : cudaFuncSetAttribute(grp::sparse_prefill_grouped_kernel<false>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)grp::kSmemBytes);
        if (e != cudaSuccess)
            return e;
    }
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess)
        return e;
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = grouped_config(sms / 2, nullptr, attr);
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, grp::sparse_prefill_grouped_kernel<false>, &cfg);
    if (e != cudaSuccess)
        return e;
    clusters = std::max(1, std::min(n, sms / 2));
    cached[dev].store(clusters, std::memory_order_release);
    return cudaSuccess;
}

cudaError_t launch_prefill_grouped(const PrefillArgs& a, bool e4m3, int rows_per_group,
                                   cudaStream_t s, long spin_limit, int stall_stage)
{
    int clusters = 0;
    cudaError_t e = grouped_prefill_clusters(clusters);
    if (e != cudaSuccess)
        return e;
    GroupArgs ga{};
    ga.a = a;
    ga.Rg = grouped_prefill_rows(a, clusters, rows_per_group);
    const int64_t groups = (a.R + ga.Rg - 1) / ga.Rg;
    ga.n_units = (int)(groups * a.Hkv);
    const int64_t blocks = a.kv_len > 0 ? ((int64_t)a.kv_len + 3) / 4 : 1;
    ga.nbw = (int)std::max<int64_t>(1, (blocks + 31) / 32);
    ga.spin_limit = spin_limit;
    ga.stall_stage = stall_stage;
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = grouped_config(std::min(ga.n_units, clusters), s, attr);
    return e4m3 ? cudaLaunchKernelEx(&cfg, grp::sparse_prefill_grouped_kernel<true>, ga)
                : cudaLaunchKernelEx(&cfg, grp::sparse_prefill_grouped_kernel<false>, ga);
}

}  // namespace pgqa
