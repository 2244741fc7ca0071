// select.cu -- QSA block selection: per query row, the top-k four-token blocks
// by score.
//
// Operation: "[Kernel][SM70] Accelerate exact Qwen3.8 decode" (1Cat-vLLM
// #415), Implementation: QSA's selection finds the pivot score with four
// radix passes over the scores and then compacts the pivot's ties by
// increasing block index.  The result is the sorted selected-block list the
// sparse prefill of "[Kernel][SM70] Accelerate Qwen3.8 QSA paged prefill"
// (#378), Changes, consumes: for a row at position p, the min(k, n) best of
// its n = floor(p / 4) causal blocks (equal scores: lower index first), in
// increasing index order, padded with -1.
//
// Design (ours): one CTA of 256 threads per row.  The row's scores become
// 32-bit keys whose unsigned order is IEEE totalOrder (flip the sign bit of
// non-negative values, all bits of negative ones).  The pivot key -- the k-th
// largest -- is fixed digit by digit, 11 + 11 + 10 bits, each digit chosen
// from a histogram of the keys that still match the digits above it; a digit
// whose keys are all to be taken ends the search early.  Only the first
// histogram runs over the whole row, fused with staging the keys in shared
// memory (rows longer than the stage read them from global memory); the keys
// of the chosen first digit are then gathered into a short index list, and
// the later digits are histogrammed over that list.  (Rows whose first-digit
// bucket overflows the list, e.g. constant rows, histogram the whole row
// again, filtered by the digits found so far.)  The output is written by one
// pass in index order: each warp owns a contiguous segment, ballots rank the
// lanes inside the warp, and per-warp counts of keys above the pivot and
// equal to it give each warp its share of the pivot's ties (the lowest
// indices) and its first output position, so the selected indices come out
// ascending without a sort.
#include <atomic>

#include "pgqa_internal.h"

namespace pgqa {

namespace {

constexpr int kSelThreads = 256;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kStageMax = 16384;     // keys staged in shared memory, at most (64 KB)
constexpr int kBins = 2048;          // histogram bins (11-bit digits)
constexpr int kListCap = 2048;       // gathered first-digit bucket, at most
constexpr int kMapWords = kStageMax / 32;   // bitmaps of the fast path

// The scores are read as 32-bit patterns (never as float values, so no
// floating-point handling of NaNs or signed zeros can touch them) and mapped
// to keys whose unsigned order is IEEE totalOrder.
__device__ __forceinline__ uint32_t order_key(uint32_t u)
{
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct SelectShared {
    uint32_t hist[kBins];
    uint32_t above_map[kMapWords];   // fast path: bit i = key i is taken
    uint32_t bucket_map[kMapWords];  // fast path: bit i = key i is in the first-digit bucket
    int32_t list[kListCap];
    int32_t list_n;
    int32_t warp_tot[kSelWarps];
    int32_t warp_gt[kSelWarps];
    int32_t warp_eq[kSelWarps];
    int32_t pick_digit, pick_above, pick_count;
};

// Keys of a row: staged in shared memory or read from global memory.
struct StagedKeys {
    const uint32_t* k;
    __device__ uint32_t operator()(int i) const { return k[i]; }
};
struct GlobalKeys {
    const uint32_t* row;
    __device__ uint32_t operator()(int i) const { return order_key(__ldg(row + i)); }
};

// From the histogram of nbins bins (digit value = bin), the digit d holding
// the need-th largest counted key: above(d) < need <= above(d) + hist[d],
// above(d) = the count of larger digits.  Writes pick_* and returns after a
// CTA barrier.  Thread t owns bins [t * per, (t + 1) * per).
__device__ __forceinline__ void pick_digit(SelectShared& sh, int nbins, int need)
{
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int per = nbins / kSelThreads;
    uint32_t s = 0;
    for (int e = 0; e < per; ++e)
        s += sh.hist[tid * per + e];
    uint32_t incl = s;                                  // this and higher lanes of the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_down_sync(0xffffffffu, incl, o);
        if (lane + o < 32)
            incl += t;
    }
    if (lane == 0)
        sh.warp_tot[w] = (int32_t)incl;
    __syncthreads();
    uint32_t above = incl - s;
    for (int v = w + 1; v < kSelWarps; ++v)
        above += (uint32_t)sh.warp_tot[v];
    if (above < (uint32_t)need && (uint32_t)need <= above + s) {
        uint32_t a = above;
        for (int e = per - 1; e >= 0; --e) {
            const uint32_t c = sh.hist[tid * per + e];
            if ((uint32_t)need <= a + c) {
                sh.pick_digit = tid * per + e;
                sh.pick_above = (int32_t)a;
                sh.pick_count = (int32_t)c;
                break;
            }
            a += c;
        }
    }
    __syncthreads();
}

// Exclusive prefix sum over the CTA's threads (in thread order) of v; also
// returns the total.  Two CTA barriers.
__device__ __forceinline__ int block_exclusive_scan(SelectShared& sh, int v, int& total)
{
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += t;
    }
    __syncthreads();                                      // warp_tot free
    if (lane == 31)
        sh.warp_tot[w] = incl;
    __syncthreads();
    int base = 0;
    total = 0;
    for (int v2 = 0; v2 < kSelWarps; ++v2) {
        base += v2 < w ? sh.warp_tot[v2] : 0;
        total += sh.warp_tot[v2];
    }
    return base + incl - v;
}

// Fast path of radix_select for rows of n <= 32 kMapWords keys whose
// first-digit bucket fits the list: bitmaps instead of ordered sweeps.
//   above_map  keys whose first digit is above the pivot's (all taken);
//   bucket_map keys in the pivot's first-digit bucket.
// The bucket is listed in index order from its bitmap, its later digits fix
// the pivot, its taken keys (above the pivot, or at it among the first
// `need` by index) join above_map, and the output is the set bits of
// above_map in index order.
template <class Keys>
__device__ void select_by_bitmaps(const Keys& key, int n, int32_t* out, SelectShared& sh,
                                  uint32_t d1, int need, int count1)
{
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int nw = (n + 31) >> 5;
    // ---- one sweep: ballots of 32 consecutive keys are the bitmap words
    for (int wd = w; wd < nw; wd += kSelWarps) {
        const int i = 32 * wd + lane;
        const uint32_t b = i < n ? key(i) >> 21 : 0u;
        const unsigned g = __ballot_sync(0xffffffffu, i < n && b > d1);
        const unsigned e = __ballot_sync(0xffffffffu, i < n && b == d1);
        if (lane == 0) {
            sh.above_map[wd] = g;
            sh.bucket_map[wd] = e;
        }
    }
    __syncthreads();
    const int per = (nw + kSelThreads - 1) / kSelThreads;   // words per thread (<= 2)
    const int w0 = min(nw, tid * per), w1 = min(nw, w0 + per);
    int total;
    if (need == count1) {
        // the whole bucket is taken
        for (int wd = w0; wd < w1; ++wd)
            sh.above_map[wd] |= sh.bucket_map[wd];
    } else {
        // ---- the bucket in index order
        int c = 0;
        for (int wd = w0; wd < w1; ++wd)
            c += __popc(sh.bucket_map[wd]);
        int pos = block_exclusive_scan(sh, c, total);
        for (int wd = w0; wd < w1; ++wd) {
            uint32_t bits = sh.bucket_map[wd];
            while (bits) {
                sh.list[pos++] = 32 * wd + __ffs(bits) - 1;
                bits &= bits - 1u;
            }
        }
        // ---- later digits over the bucket
        uint32_t prefix = d1 << 21, mask = 0xFFE00000u;
#pragma unroll 1
        for (int pass = 0; pass < 2; ++pass) {
            const int shift = pass == 0 ? 10 : 0;
            const uint32_t dmask = pass == 0 ? 2047u : 1023u;
            __syncthreads();                              // list complete / picks read
            for (int i = tid; i < kBins; i += kSelThreads)
                sh.hist[i] = 0;
            __syncthreads();
            for (int j = tid; j < count1; j += kSelThreads) {
                const uint32_t kv = key(sh.list[j]);
                if ((kv & mask) == prefix)
                    atomicAdd(&sh.hist[(kv >> shift) & dmask], 1u);
            }
            __syncthreads();
            pick_digit(sh, pass == 0 ? kBins : 1024, need);
            need -= sh.pick_above;
            prefix |= (uint32_t)sh.pick_digit << shift;
            mask |= dmask << shift;
            if (sh.pick_count == need)
                break;                                    // CTA-uniform
        }
        // ---- taken bucket keys: contiguous list ranges per thread, ties by index
        const int lper = (count1 + kSelThreads - 1) / kSelThreads;
        const int j0 = min(count1, tid * lper), j1 = min(count1, j0 + lper);
        int eq = 0;
        for (int j = j0; j < j1; ++j)
            eq += (key(sh.list[j]) & mask) == prefix;
        int rank = block_exclusive_scan(sh, eq, total);
        for (int j = j0; j < j1; ++j) {
            const int i = sh.list[j];
            const uint32_t kv = key(i) & mask;
            bool take = kv > prefix;
            if (kv == prefix)
                take = rank++ < need;
            if (take)
                atomicOr(&sh.above_map[i >> 5], 1u << (i & 31));
        }
    }
    __syncthreads();
    // ---- output: set bits of above_map in index order
    int c = 0;
    for (int wd = w0; wd < w1; ++wd)
        c += __popc(sh.above_map[wd]);
    int pos = block_exclusive_scan(sh, c, total);
    for (int wd = w0; wd < w1; ++wd) {
        uint32_t bits = sh.above_map[wd];
        while (bits) {
            out[pos++] = 32 * wd + __ffs(bits) - 1;
            bits &= bits - 1u;
        }
    }
}

// Writes the k outputs of row `out` for the selection of the n keys of
// `key` (n > k >= 1).  When kStage, the first sweep also stores the keys of
// `row` into stage (which `key` reads).
template <bool kStage, class Keys>
__device__ void radix_select(const uint32_t* row, uint32_t* stage, const Keys& key, int n, int k,
                             int32_t* out, SelectShared& sh)
{
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const unsigned lt = (1u << lane) - 1u;
    const int seg = ((n + kSelWarps - 1) / kSelWarps + 31) & ~31;   // warp w: [w seg, (w+1) seg)
    const int lo = min(n, w * seg), hi = min(n, lo + seg);

    // ---- digit 1 (key bits 31..21) over the whole row, fused with staging
    for (int i = tid; i < kBins; i += kSelThreads)
        sh.hist[i] = 0;
    if (tid == 0)
        sh.list_n = 0;
    __syncthreads();
    if (kStage && (reinterpret_cast<uintptr_t>(row) & 15u) == 0) {
        // 16-byte loads, kUnroll of them in flight per thread before any is used
        constexpr int kUnroll = 8;
        const int n4 = n >> 2;
        const uint4* row4 = reinterpret_cast<const uint4*>(row);
        uint4* stage4 = reinterpret_cast<uint4*>(stage);
        for (int j0 = tid; j0 < n4; j0 += kSelThreads * kUnroll) {
            uint4 v[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int j = j0 + u * kSelThreads;
                v[u] = j < n4 ? __ldg(row4 + j) : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int j = j0 + u * kSelThreads;
                if (j < n4) {
                    const uint4 kv = make_uint4(order_key(v[u].x), order_key(v[u].y),
                                                order_key(v[u].z), order_key(v[u].w));
                    stage4[j] = kv;
                    atomicAdd(&sh.hist[kv.x >> 21], 1u);
                    atomicAdd(&sh.hist[kv.y >> 21], 1u);
                    atomicAdd(&sh.hist[kv.z >> 21], 1u);
                    atomicAdd(&sh.hist[kv.w >> 21], 1u);
                }
            }
        }
        for (int i = 4 * n4 + tid; i < n; i += kSelThreads) {
            const uint32_t kv = order_key(__ldg(row + i));
            stage[i] = kv;
            atomicAdd(&sh.hist[kv >> 21], 1u);
        }
    } else {
        constexpr int kUnroll = 8;
        for (int i0 = tid; i0 < n; i0 += kSelThreads * kUnroll) {
            uint32_t v[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int i = i0 + u * kSelThreads;
                v[u] = i < n ? (kStage ? order_key(__ldg(row + i)) : key(i)) : 0u;
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int i = i0 + u * kSelThreads;
                if (i < n) {
                    if (kStage)
                        stage[i] = v[u];
                    atomicAdd(&sh.hist[v[u] >> 21], 1u);
                }
            }
        }
    }
    __syncthreads();
    pick_digit(sh, kBins, k);
    const uint32_t d1 = (uint32_t)sh.pick_digit;
    int need = k - sh.pick_above;
    const int count1 = sh.pick_count;
    uint32_t prefix = d1 << 21, mask = 0xFFE00000u;
    const bool done1 = count1 == need;                   // the whole bucket is taken
    const bool use_list = !done1 && count1 <= kListCap;
    if (n <= 32 * kMapWords && (done1 || use_list)) {
        select_by_bitmaps(key, n, out, sh, d1, need, count1);
        return;
    }

    // ---- per-warp counts above / in the bucket; gather the bucket
    int gt_w = 0, eq_w = 0;
    for (int i0 = lo; i0 < hi; i0 += 32) {
        const int i = i0 + lane;
        const uint32_t b = i < hi ? key(i) >> 21 : 0u;
        const unsigned g = __ballot_sync(0xffffffffu, i < hi && b > d1);
        const unsigned e = __ballot_sync(0xffffffffu, i < hi && b == d1);
        gt_w += __popc(g);
        eq_w += __popc(e);
        if (use_list && e != 0u) {
            int base = 0;
            if (lane == 0)
                base = atomicAdd(&sh.list_n, __popc(e));
            base = __shfl_sync(0xffffffffu, base, 0);
            if ((e >> lane) & 1u)
                sh.list[base + __popc(e & lt)] = i;
        }
    }
    if (lane == 0) {
        sh.warp_gt[w] = gt_w;
        sh.warp_eq[w] = done1 ? eq_w : 0;
    }

    if (!done1) {
        // ---- digits 2 (bits 20..10) and 3 (bits 9..0) over the bucket
#pragma unroll 1
        for (int pass = 0; pass < 2; ++pass) {
            const int shift = pass == 0 ? 10 : 0;
            const uint32_t dmask = pass == 0 ? 2047u : 1023u;
            __syncthreads();                              // list and previous picks complete
            for (int i = tid; i < kBins; i += kSelThreads)
                sh.hist[i] = 0;
            __syncthreads();
            if (use_list) {
                for (int j = tid; j < count1; j += kSelThreads) {
                    const uint32_t kv = key(sh.list[j]);
                    if ((kv & mask) == prefix)
                        atomicAdd(&sh.hist[(kv >> shift) & dmask], 1u);
                }
            } else {
                for (int i = tid; i < n; i += kSelThreads) {
                    const uint32_t kv = key(i);
                    if ((kv & mask) == prefix)
                        atomicAdd(&sh.hist[(kv >> shift) & dmask], 1u);
                }
            }
            __syncthreads();
            pick_digit(sh, pass == 0 ? kBins : 1024, need);
            need -= sh.pick_above;
            prefix |= (uint32_t)sh.pick_digit << shift;
            mask |= dmask << shift;
            if (sh.pick_count == need)
                break;                                    // CTA-uniform
        }
        // ---- per-warp counts of the bucket's keys above / at the pivot
        if (use_list) {
            for (int j = tid; j < count1; j += kSelThreads) {
                const int i = sh.list[j];
                const uint32_t kv = key(i) & mask;
                if (kv > prefix)
                    atomicAdd(&sh.warp_gt[i / seg], 1);
                else if (kv == prefix)
                    atomicAdd(&sh.warp_eq[i / seg], 1);
            }
        } else {
            int g2 = 0, e2 = 0;
            for (int i0 = lo; i0 < hi; i0 += 32) {
                const int i = i0 + lane;
                const uint32_t kv = i < hi ? key(i) & mask : 0u;
                g2 += __popc(__ballot_sync(0xffffffffu, i < hi && kv > prefix));
                e2 += __popc(__ballot_sync(0xffffffffu, i < hi && kv == prefix));
            }
            __syncthreads();                              // warp_gt from the bucket sweep read
            if (lane == 0) {
                sh.warp_gt[w] = g2;
                sh.warp_eq[w] = e2;
            }
        }
    }
    __syncthreads();

    // ---- ordered write: above the pivot, or at it among the first `need`
    int eq_base = 0, sel_base = 0;
    for (int v = 0; v < w; ++v) {
        sel_base += sh.warp_gt[v] + max(0, min(need - eq_base, sh.warp_eq[v]));
        eq_base += sh.warp_eq[v];
    }
    for (int i0 = lo; i0 < hi; i0 += 32) {
        const int i = i0 + lane;
        const uint32_t kv = i < hi ? key(i) & mask : 0u;
        const bool gt = i < hi && kv > prefix;
        const bool eq = i < hi && kv == prefix;
        const unsigned e = __ballot_sync(0xffffffffu, eq);
        const bool take = gt || (eq && eq_base + __popc(e & lt) < need);
        const unsigned s = __ballot_sync(0xffffffffu, take);
        if (take)
            out[sel_base + __popc(s & lt)] = i;
        eq_base += __popc(e);
        sel_base += __popc(s);
    }
}

}  // namespace

__global__ void __launch_bounds__(kSelThreads, 4) qsa_select_kernel(SelectArgs a)
{
    extern __shared__ __align__(16) unsigned char sel_smem[];
    __shared__ SelectShared sh;
    const int r = blockIdx.x, tid = threadIdx.x;
    int32_t* out = a.out + (int64_t)r * a.k;
    int flags = 0;
    int64_t p = __ldg(a.q_pos + r);
    int n = 0;
    if (p < 0 || a.kv_len <= 0) {
        flags |= PAGED_GQA_FLAG_EMPTY_ROW;
    } else {
        if (p >= a.kv_len) {
            flags |= PAGED_GQA_FLAG_QPOS_CLAMPED;
            p = a.kv_len - 1;
        }
        int64_t nc = p / 4;                               // blocks before the row's own
        if (nc > a.n_blocks) {
            flags |= PAGED_GQA_FLAG_SCORES_SHORT;
            nc = a.n_blocks;
        }
        n = (int)nc;
    }
    if (tid == 0)
        raise_flag(a.err, flags);
    if (n <= a.k) {
        // every candidate is taken: 0 .. n-1, then padding
        for (int i = tid; i < a.k; i += kSelThreads)
            out[i] = i < n ? i : -1;
        return;
    }
    const uint32_t* row = reinterpret_cast<const uint32_t*>(a.scores) + (int64_t)r * a.stride;
    if (n <= a.stage_keys) {
        uint32_t* stage = reinterpret_cast<uint32_t*>(sel_smem);
        radix_select<true>(row, stage, StagedKeys{stage}, n, a.k, out, sh);
    } else {
        radix_select<false>(row, nullptr, GlobalKeys{row}, n, a.k, out, sh);
    }
}

// Keys staged per CTA for a call whose rows have at most n_blocks candidates.
int select_stage_keys(int n_blocks)
{
    return n_blocks < kStageMax ? n_blocks : kStageMax;
}

cudaError_t launch_select(const SelectArgs& a, cudaStream_t s)
{
    static std::atomic<int> done[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev >= kMaxDevices || !done[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(qsa_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)(kStageMax * sizeof(uint32_t)));
        if (e != cudaSuccess)
            return e;
        if (dev < kMaxDevices)
            done[dev].store(1, std::memory_order_release);
    }
    const size_t smem = (size_t)a.stage_keys * sizeof(uint32_t);
    qsa_select_kernel<<<a.R, kSelThreads, smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace pgqa
