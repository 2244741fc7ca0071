// select_core.cuh -- radix top-k selection of one row of 32-bit keys by one
// CTA, shared by the QSA block selection (select.cu) and the top-k/top-p
// masking (sample_mask.cu).
//
// The k largest of n keys (equal keys: the lower index first) are found by
// fixing the pivot key digit by digit, 11 + 11 + 10 bits, each digit chosen
// from a histogram of the keys that still match the digits above it; a digit
// whose keys are all to be taken ends the search early.  The first histogram
// runs over the whole row, fused with staging the keys in shared memory
// (rows longer than the stage read them from global memory).  For rows of at
// most 32 kMapWords keys whose first-digit bucket fits the list, one ballot
// sweep writes bitmaps of the keys above the pivot's first digit and in its
// bucket; the bucket, listed in index order from its bitmap, fixes the later
// digits; the output is the final bitmap's set bits in index order.  Other
// rows (long ones, or constant ones whose bucket overflows the list) take a
// general path: filtered histograms over the whole row and an ordered write
// in which each warp owns a contiguous segment, ballots rank the lanes, and
// per-warp counts above and at the pivot give each warp its share of the
// pivot's ties and its first output position.  Either way the selected
// indices come out ascending without a sort.
#pragma once

#include "pgqa_internal.h"

namespace pgqa {
namespace selcore {

constexpr int kBins = 2048;          // histogram bins (11-bit digits)
constexpr int kListCap = 2048;       // gathered first-digit bucket, at most

// The scores are read as 32-bit patterns (never as float values, so no
// floating-point handling of NaNs or signed zeros can touch them) and mapped
// to keys whose unsigned order is IEEE totalOrder.
__device__ __forceinline__ uint32_t order_key(uint32_t u)
{
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Key maps handed to radix_select for staging: totalOrder (every bit pattern
// ordered) or numeric order of values (-0 and +0 equal; NaN excluded by the
// caller's contract).
struct TotalOrderKey {
    __device__ uint32_t operator()(uint32_t u) const { return order_key(u); }
};
struct ValueOrderKey {
    __device__ uint32_t operator()(uint32_t u) const { return order_key(u == 0x80000000u ? 0u : u); }
};

template <int kThreads_, int kMapWords_>
struct SelectShared {
    static constexpr int kThreads = kThreads_;
    static constexpr int kMapWords = kMapWords_;
    static constexpr int kWarps = kThreads / 32;
    uint32_t hist[kBins];
    uint32_t above_map[kMapWords];   // fast path: bit i = key i is taken
    uint32_t bucket_map[kMapWords];  // fast path: bit i = key i is in the first-digit bucket
    int32_t list[kListCap];
    int32_t list_n;
    int32_t warp_tot[kWarps];
    int32_t warp_gt[kWarps];
    int32_t warp_eq[kWarps];
    int32_t pick_digit, pick_above, pick_count;
    uint32_t low_and, low_or;        // AND / OR of bits 9..0 over the first digit's bucket
};

// Keys of a row: staged in shared memory or read from global memory.
struct StagedKeys {
    const uint32_t* k;
    __device__ uint32_t operator()(int i) const { return k[i]; }
};
template <class KeyFn>
struct GlobalKeys {
    const uint32_t* row;
    KeyFn kf;
    __device__ uint32_t operator()(int i) const { return kf(__ldg(row + i)); }
};

// From the histogram of nbins bins (digit value = bin), the digit d holding
// the need-th largest counted key: above(d) < need <= above(d) + hist[d],
// above(d) = the count of larger digits.  Writes pick_* and returns after a
// CTA barrier.  Thread t owns bins [t * per, (t + 1) * per).
template <class Sh>
__device__ __forceinline__ void pick_digit(Sh& sh, int nbins, int need)
{
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int per = nbins / Sh::kThreads;
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
    for (int v = w + 1; v < Sh::kWarps; ++v)
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
template <class Sh>
__device__ __forceinline__ int block_exclusive_scan(Sh& sh, int v, int& total)
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
    for (int v2 = 0; v2 < Sh::kWarps; ++v2) {
        base += v2 < w ? sh.warp_tot[v2] : 0;
        total += sh.warp_tot[v2];
    }
    return base + incl - v;
}

// Digits 2 (bits 20..10) and 3 (bits 9..0) of the pivot, from the keys
// key_at(0 .. m) that match prefix/mask (the first digit): need is the rank
// of the pivot among them on entry and among its equals on return; prefix and
// mask then cover every fixed bit.  When the keys matching the first digit
// all share bits 9..0 (known from an AND and an OR taken in the second pass),
// so do those matching the first two, and the third pass is skipped: those
// bits are the pivot's.  Starts with a CTA barrier; every thread leaves after
// the same last one.
template <class Sh, class KeyAt>
__device__ __forceinline__ void later_digits(Sh& sh, const KeyAt& key_at, int m, int& need,
                                             uint32_t& prefix, uint32_t& mask)
{
    const int tid = threadIdx.x, lane = tid & 31;
#pragma unroll 1
    for (int pass = 0; pass < 2; ++pass) {
        const int shift = pass == 0 ? 10 : 0;
        const uint32_t dmask = pass == 0 ? 2047u : 1023u;
        __syncthreads();                              // list and previous picks complete
        for (int i = tid; i < kBins; i += Sh::kThreads)
            sh.hist[i] = 0;
        if (tid == 0) {
            sh.low_and = 0xFFFFFFFFu;
            sh.low_or = 0u;
        }
        __syncthreads();
        uint32_t land = 0xFFFFFFFFu, lor = 0u;
        for (int j = tid; j < m; j += Sh::kThreads) {
            const uint32_t kv = key_at(j);
            if ((kv & mask) == prefix) {
                atomicAdd(&sh.hist[(kv >> shift) & dmask], 1u);
                land &= kv;
                lor |= kv;
            }
        }
        if (pass == 0) {
            land = __reduce_and_sync(0xffffffffu, land & 1023u);
            lor = __reduce_or_sync(0xffffffffu, lor & 1023u);
            if (lane == 0) {
                atomicAnd(&sh.low_and, land);
                atomicOr(&sh.low_or, lor);
            }
        }
        __syncthreads();
        pick_digit(sh, pass == 0 ? kBins : 1024, need);
        need -= sh.pick_above;
        prefix |= (uint32_t)sh.pick_digit << shift;
        mask |= dmask << shift;
        if (sh.pick_count == need)
            break;                                    // CTA-uniform
        if (pass == 0 && sh.low_and == sh.low_or) {   // CTA-uniform: bits 9..0 are shared
            prefix |= sh.low_and;
            mask |= 1023u;
            break;
        }
    }
}

// Fast path of radix_select for rows of n <= 32 kMapWords keys whose
// first-digit bucket fits the list: bitmaps instead of ordered sweeps.
//   above_map  keys whose first digit is above the pivot's (all taken);
//   bucket_map keys in the pivot's first-digit bucket.
// The bucket is listed in index order from its bitmap, its later digits fix
// the pivot, its taken keys (above the pivot, or at it among the first
// `need` by index) join above_map, and the output is the set bits of
// above_map in index order.
template <class Sh, class Keys>
__device__ void select_by_bitmaps(const Keys& key, int n, int32_t* out, Sh& sh,
                                  uint32_t d1, int need, int count1)
{
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int nw = (n + 31) >> 5;
    // ---- one sweep: ballots of 32 consecutive keys are the bitmap words
#pragma unroll 4
    for (int wd = w; wd < nw; wd += Sh::kWarps) {
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
    const int per = (nw + Sh::kThreads - 1) / Sh::kThreads;   // words per thread (<= 2)
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
        later_digits(sh, [&](int j) { return key(sh.list[j]); }, count1, need, prefix, mask);
        // ---- taken bucket keys: contiguous list ranges per thread, ties by index
        const int lper = (count1 + Sh::kThreads - 1) / Sh::kThreads;
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
template <bool kStage, class Sh, class KeyFn, class Keys>
__device__ void radix_select(const uint32_t* row, uint32_t* stage, const Keys& key, KeyFn kf,
                             int n, int k, int32_t* out, Sh& sh)
{
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const unsigned lt = (1u << lane) - 1u;
    const int seg = ((n + Sh::kWarps - 1) / Sh::kWarps + 31) & ~31;   // warp w: [w seg, (w+1) seg)
    const int lo = min(n, w * seg), hi = min(n, lo + seg);

    // ---- digit 1 (key bits 31..21) over the whole row, fused with staging
    for (int i = tid; i < kBins; i += Sh::kThreads)
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
        for (int j0 = tid; j0 < n4; j0 += Sh::kThreads * kUnroll) {
            uint4 v[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int j = j0 + u * Sh::kThreads;
                v[u] = j < n4 ? __ldg(row4 + j) : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int j = j0 + u * Sh::kThreads;
                if (j < n4) {
                    const uint4 kv = make_uint4(kf(v[u].x), kf(v[u].y), kf(v[u].z), kf(v[u].w));
                    stage4[j] = kv;
                    atomicAdd(&sh.hist[kv.x >> 21], 1u);
                    atomicAdd(&sh.hist[kv.y >> 21], 1u);
                    atomicAdd(&sh.hist[kv.z >> 21], 1u);
                    atomicAdd(&sh.hist[kv.w >> 21], 1u);
                }
            }
        }
        for (int i = 4 * n4 + tid; i < n; i += Sh::kThreads) {
            const uint32_t kv = kf(__ldg(row + i));
            stage[i] = kv;
            atomicAdd(&sh.hist[kv >> 21], 1u);
        }
    } else {
        constexpr int kUnroll = 8;
        for (int i0 = tid; i0 < n; i0 += Sh::kThreads * kUnroll) {
            uint32_t v[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int i = i0 + u * Sh::kThreads;
                v[u] = i < n ? (kStage ? kf(__ldg(row + i)) : key(i)) : 0u;
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int i = i0 + u * Sh::kThreads;
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
    if (n <= 32 * Sh::kMapWords && (done1 || use_list)) {
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
        if (use_list)
            later_digits(sh, [&](int j) { return key(sh.list[j]); }, count1, need, prefix, mask);
        else
            later_digits(sh, key, n, need, prefix, mask);
        // ---- per-warp counts of the bucket's keys above / at the pivot
        if (use_list) {
            for (int j = tid; j < count1; j += Sh::kThreads) {
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

}  // namespace selcore
}  // namespace pgqa
