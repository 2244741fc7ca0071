// sample_mask.cu -- combined top-k/top-p masking of the decode step's logits.
//
// Operation: "[Kernel][SM70] Scale NVFP4 E4M3 decode batches" (1Cat-vLLM
// #282), Purpose: the decode step's second operator masks B8/B16 rows of
// 248,320 logits with top-k and top-p together (run at top-k 20, top-p 0.95 in
// its Performance contract).  Per row: top-k keeps the min(k, V) largest
// logits (equal logits: the lower index first); top-p keeps, of those in that
// order, the shortest leading run whose softmax mass (over the top-k logits)
// reaches p; every other logit becomes -infinity.  The top-p mass is computed
// in FP64: e_j = exp(x_j - x_0), suffix sums S_j = e_j + S_{j+1} of the list
// (formed by a shuffle scan here), logit j kept iff S_j > (1 - p) S_0.
//
// Design (ours): one thread-block cluster of kMaskCtas CTAs per row, so a
// handful of rows still spreads over the GPU.  Each CTA sweeps its slice of
// the row once from HBM (keys: unsigned order = numeric order of the
// logits).  A bound that at least k keys reach needs no CTA-wide sort: each
// warp sorts its lanes' maxima with shuffles, and the smallest over the warps
// of their ceil(k / 16)-th largest is reached by at least 16 ceil(k / 16) >= k
// maxima.  The sweep's first batch (8 16-byte loads per thread) stays in
// registers until such a bound over it is known; the keys reaching it are
// collected from the registers, the later batches are collected as they
// stream, and the same bound over the whole slice's maxima then filters the
// list (a few times k keys).  Ranking the survivors -- every thread counts,
// for one (key, 32-key chunk) pair, the chunk's larger keys -- gives the
// slice's exact top-k; a tie-saturated slice, where too many keys reach the
// bound, uses the radix selection of select_core.cuh over global memory.
// When out is not the input, -infinity goes into out during the sweep.  Each
// CTA stores its top-k into the shared memory of every CTA of the cluster
// (st.shared::cluster) -- masking in place, it writes -infinity over the
// rest of its slice while the barrier completes -- and then every CTA ranks
// the union (larger key first, equal keys by index) the same way and runs the
// FP64 top-p (for k <= 32 in one warp's registers: exp per lane, suffix sums
// by a shuffle scan), and settles its own top-k: kept logits carry their
// original bits (read again from the input, which nothing has overwritten
// there), the others -infinity.  A logit outside its slice's top-k cannot be
// kept.  A split barrier at the start makes sure every CTA of the cluster
// runs before the first remote store; nothing touches another CTA's shared
// memory after the second barrier.  HBM traffic: the row read once, written
// once.
#include <atomic>

#include "select_core.cuh"

namespace pgqa {

namespace {

constexpr int kMaskThreads = 512;
constexpr int kMaskWarps = kMaskThreads / 32;
constexpr int kMaskCtas = 8;            // CTAs per row: one cluster
constexpr int kMaskSliceMax = 40960;    // columns per CTA, at most
constexpr int kMaskKMax = 128;          // largest k served
constexpr int kFilterCap = 1024;        // keys the first bound may let through
constexpr int kBatch = 8;               // 16-byte loads per thread in flight
constexpr int kFillBytes = 8192;        // -inf source of the bulk fill
constexpr size_t kFillOffset = (sizeof(selcore::SelectShared<kMaskThreads, kMaskSliceMax / 32>) + 127) & ~size_t(127);
constexpr size_t kMaskDynSmem = kFillOffset + kFillBytes;
static_assert(kMaskKMax <= 8 * kMaskWarps, "the bound takes at most the 8th largest of a warp");
using MaskShared = selcore::SelectShared<kMaskThreads, kMaskSliceMax / 32>;

// Written by every CTA of the cluster into every CTA's copy.
struct MaskCluster {
    int32_t cnt[kMaskCtas];                        // top-k size of each CTA's slice
    uint32_t key[kMaskCtas * kMaskKMax];           //   ... its keys (slot r * kMaskKMax + i)
    int32_t idx[kMaskCtas * kMaskKMax];            //   ... their row columns
};

// Per-CTA scratch of the slice's top-k.
struct MaskLocal {
    uint32_t wbound[kMaskWarps];                   // each warp's bound candidate
    int32_t n, n2;                                 // keys collected at or above the bound / kept
    uint64_t comp[kFilterCap];                     //   ... as composites (value keys)
    int32_t rank[kFilterCap];                      //   ... their rank in the slice
    uint32_t cand_key[kMaskKMax];                  // the slice's top-k (radix fallback)
    int32_t cand_idx[kMaskKMax];                   // slice columns of the top-k, by rank
};

// Every CTA's scratch for ranking the cluster's candidates.
struct MaskMerge {
    int32_t grank[kMaskCtas * kMaskKMax];          // rank in the row of candidate slot r kMaskKMax + i
    int32_t order[kMaskKMax];                      // slot at each rank
    double e[kMaskKMax];                           // e_j (k > 32)
};

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Split cluster barrier: arrive (release or relaxed), later wait (acquire).
// Every thread of every CTA of the cluster takes part.
__device__ __forceinline__ void cluster_arrive_relaxed()
{
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive()
{
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait()
{
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t dsmem(const void* p, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}

__device__ __forceinline__ void st_dsmem(uint32_t addr, uint32_t v)
{
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// Bulk copy (the copy engine, no per-thread stores) of `bytes` (a multiple of
// 16; both addresses 16-byte aligned) from shared to global memory.
__device__ __forceinline__ void bulk_store(void* gdst, const void* ssrc, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                 ::"l"(gdst), "r"(smem_u32(ssrc)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bulk_commit()
{
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Waits until this thread's committed bulk copies have completed and orders
// their writes before the thread's later generic-proxy accesses.
__device__ __forceinline__ void bulk_wait_all()
{
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// A candidate as one 64-bit value whose unsigned order is the selection
// order: the key above, the bitwise complement of the column below (a larger
// key, or an equal key at a lower column, is larger).
__device__ __forceinline__ uint64_t composite(uint32_t key, int col)
{
    return ((uint64_t)key << 32) | (uint32_t)~(uint32_t)col;
}
__device__ __forceinline__ uint32_t comp_key(uint64_t c) { return (uint32_t)(c >> 32); }
__device__ __forceinline__ int comp_col(uint64_t c) { return (int)~(uint32_t)c; }

// IEEE totalOrder key of a float's bits (two instructions).  0xFFFFFFFF, the
// padding of loads past the slice, has key 0, the smallest.  It orders the
// values as their value keys do except -0 < +0; a bound b in this order is
// widened to take -0 along with +0 (value_bound).
__device__ __forceinline__ uint32_t tkey(uint32_t u)
{
    return u ^ ((uint32_t)((int32_t)u >> 31) | 0x80000000u);
}
// The totalOrder threshold that keeps every value >= the value of bound b.
__device__ __forceinline__ uint32_t total_bound(uint32_t b)
{
    return b == 0x80000000u ? 0x7FFFFFFFu : b;
}
// The value-key threshold that keeps every value >= the value of bound b.
__device__ __forceinline__ uint32_t value_bound(uint32_t b)
{
    return b == 0x7FFFFFFFu ? 0x80000000u : b;
}

// Descending sort of one value per lane across the warp (bitonic, shuffles
// only): lane i ends with the i-th largest.
__device__ __forceinline__ uint32_t warp_sort_descending(uint32_t v)
{
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const uint32_t o = __shfl_xor_sync(0xffffffffu, v, stride);
            const bool desc = (lane & size) == 0 || size == 32, low = (lane & stride) == 0;
            v = (desc == low) ? max(v, o) : min(v, o);
        }
    }
    return v;
}

// rank[q] += how many of comp[0 .. n) are larger than comp[q], for every
// q < n, by all threads of the CTA: each takes (key q, 32-key chunk g) pairs,
// consecutive threads consecutive keys of one chunk (the chunk's reads are
// broadcasts).  rank must be zero on entry; the caller synchronises after.
__device__ __forceinline__ void rank_all(const uint64_t* comp, int n, int32_t* rank)
{
    const int items = n * ((n + 31) >> 5);
    for (int it = threadIdx.x; it < items; it += kMaskThreads) {
        const int g = it / n, q = it - g * n;
        const uint64_t c = comp[q];
        const int u0 = 32 * g, u1 = min(n, u0 + 32);
        int cnt = 0;
#pragma unroll 8
        for (int u = u0; u < u1; ++u)
            cnt += comp[u] > c;
        if (cnt != 0)
            atomicAdd(&rank[q], cnt);
    }
}

// grank[r kMaskKMax + i] = the rank in the row of candidate i of CTA r (how
// many of the cluster's T candidates are larger), for i < cnt[r]: each CTA's list is in descending order, so every thread takes
// (candidate, list) pairs and binary-searches the list (the candidate's own
// list contributes its index).  grank must be zero on entry; the caller
// synchronises after.
__device__ __forceinline__ void rank_cluster(const MaskCluster& mc, int T, int32_t* grank)
{
    for (int it = threadIdx.x; it < T * kMaskCtas; it += kMaskThreads) {
        const int r = it / T;
        int ro = 0, io = it - r * T;              // candidate q = it - r T as (list, index)
        while (io >= mc.cnt[ro])
            io -= mc.cnt[ro++];
        int lo = io;
        if (r != ro) {
            const uint64_t c = composite(mc.key[ro * kMaskKMax + io], mc.idx[ro * kMaskKMax + io]);
            lo = 0;
            int hi = mc.cnt[r];
            while (lo < hi) {                         // first entry of list r not above c
                const int mid = (lo + hi) >> 1;
                if (composite(mc.key[r * kMaskKMax + mid], mc.idx[r * kMaskKMax + mid]) > c)
                    lo = mid + 1;
                else
                    hi = mid;
            }
        }
        if (lo > 0)
            atomicAdd(&grank[ro * kMaskKMax + io], lo);
    }
}

// A key that at least k of the CTA's keys reach, from the threads' largest
// keys (lane_max; threads 0 .. active - 1 hold at least one key): over the
// wf = active / 32 warps whose lanes all hold keys, the smallest of each
// warp's c-th largest lane maximum, c = ceil(k / wf) -- reached by the
// maxima of wf c >= k threads; 0 (every key) when c would exceed 32.  Every
// thread calls it, once per kernel; it synchronises the CTA once.
__device__ __forceinline__ uint32_t cta_bound(uint32_t lane_max, int k, int active,
                                              uint32_t* wbound)
{
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int wf = min(active, kMaskThreads) >> 5;
    const int c = wf > 0 ? (k + wf - 1) / wf : 33;
    const uint32_t srt = warp_sort_descending(lane_max);
    const uint32_t wb = __shfl_sync(0xffffffffu, srt, min(c, 32) - 1);
    if (lane == 0)
        wbound[w] = wb;
    __syncthreads();
    if (c > 32)
        return 0u;
    uint32_t b = 0xffffffffu;
    for (int v = 0; v < wf; ++v)
        b = min(b, wbound[v]);
    return b;
}

// The logit value of a key (ValueOrderKey maps -0 to +0; the value is the
// same number).
__device__ __forceinline__ float key_value(uint32_t k)
{
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// The slice's top-k (k < n) by the radix selection of select_core.cuh over
// global memory: columns (in index order) into cand_idx, their value keys
// into cand_key.  Out of line: only tie-saturated slices take it.
__device__ __noinline__ void slice_radix_top_k(const uint32_t* row, int n, int k,
                                               int32_t* cand_idx, uint32_t* cand_key,
                                               MaskShared& sh)
{
    const selcore::ValueOrderKey key_of{};
    using Keys = selcore::GlobalKeys<selcore::ValueOrderKey>;
    selcore::radix_select<false>(row, nullptr, Keys{row, key_of}, key_of, n, k, cand_idx, sh);
    __syncthreads();
    for (int i = threadIdx.x; i < k; i += kMaskThreads)
        cand_key[i] = key_of(__ldg(row + cand_idx[i]));
}

}  // namespace

__global__ void __launch_bounds__(kMaskThreads, 2) topk_topp_kernel(MaskArgs a)
{
    extern __shared__ __align__(16) unsigned char mask_smem[];
    MaskShared& sh = *reinterpret_cast<MaskShared*>(mask_smem);   // radix state, candidate map
    __shared__ MaskCluster mc;
    __shared__ MaskLocal loc;
    __shared__ MaskMerge mm;
    cluster_arrive_relaxed();                     // paired with the wait before the first remote store
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const uint32_t rank = cluster_rank();
    const int b = blockIdx.x / kMaskCtas;
    const int lo = min(a.V, (int)rank * a.slice), hi = min(a.V, lo + a.slice), n = hi - lo;
    const float* xrow = a.x + (int64_t)b * a.x_stride;
    const float* xs = xrow + lo;
    const uint32_t* row = reinterpret_cast<const uint32_t*>(xs);
    float* orow = a.out + (int64_t)b * a.out_stride + lo;
    const int K = min(a.k, a.V);
    const selcore::ValueOrderKey key_of{};
    const float ninf = -INFINITY;
    const bool early = orow != xs;                // out is not the input: -inf while sweeping
    const bool vec = (reinterpret_cast<uintptr_t>(row) & 15u) == 0;
    const bool ovec = (reinterpret_cast<uintptr_t>(orow) & 15u) == 0;
    // Thread tid's columns: with 16-byte loads, batch t register 4u + c holds
    // column 4 (tid + (t kBatch + u) kMaskThreads) + c (below 4 n4), then the
    // columns 4 n4 + tid + i kMaskThreads; otherwise tid + i kMaskThreads.
    const int n4 = vec ? n >> 2 : 0;
    if (tid == 0) {
        loc.n = 0;
        loc.n2 = 0;
    }
    for (int i = tid; i < kFilterCap; i += kMaskThreads)
        loc.rank[i] = 0;
    for (int i = tid; i < kMaskCtas * kMaskKMax; i += kMaskThreads)
        mm.grank[i] = 0;
    // out is not the input and 16-byte aligned: the copy engine writes -inf
    // over the slice's whole vectors from a shared buffer while the threads
    // sweep (the rest: plain stores during the sweep)
    const bool bulk = early && ovec && n >= 4;
    const bool vec1 = vec && n4 > 0;              // 16-byte loads: the slice has a whole vector
    float* fill_src = reinterpret_cast<float*>(mask_smem + kFillOffset);
    if (bulk) {
        for (int i = tid; i < kFillBytes / 4; i += kMaskThreads)
            fill_src[i] = ninf;
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        if (tid < (n & 3))
            orow[4 * (n >> 2) + tid] = ninf;
    }
    __syncthreads();                              // loc, the fill source
    if (bulk && tid == 0) {
        const uint32_t bytes = (uint32_t)(n >> 2) * 16u;
        for (uint32_t off = 0; off < bytes; off += kFillBytes)
            bulk_store(reinterpret_cast<char*>(orow) + off, fill_src,
                       min((uint32_t)kFillBytes, bytes - off));
        bulk_commit();
    }

    // ---- sweep.  Keys here are totalOrder keys; mx is the thread's largest
    // (0: none).  16-byte loads: batch bb covers vectors j = tid + (bb kBatch
    // + u) kMaskThreads < n4, padded with key 0 past n4; the first batch stays
    // in registers until a bound over it is known, and every batch's keys at
    // or above the bound are collected as composites of value keys.
    uint32_t mx = 0u, bound = 0u, beff = 0u;
    auto push = [&](uint32_t u, int col) {
        const int pos = atomicAdd(&loc.n, 1);
        if (pos < kFilterCap)
            loc.comp[pos] = composite(key_of(u), col);
    };
    if (vec1) {
        const int nb = (n4 + kBatch * kMaskThreads - 1) / (kBatch * kMaskThreads);
        const uint4* row4 = reinterpret_cast<const uint4*>(row);
#pragma unroll 1
        for (int bb = 0; bb < nb; ++bb) {
            const int j0 = tid + bb * kBatch * kMaskThreads;
            uint32_t r[4 * kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int j = j0 + u * kMaskThreads;
                const uint4 t = j < n4 ? __ldg(row4 + j) : make_uint4(~0u, ~0u, ~0u, ~0u);
                r[4 * u] = t.x;
                r[4 * u + 1] = t.y;
                r[4 * u + 2] = t.z;
                r[4 * u + 3] = t.w;
            }
            if (early && !bulk) {
#pragma unroll
                for (int u = 0; u < kBatch; ++u) {
                    const int j = j0 + u * kMaskThreads;
                    if (j < n4) {
#pragma unroll
                        for (int c = 0; c < 4; ++c)
                            orow[4 * j + c] = ninf;
                    }
                }
            }
#pragma unroll
            for (int e = 0; e < 4 * kBatch; ++e)
                mx = max(mx, tkey(r[e]));
            if (bb == 0) {
                bound = n > a.k ? cta_bound(mx, a.k, n4, loc.wbound) : 0u;
                beff = total_bound(bound);
            }
            uint32_t hm = 0u;
#pragma unroll
            for (int e = 0; e < 4 * kBatch; ++e)
                hm |= (uint32_t)(tkey(r[e]) >= beff) << e;
            if (hm != 0u) {
#pragma unroll
                for (int u = 0; u < kBatch; ++u)
                    if (j0 + u * kMaskThreads >= n4)
                        hm &= ~(15u << (4 * u));      // padding
#pragma unroll
                for (int e = 0; e < 4 * kBatch; ++e)
                    if ((hm >> e) & 1u)
                        push(r[e], 4 * (j0 + (e >> 2) * kMaskThreads) + (e & 3));
            }
        }
        // the last n - 4 n4 (< 4) columns
        const int i = 4 * n4 + tid;
        if (i < n) {
            const uint32_t u = __ldg(row + i);
            mx = max(mx, tkey(u));
            if (early && !bulk)
                orow[i] = ninf;
            if (tkey(u) >= beff)
                push(u, i);
        }
    } else {
        // unaligned rows or slices of fewer than 4 columns: one sweep for the
        // bound, a second (from L2) to collect
#pragma unroll 4
        for (int i = tid; i < n; i += kMaskThreads) {
            mx = max(mx, tkey(__ldg(row + i)));
            if (early && !bulk)
                orow[i] = ninf;
        }
        bound = n > a.k ? cta_bound(mx, a.k, n, loc.wbound) : 0u;
        beff = total_bound(bound);
#pragma unroll 4
        for (int i = tid; i < n; i += kMaskThreads) {
            const uint32_t u = __ldg(row + i);
            if (tkey(u) >= beff)
                push(u, i);
        }
    }

    __syncthreads();                              // the list is complete
    int C = loc.n;
    if (C <= kFilterCap) {
        // ---- the same bound over the whole slice's maxima thins the list
        const uint32_t v2 =
            value_bound(n > a.k ? cta_bound(mx, a.k, vec1 ? n4 : n, loc.wbound) : 0u);
        uint64_t keep[(kFilterCap + kMaskThreads - 1) / kMaskThreads];
        int nk = 0;
#pragma unroll
        for (int t = 0; t < (kFilterCap + kMaskThreads - 1) / kMaskThreads; ++t) {
            const int c = tid + t * kMaskThreads;
            keep[t] = c < C ? loc.comp[c] : 0u;
            nk += c < C && comp_key(keep[t]) >= v2;
        }
        __syncthreads();                          // every entry read
        if (nk != 0) {
            int pos = atomicAdd(&loc.n2, nk);
#pragma unroll
            for (int t = 0; t < (kFilterCap + kMaskThreads - 1) / kMaskThreads; ++t)
                if (tid + t * kMaskThreads < C && comp_key(keep[t]) >= v2)
                    loc.comp[pos++] = keep[t];
        }
        __syncthreads();
        C = loc.n2;
    } else {
        // ---- a tie-saturated slice: radix selection over global memory
        slice_radix_top_k(row, n, a.k, loc.cand_idx, loc.cand_key, sh);
        for (int i = tid; i < a.k; i += kMaskThreads)
            loc.comp[i] = composite(loc.cand_key[i], loc.cand_idx[i]);
        __syncthreads();
        C = a.k;
    }
    const int cn = min(C, a.k);

    // ---- the slice's top-k, in rank order, into every CTA of the cluster
    rank_all(loc.comp, C, loc.rank);
    __syncthreads();
    cluster_wait();                               // every CTA of the cluster runs
    for (int c = tid; c < C; c += kMaskThreads) {
        const int better = loc.rank[c];
        if (better < a.k) {
            const uint64_t cc = loc.comp[c];
            loc.cand_idx[better] = comp_col(cc);
            const int slot = (int)rank * kMaskKMax + better;
#pragma unroll 1
            for (int r = 0; r < kMaskCtas; ++r) {
                st_dsmem(dsmem(&mc.key[slot], r), comp_key(cc));
                st_dsmem(dsmem(&mc.idx[slot], r), (uint32_t)(lo + comp_col(cc)));
            }
        }
    }
    if (tid < kMaskCtas)
        st_dsmem(dsmem(&mc.cnt[rank], tid), (uint32_t)cn);
    cluster_arrive();

    // ---- in place, meanwhile: -inf over the slice except its top-k
    if (!early) {
        uint32_t* cand_map = sh.above_map;        // bit i: slice column i is a candidate
        const int nw = (n + 31) >> 5;
        for (int v = tid; v < nw; v += kMaskThreads)
            cand_map[v] = 0u;
        __syncthreads();
        for (int i = tid; i < cn; i += kMaskThreads)
            atomicOr(&cand_map[loc.cand_idx[i] >> 5], 1u << (loc.cand_idx[i] & 31));
        __syncthreads();
        if (ovec) {
            const int m4 = n >> 2;
            for (int i4 = tid; i4 < m4; i4 += kMaskThreads) {
                const uint32_t bits = (cand_map[i4 >> 3] >> ((i4 & 7) * 4)) & 15u;
                if (bits == 0u) {
                    reinterpret_cast<float4*>(orow)[i4] = make_float4(ninf, ninf, ninf, ninf);
                } else {
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        if (!((bits >> u) & 1u))
                            orow[4 * i4 + u] = ninf;
                }
            }
            for (int i = 4 * m4 + tid; i < n; i += kMaskThreads)
                if (!((cand_map[i >> 5] >> (i & 31)) & 1u))
                    orow[i] = ninf;
        } else {
            for (int i = tid; i < n; i += kMaskThreads)
                if (!((cand_map[i >> 5] >> (i & 31)) & 1u))
                    orow[i] = ninf;
        }
    }
    cluster_wait();

    // ---- the row's top-K and top-p, in every CTA
    int T = 0;
#pragma unroll
    for (int r = 0; r < kMaskCtas; ++r)
        T += mc.cnt[r];
    rank_cluster(mc, T, mm.grank);
    __syncthreads();
    for (int q = tid; q < T; q += kMaskThreads) {
        int r = 0, i = q;
        while (i >= mc.cnt[r])
            i -= mc.cnt[r++];
        const int slot = r * kMaskKMax + i;
        if (mm.grank[slot] < K)
            mm.order[mm.grank[slot]] = slot;
    }
    __syncthreads();
    // FP64 masses of the top-K logits (their values are their keys mapped back)
    auto value_at = [&](int j) { return key_value(mc.key[mm.order[j]]); };
    const float x0f = value_at(0);
    const bool usable = !(isnan(x0f) || isinf(x0f));   // -inf, +inf or NaN at the top
    const double x0 = (double)x0f;
    if (usable && K > 32) {
        for (int j = tid; j < K; j += kMaskThreads)
            mm.e[j] = exp((double)value_at(j) - x0);
        __syncthreads();
    }
    if (w != 0)
        return;
    // one warp from here: S_j = e_j + S_{j+1}, lane l holding j = l per ..
    // l per + per - 1: a suffix within the lane, then a shuffle scan over the
    // lanes above
    int m = K;
    if (usable) {
        const int per = (K + 31) >> 5;                    // 1 .. 4
        double s[4];
        double acc = 0.0;
        if (per == 1) {
            if (lane < K)
                acc = exp((double)value_at(lane) - x0);
            s[0] = acc;
        } else {
#pragma unroll
            for (int i = 3; i >= 0; --i) {
                const int j = lane * per + i;
                if (i < per && j < K)
                    acc = mm.e[j] + acc;
                s[i] = acc;
            }
        }
        double incl = acc;                                // lanes lane .. 31
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const double u = __shfl_down_sync(0xffffffffu, incl, o);
            if (lane + o < 32)
                incl = u + incl;
        }
        double above = __shfl_down_sync(0xffffffffu, incl, 1);   // lanes lane+1 .. 31
        if (lane == 31)
            above = 0.0;
        const double sum0 = __shfl_sync(0xffffffffu, s[0] + above, 0);
        const double cut = (1.0 - (double)a.p) * sum0;
        int cnt = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int j = lane * per + i;
            if (i < per && j < K && s[i] + above > cut)
                ++cnt;
        }
        m = __reduce_add_sync(0xffffffffu, cnt);          // S is non-increasing in j
    } else if (lane == 0 && !(x0f == -INFINITY) && rank == 0) {
        raise_flag(a.err, PAGED_GQA_FLAG_BAD_LOGIT);
    }

    // ---- this slice's top-k: kept logits carry their bits, the others -inf
    // (already there unless masking in place); the bulk fill lands first
    if (bulk && lane == 0)
        bulk_wait_all();
    __syncwarp();
    for (int i = lane; i < cn; i += 32) {
        const int col = loc.cand_idx[i];
        if (mm.grank[(int)rank * kMaskKMax + i] >= m) {
            if (!early)
                orow[col] = ninf;
        } else if (early) {
            orow[col] = xs[col];
        }
    }
}

int mask_slice(int V)
{
    const int s = (V + kMaskCtas - 1) / kMaskCtas;
    return (s + 3) & ~3;
}

bool mask_supported(int V, int k)
{
    return k >= 1 && k <= kMaskKMax && V >= 1 && mask_slice(V) <= kMaskSliceMax;
}

cudaError_t launch_topk_topp(const MaskArgs& a, cudaStream_t s)
{
    static std::atomic<int> done[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev >= kMaxDevices || !done[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(topk_topp_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kMaskDynSmem);
        if (e != cudaSuccess)
            return e;
        if (dev < kMaxDevices)
            done[dev].store(1, std::memory_order_release);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.B * kMaskCtas);
    cfg.blockDim = dim3(kMaskThreads);
    cfg.dynamicSmemBytes = kMaskDynSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kMaskCtas;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, topk_topp_kernel, a);
}

}  // namespace pgqa
