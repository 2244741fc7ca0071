// sample_mask.cu -- combined top-k/top-p masking of the decode step's logits.
//
// Operation: "[Kernel][SM70] Scale NVFP4 E4M3 decode batches" (1Cat-vLLM
// #282), Purpose: the decode step's second operator masks B8/B16 rows of
// 248,320 logits with top-k and top-p together (run at top-k 20, top-p 0.95 in
// its Performance contract).  Per row: top-k keeps the min(k, V) largest
// logits (equal logits: the lower index first); top-p keeps, of those in that
// order, the shortest leading run whose softmax mass (over the top-k logits)
// reaches p; every other logit becomes -infinity.  The top-p mass is computed
// in FP64: e_j = exp(x_j - x_0), suffix sums S_j = e_j + S_{j+1} from the end
// of the list, logit j kept iff S_j > (1 - p) S_0.
//
// Design (ours): one thread-block cluster of kMaskCtas CTAs per row, so a
// handful of rows still spreads over the GPU.  Each CTA finds the top-k of
// its slice of the row (keys whose unsigned order is the numeric order of the
// logits); the row's top-k is among the union of those lists.  The CTA
// bitonic-sorts its threads' maxima, and their k-th largest -- a key that at
// least k keys reach -- bounds the slice's k-th largest key from below; one
// more sweep collects the keys at or above it (typically a few more than k)
// and ranking them gives the exact top-k (a tie-saturated slice, where too
// many keys reach the bound, uses the radix selection of select_core.cuh).  Each CTA then stores its candidates
// straight into rank 0's shared memory (st.shared::cluster) and, while rank 0
// ranks the union (larger key first, equal keys by index), runs the FP64
// top-p and stores the kept columns back into every CTA's shared memory,
// writes -infinity over the rest of its slice: a logit outside its slice's
// top-k cannot be kept.  After the second cluster barrier each CTA settles
// its own candidates.  A split barrier at the start makes sure every CTA of
// the cluster runs before the first remote store; nothing touches another
// CTA's shared memory after the second barrier.  HBM traffic: the row read
// once (its second sweep hits L2), written once.
#include <atomic>

#include "select_core.cuh"

namespace pgqa {

namespace {

constexpr int kMaskThreads = 512;
constexpr int kMaskWarps = kMaskThreads / 32;
constexpr int kMaskCtas = 8;            // CTAs per row: one cluster
constexpr int kMaskSliceMax = 40960;    // columns per CTA, at most
constexpr int kMaskKMax = 128;          // largest k served
constexpr int kBoundK = kMaskThreads;   // k up to which the threads' maxima give the bound
constexpr int kFilterCap = 1024;        // keys the bound may let through
using MaskShared = selcore::SelectShared<kMaskThreads, kMaskSliceMax / 32>;

// Shared state written across the cluster.
struct MaskCluster {
    int32_t cnt[kMaskCtas];                        // rank 0's copy: candidates of each CTA
    uint32_t key[kMaskCtas * kMaskKMax];           //   ... their keys (slot r * kMaskKMax + i)
    int32_t idx[kMaskCtas * kMaskKMax];            //   ... their columns
    int32_t kept_n;                                // every copy: logits the row keeps
    int32_t kept_idx[kMaskKMax];                   //   ... their columns
};

// Per-CTA scratch of the slice's top-k.
struct MaskLocal {
    uint32_t sortbuf[kMaskThreads];                // the lanes' maxima while they are sorted
    uint32_t bound;
    uint64_t comp[kFilterCap];                     // keys at or above the bound, as composites
    int32_t n;
    int32_t cand_n;
    uint32_t cand_key[kMaskKMax];                  // the slice's top-k
    int32_t cand_idx[kMaskKMax];                   // (slice-relative columns)
};

// Rank 0's scratch for ranking the cluster's candidates.
struct MaskMerge {
    int32_t base[kMaskCtas + 1];
    uint64_t comp[kMaskCtas * kMaskKMax];          // the cluster's candidates, as composites
    int32_t order[kMaskKMax];                      // candidate at each rank
    double s[kMaskKMax];                           // e_j, then the suffix sums S_j
    int32_t m;
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

// A candidate as one 64-bit value whose unsigned order is the selection
// order: the key above, the bitwise complement of the column below (a larger
// key, or an equal key at a lower column, is larger).
__device__ __forceinline__ uint64_t composite(uint32_t key, int col)
{
    return ((uint64_t)key << 32) | (uint32_t)~(uint32_t)col;
}
__device__ __forceinline__ uint32_t comp_key(uint64_t c) { return (uint32_t)(c >> 32); }
__device__ __forceinline__ int comp_col(uint64_t c) { return (int)~(uint32_t)c; }

// Rank of c among comp[0 .. n): how many are larger.
__device__ __forceinline__ int rank_in(const uint64_t* comp, int n, uint64_t c)
{
    int better = 0;
#pragma unroll 8
    for (int u = 0; u < n; ++u)
        better += comp[u] > c;
    return better;
}

// The logit value of a key (ValueOrderKey maps -0 to +0; the value is the
// same number).
__device__ __forceinline__ float key_value(uint32_t k)
{
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Ascending bitonic sort of one value per thread across the CTA: partners
// closer than a warp trade through shuffles, the others through buf (one
// slot per thread).  Thread t ends with the t-th smallest value.
__device__ __forceinline__ uint32_t block_sort_ascending(uint32_t v, uint32_t* buf)
{
    const int tid = threadIdx.x;
#pragma unroll
    for (int size = 2; size <= kMaskThreads; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            uint32_t o;
            if (stride >= 32) {
                buf[tid] = v;
                __syncthreads();
                o = buf[tid ^ stride];
                __syncthreads();
            } else {
                o = __shfl_xor_sync(0xffffffffu, v, stride);
            }
            const bool asc = (tid & size) == 0, low = (tid & stride) == 0;
            v = (asc == low) ? min(v, o) : max(v, o);
        }
    }
    return v;
}

// The top-k (k < n) of the slice's n keys, read from global memory, into
// loc.cand_key / loc.cand_idx (any order; ties to the lower column).
template <class Sh>
__device__ void slice_top_k(const uint32_t* row, int n, int k, MaskLocal& loc, Sh& sh)
{
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const selcore::ValueOrderKey key_of{};
    if (k <= kBoundK) {
        // ---- each thread's largest key (0, below every logit's key, if none)
        uint32_t mx = 0u;
        if ((reinterpret_cast<uintptr_t>(row) & 15u) == 0) {
            const int n4 = n >> 2;
            const uint4* row4 = reinterpret_cast<const uint4*>(row);
            constexpr int kUnroll = 8;
            for (int j0 = tid; j0 < n4; j0 += kMaskThreads * kUnroll) {
                uint4 v[kUnroll];
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    const int j = j0 + u * kMaskThreads;
                    v[u] = j < n4 ? __ldg(row4 + j) : make_uint4(0u, 0u, 0u, 0u);
                }
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    if (j0 + u * kMaskThreads < n4)
                        mx = max(mx, max(max(key_of(v[u].x), key_of(v[u].y)),
                                         max(key_of(v[u].z), key_of(v[u].w))));
                }
            }
            for (int i = 4 * n4 + tid; i < n; i += kMaskThreads)
                mx = max(mx, key_of(__ldg(row + i)));
        } else {
            for (int i = tid; i < n; i += kMaskThreads)
                mx = max(mx, key_of(__ldg(row + i)));
        }
        // ---- bound: the k-th largest of the threads' maxima
        const uint32_t sorted = block_sort_ascending(mx, loc.sortbuf);
        if (tid == kMaskThreads - k)
            loc.bound = sorted;
        if (tid == 0)
            loc.n = 0;
        __syncthreads();
        const uint32_t bound = loc.bound;
        // ---- the keys at or above it (a second sweep; the slice is in L2 now)
        auto collect = [&](bool hit, uint32_t kv, int i) {
            const unsigned hits = __ballot_sync(0xffffffffu, hit);
            if (hits != 0u) {
                int base = 0;
                if (lane == 0)
                    base = atomicAdd(&loc.n, __popc(hits));
                base = __shfl_sync(0xffffffffu, base, 0) + __popc(hits & ((1u << lane) - 1u));
                if (hit && base < kFilterCap)
                    loc.comp[base] = composite(kv, i);
            }
        };
        {
            int done = 0;
            if ((reinterpret_cast<uintptr_t>(row) & 15u) == 0) {
                const int n4 = n >> 2;
                const uint4* row4 = reinterpret_cast<const uint4*>(row);
                constexpr int kUnroll = 4;
                for (int j0 = w * 32; j0 < n4; j0 += kMaskThreads * kUnroll) {
                    uint4 v[kUnroll];
#pragma unroll
                    for (int u = 0; u < kUnroll; ++u) {
                        const int j = j0 + u * kMaskThreads + lane;
                        v[u] = j < n4 ? __ldg(row4 + j) : make_uint4(0u, 0u, 0u, 0u);
                    }
#pragma unroll
                    for (int u = 0; u < kUnroll; ++u) {
                        const int j = j0 + u * kMaskThreads + lane;
                        const bool in = j < n4;
                        const uint32_t k0 = key_of(v[u].x), k1 = key_of(v[u].y);
                        const uint32_t k2 = key_of(v[u].z), k3 = key_of(v[u].w);
                        collect(in && k0 >= bound, k0, 4 * j);
                        collect(in && k1 >= bound, k1, 4 * j + 1);
                        collect(in && k2 >= bound, k2, 4 * j + 2);
                        collect(in && k3 >= bound, k3, 4 * j + 3);
                    }
                }
                done = 4 * n4;
            }
            for (int i0 = done + w * 32; i0 < n; i0 += kMaskThreads) {
                const int i = i0 + lane;
                const uint32_t kv = i < n ? key_of(__ldg(row + i)) : 0u;
                collect(i < n && kv >= bound, kv, i);
            }
        }
        __syncthreads();
        const int C = loc.n;
        if (C <= kFilterCap) {
            for (int c = tid; c < C; c += kMaskThreads) {
                const uint64_t cc = loc.comp[c];
                const int better = rank_in(loc.comp, C, cc);
                if (better < k) {
                    loc.cand_key[better] = comp_key(cc);
                    loc.cand_idx[better] = comp_col(cc);
                }
            }
            __syncthreads();
            return;
        }
    }
    // ---- larger k, or a bound that lets too many keys through: radix selection
    using Keys = selcore::GlobalKeys<selcore::ValueOrderKey>;
    selcore::radix_select<false>(row, nullptr, Keys{row, key_of}, key_of, n, k, loc.cand_idx, sh);
    __syncthreads();
    for (int i = tid; i < k; i += kMaskThreads)
        loc.cand_key[i] = key_of(__ldg(row + loc.cand_idx[i]));
    __syncthreads();
}

}  // namespace

__global__ void __launch_bounds__(kMaskThreads, 1) topk_topp_kernel(MaskArgs a)
{
    extern __shared__ __align__(16) unsigned char mask_smem[];
    MaskShared& sh = *reinterpret_cast<MaskShared*>(mask_smem);   // radix state, candidate map
    __shared__ MaskCluster mc;
    __shared__ MaskLocal loc;
    __shared__ MaskMerge mm;
    cluster_arrive_relaxed();                     // paired with the wait before the first remote store
    const int tid = threadIdx.x;
    const uint32_t rank = cluster_rank();
    const int b = blockIdx.x / kMaskCtas;
    const int lo = min(a.V, (int)rank * a.slice), hi = min(a.V, lo + a.slice), n = hi - lo;
    const float* xrow = a.x + (int64_t)b * a.x_stride;
    const uint32_t* row = reinterpret_cast<const uint32_t*>(xrow) + lo;
    const int K = min(a.k, a.V);
    const selcore::ValueOrderKey key_of{};

    // ---- this slice's top-k (all of it when it has no more than k)
    int cn;
    if (n > a.k) {
        slice_top_k(row, n, a.k, loc, sh);
        cn = a.k;
    } else {
        for (int i = tid; i < n; i += kMaskThreads) {
            loc.cand_key[i] = key_of(__ldg(row + i));
            loc.cand_idx[i] = i;
        }
        __syncthreads();
        cn = n;
    }

    // ---- candidates into rank 0's shared memory
    cluster_wait();
    if (tid == 0)
        st_dsmem(dsmem(&mc.cnt[rank], 0), (uint32_t)cn);
    for (int i = tid; i < cn; i += kMaskThreads) {
        const int slot = (int)rank * kMaskKMax + i;
        st_dsmem(dsmem(&mc.key[slot], 0), loc.cand_key[i]);
        st_dsmem(dsmem(&mc.idx[slot], 0), (uint32_t)(lo + loc.cand_idx[i]));
    }
    cluster_arrive();

    // ---- meanwhile: -inf over the slice except this CTA's candidates
    uint32_t* cand_map = sh.above_map;                 // bit i: column lo + i is a candidate
    const int nw = (n + 31) >> 5;
    for (int w = tid; w < nw; w += kMaskThreads)
        cand_map[w] = 0u;
    __syncthreads();
    for (int i = tid; i < cn; i += kMaskThreads)
        atomicOr(&cand_map[loc.cand_idx[i] >> 5], 1u << (loc.cand_idx[i] & 31));
    __syncthreads();
    float* orow = a.out + (int64_t)b * a.out_stride + lo;
    const float* xs = xrow + lo;
    const float ninf = -INFINITY;
    if ((reinterpret_cast<uintptr_t>(orow) & 15u) == 0) {
        const int n4 = n >> 2;
        for (int i4 = tid; i4 < n4; i4 += kMaskThreads) {
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
        for (int i = 4 * n4 + tid; i < n; i += kMaskThreads)
            if (!((cand_map[i >> 5] >> (i & 31)) & 1u))
                orow[i] = ninf;
    } else {
        for (int i = tid; i < n; i += kMaskThreads)
            if (!((cand_map[i >> 5] >> (i & 31)) & 1u))
                orow[i] = ninf;
    }
    cluster_wait();

    // ---- rank 0: the row's top-k and top-p; kept columns into every CTA
    if (rank == 0) {
        if (tid == 0) {
            mm.base[0] = 0;
            for (int r = 0; r < kMaskCtas; ++r)
                mm.base[r + 1] = mm.base[r] + mc.cnt[r];
        }
        __syncthreads();
        for (int r = 0; r < kMaskCtas; ++r) {
            for (int i = tid; i < mc.cnt[r]; i += kMaskThreads)
                mm.comp[mm.base[r] + i] = composite(mc.key[r * kMaskKMax + i],
                                                    mc.idx[r * kMaskKMax + i]);
        }
        __syncthreads();
        const int T = mm.base[kMaskCtas];
        for (int c = tid; c < T; c += kMaskThreads) {
            const int better = rank_in(mm.comp, T, mm.comp[c]);
            if (better < K)
                mm.order[better] = c;
        }
        __syncthreads();
        // FP64 masses of the top-K logits (their values are their keys mapped back)
        const float x0f = key_value(comp_key(mm.comp[mm.order[0]]));
        const bool usable = !(isnan(x0f) || isinf(x0f));   // -inf, +inf or NaN at the top
        if (usable) {
            const double x0 = (double)x0f;
            for (int j = tid; j < K; j += kMaskThreads)
                mm.s[j] = exp((double)key_value(comp_key(mm.comp[mm.order[j]])) - x0);
        }
        __syncthreads();
        if (tid == 0) {
            int m = K;
            if (usable) {
                double acc = 0.0;
                for (int j = K - 1; j >= 0; --j) {
                    acc = mm.s[j] + acc;
                    mm.s[j] = acc;
                }
                const double cut = (1.0 - (double)a.p) * mm.s[0];
                m = 0;
                while (m < K && mm.s[m] > cut)
                    ++m;
            } else if (!(x0f == -INFINITY)) {
                raise_flag(a.err, PAGED_GQA_FLAG_BAD_LOGIT);
            }
            mm.m = m;
        }
        __syncthreads();
        const int m = mm.m;
        for (int t = tid; t < kMaskCtas * (m + 1); t += kMaskThreads) {
            const int r = t / (m + 1), j = t - r * (m + 1);
            if (j == m)
                st_dsmem(dsmem(&mc.kept_n, r), (uint32_t)m);
            else
                st_dsmem(dsmem(&mc.kept_idx[j], r), (uint32_t)comp_col(mm.comp[mm.order[j]]));
        }
    }
    cluster_arrive();
    cluster_wait();

    // ---- this CTA's candidates: kept ones carry their logit, the others -inf
    const int m = mc.kept_n;
    const bool in_place = orow == xs;
    for (int i = tid; i < cn; i += kMaskThreads) {
        const int col = lo + loc.cand_idx[i];
        bool keep = false;
        for (int j = 0; j < m; ++j)
            keep |= mc.kept_idx[j] == col;
        if (!keep)
            orow[loc.cand_idx[i]] = ninf;
        else if (!in_place)
            orow[loc.cand_idx[i]] = xs[loc.cand_idx[i]];
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
                                 (int)sizeof(MaskShared));
        if (e != cudaSuccess)
            return e;
        if (dev < kMaxDevices)
            done[dev].store(1, std::memory_order_release);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.B * kMaskCtas);
    cfg.blockDim = dim3(kMaskThreads);
    cfg.dynamicSmemBytes = sizeof(MaskShared);
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
