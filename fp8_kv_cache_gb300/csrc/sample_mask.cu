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
// handful of rows still spreads over the GPU.  Each CTA stages its slice of
// the row (keys whose unsigned order is the numeric order of the logits) in
// shared memory and finds the slice's own top-k with the radix selection of
// select_core.cuh; the global top-k is among the union of those candidate
// lists.  After a cluster barrier, rank 0 reads every CTA's candidates
// through distributed shared memory (mapa + ld.shared::cluster), ranks them
// (larger key first, equal keys by index), and runs the FP64 top-p over the
// first min(k, V); after a second barrier every CTA reads the kept list from
// rank 0 and writes its slice: -infinity everywhere except the kept logits,
// which keep their bits.  A last barrier keeps rank 0's shared memory alive
// until every CTA has read it.  HBM traffic: the row read once, written once.
#include <atomic>

#include "select_core.cuh"

namespace pgqa {

namespace {

constexpr int kMaskThreads = 512;
constexpr int kMaskCtas = 8;            // CTAs per row: one cluster
constexpr int kMaskSliceMax = 40960;    // logits a CTA stages (160 KB)
constexpr int kMaskKMax = 128;          // largest k served
using MaskShared = selcore::SelectShared<kMaskThreads, kMaskSliceMax / 32>;

// Per-CTA state read across the cluster.
struct MaskCluster {
    int32_t cand_n;
    int32_t kept_n;                         // rank 0: logits kept in the row
    int32_t cand_idx[kMaskKMax];            // column of each candidate
    uint32_t cand_key[kMaskKMax];
    int32_t kept_idx[kMaskKMax];            // rank 0: their columns
};

// Rank 0's scratch for ranking the cluster's candidates.
struct MaskMerge {
    int32_t base[kMaskCtas + 1];
    int32_t cnt[kMaskCtas];
    uint32_t key[kMaskCtas * kMaskKMax];
    int32_t idx[kMaskCtas * kMaskKMax];
    int32_t order[kMaskKMax];               // candidate at each rank
    double s[kMaskKMax];                    // e_j, then the suffix sums S_j
    int32_t m;
};

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Every thread of every CTA of the cluster; orders the shared-memory writes
// before it against the reads after it, across the cluster.
__device__ __forceinline__ void cluster_barrier()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t dsmem(const void* p, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}

__device__ __forceinline__ uint32_t ld_dsmem(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

}  // namespace

__global__ void __launch_bounds__(kMaskThreads, 1) topk_topp_kernel(MaskArgs a)
{
    extern __shared__ __align__(16) unsigned char mask_smem[];
    __shared__ MaskShared sh;
    __shared__ MaskCluster mc;
    __shared__ MaskMerge mm;
    const int tid = threadIdx.x;
    const uint32_t rank = cluster_rank();
    const int b = blockIdx.x / kMaskCtas;
    const int lo = min(a.V, (int)rank * a.slice), hi = min(a.V, lo + a.slice), n = hi - lo;
    const float* xrow = a.x + (int64_t)b * a.x_stride;
    const uint32_t* row = reinterpret_cast<const uint32_t*>(xrow) + lo;
    const int K = min(a.k, a.V);
    const selcore::ValueOrderKey key_of{};

    // ---- this slice's top-k candidates (all of it when it has no more than k)
    if (n > a.k) {
        uint32_t* stage = reinterpret_cast<uint32_t*>(mask_smem);
        selcore::radix_select<true>(row, stage, selcore::StagedKeys{stage}, key_of, n, a.k,
                                    mc.cand_idx, sh);
        __syncthreads();
        for (int i = tid; i < a.k; i += kMaskThreads) {
            const int li = mc.cand_idx[i];
            mc.cand_key[i] = stage[li];
            mc.cand_idx[i] = lo + li;
        }
        if (tid == 0)
            mc.cand_n = a.k;
    } else {
        for (int i = tid; i < n; i += kMaskThreads) {
            mc.cand_key[i] = key_of(__ldg(row + i));
            mc.cand_idx[i] = lo + i;
        }
        if (tid == 0)
            mc.cand_n = n;
    }
    cluster_barrier();

    // ---- rank 0: the row's top-k and top-p
    if (rank == 0) {
        if (tid < kMaskCtas)
            mm.cnt[tid] = (int32_t)ld_dsmem(dsmem(&mc.cand_n, tid));
        __syncthreads();
        if (tid == 0) {
            mm.base[0] = 0;
            for (int r = 0; r < kMaskCtas; ++r)
                mm.base[r + 1] = mm.base[r] + mm.cnt[r];
        }
        __syncthreads();
        for (int r = 0; r < kMaskCtas; ++r) {
            for (int i = tid; i < mm.cnt[r]; i += kMaskThreads) {
                mm.key[mm.base[r] + i] = ld_dsmem(dsmem(&mc.cand_key[i], r));
                mm.idx[mm.base[r] + i] = (int32_t)ld_dsmem(dsmem(&mc.cand_idx[i], r));
            }
        }
        __syncthreads();
        const int T = mm.base[kMaskCtas];
        for (int c = tid; c < T; c += kMaskThreads) {
            const uint32_t kc = mm.key[c];
            const int ic = mm.idx[c];
            int better = 0;
            for (int u = 0; u < T; ++u) {
                const uint32_t ku = mm.key[u];
                better += ku > kc || (ku == kc && mm.idx[u] < ic);
            }
            if (better < K)
                mm.order[better] = c;
        }
        __syncthreads();
        // FP64 masses of the top-K logits, read back from the row itself
        const float x0f = __ldg(xrow + mm.idx[mm.order[0]]);
        const bool usable = !(isnan(x0f) || isinf(x0f));   // -inf, +inf or NaN at the top
        if (usable) {
            const double x0 = (double)x0f;
            for (int j = tid; j < K; j += kMaskThreads)
                mm.s[j] = exp((double)__ldg(xrow + mm.idx[mm.order[j]]) - x0);
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
            mc.kept_n = m;
        }
        __syncthreads();
        for (int j = tid; j < mm.m; j += kMaskThreads)
            mc.kept_idx[j] = mm.idx[mm.order[j]];
    }
    cluster_barrier();

    // ---- this slice: -inf except the kept logits
    const int m = (int)ld_dsmem(dsmem(&mc.kept_n, 0));
    uint32_t* kept = sh.above_map;                      // free again: bit i = column lo + i kept
    const int nw = (n + 31) >> 5;
    for (int w = tid; w < nw; w += kMaskThreads)
        kept[w] = 0u;
    __syncthreads();
    for (int j = tid; j < m; j += kMaskThreads) {
        const int col = (int)ld_dsmem(dsmem(&mc.kept_idx[j], 0));
        if (col >= lo && col < hi)
            atomicOr(&kept[(col - lo) >> 5], 1u << ((col - lo) & 31));
    }
    __syncthreads();
    float* orow = a.out + (int64_t)b * a.out_stride + lo;
    const float* xs = xrow + lo;
    const bool in_place = orow == xs;
    const float ninf = -INFINITY;
    if ((reinterpret_cast<uintptr_t>(orow) & 15u) == 0) {
        const int n4 = n >> 2;
        for (int i4 = tid; i4 < n4; i4 += kMaskThreads) {
            const uint32_t bits = (kept[i4 >> 3] >> ((i4 & 7) * 4)) & 15u;
            if (bits == 0u) {
                reinterpret_cast<float4*>(orow)[i4] = make_float4(ninf, ninf, ninf, ninf);
            } else {
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int i = 4 * i4 + u;
                    if (!((bits >> u) & 1u))
                        orow[i] = ninf;
                    else if (!in_place)
                        orow[i] = xs[i];
                }
            }
        }
        for (int i = 4 * n4 + tid; i < n; i += kMaskThreads) {
            const bool k1 = (kept[i >> 5] >> (i & 31)) & 1u;
            if (!k1)
                orow[i] = ninf;
            else if (!in_place)
                orow[i] = xs[i];
        }
    } else {
        for (int i = tid; i < n; i += kMaskThreads) {
            const bool k1 = (kept[i >> 5] >> (i & 31)) & 1u;
            if (!k1)
                orow[i] = ninf;
            else if (!in_place)
                orow[i] = xs[i];
        }
    }
    cluster_barrier();                                  // rank 0's lists were read by all
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
                                 (int)(kMaskSliceMax * sizeof(uint32_t)));
        if (e != cudaSuccess)
            return e;
        if (dev < kMaxDevices)
            done[dev].store(1, std::memory_order_release);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.B * kMaskCtas);
    cfg.blockDim = dim3(kMaskThreads);
    cfg.dynamicSmemBytes = (size_t)a.slice * sizeof(uint32_t);
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
