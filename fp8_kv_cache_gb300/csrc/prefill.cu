// prefill.cu -- selected-sparse paged prefill over four-token blocks.
//
// Operation: "[Kernel][SM70] Accelerate Qwen3.8 QSA paged prefill"
// (1Cat-vLLM #378), Changes: every query row attends to its selected
// four-token blocks, read in place from the page-16 cache (a four-token block
// never straddles a page because page_size is a multiple of 4), followed by
// its own causal partial block; padded or stale positions are clamped and
// invalid rows are inert.  Contiguous and interleaved K/V strides are both
// plain strides here.
//
// Design (ours): one CTA per (query row, KV head).  Its four warps take the
// row's 16-token tiles (four block entries each) round-robin; for each half
// of a tile, lane t of 0..7 resolves token t (selected block id -> token ->
// page -> row address) and the warp copies the K and V rows into its
// shared-memory ring with 16-byte asynchronous copies, so the gather runs
// through the same tensor-core
// pipeline as decode; the warps then merge through shared memory and the CTA
// writes the row's FP16 outputs.  No table of virtual pages is built: the
// four-token block addresses are computed inline.
#include <atomic>

#include "pgqa_internal.h"

namespace pgqa {

template <bool kE4M3>
__global__ void __launch_bounds__(kThreads, kMinCtas<kE4M3>()) sparse_prefill_kernel(PrefillArgs a)
{
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const int r = blockIdx.x, j = blockIdx.y;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int flags = 0;
    __half* out_rows = a.out + ((size_t)r * a.Hq + (size_t)j * a.G) * kD;

    int p = __ldg(a.q_pos + r);
    if (p < 0 || a.kv_len <= 0) {
        for (int i = threadIdx.x; i < a.G * kD; i += blockDim.x)
            out_rows[i] = __float2half_rn(0.f);
        if (threadIdx.x == 0)
            raise_flag(a.err, PAGED_GQA_FLAG_EMPTY_ROW);
        return;
    }
    if (p >= a.kv_len) {
        p = a.kv_len - 1;
        if (threadIdx.x == 0)
            flags |= PAGED_GQA_FLAG_QPOS_CLAMPED;
    }
    const int own = p >> 2;
    const int32_t* sel_row = a.sel + (size_t)r * a.n_sel;

    // FP16 rows leave registers to spare: the Q fragments stay in registers.
    using Core = WarpCore<kE4M3, !kE4M3>;
    const CtaSmem<kE4M3> cs = CtaSmem<kE4M3>::carve(smem_raw, w);
    WarpRing<kE4M3, kStages<kE4M3>()> rg;
    rg.init(cs.ring, cs.masks);
    Core::stage_q(cs.qs, a.q + ((size_t)r * a.Hq + (size_t)j * a.G) * kD, a.G, lane, w, kWarps);
    Core wc;
    wc.reset();
    bool q_loaded = false;
    // Chunks of block entries (selected blocks, then the tail entry): the CTA
    // resolves a chunk's entries (selection index -> block -> page) into the
    // address table first, so the ring fills need no dependent global load.
    int2* tab = reinterpret_cast<int2*>(cs.tail);
    constexpr int kCap = SmemPlan<kE4M3>::kPrefillEntries;   // a multiple of 4
    const int n_entries = a.n_sel + 1;
    for (int e0 = 0; e0 < n_entries; e0 += kCap) {
        const int e1 = min(n_entries, e0 + kCap);
        __syncthreads();                             // Q staged / previous chunk done with tab
        for (int e = e0 + (int)threadIdx.x; e < e1; e += blockDim.x) {
            int first, page;
            prefill_entry(a.kv, a.bt, sel_row, a.n_sel, own, e, first, page, flags);
            tab[e - e0] = make_int2(first, page);
        }
        __syncthreads();
        if (!q_loaded) {
            wc.load_q(cs.qs, lane);                  // Q staged before the first chunk's barrier
            q_loaded = true;
        }
        // half-tile h = block entries 2h, 2h+1 (8 tokens); lane t < 8 takes token t
        auto offset = [&](int h) -> int64_t {
            if (lane < kHalf) {
                const int e = 2 * h + (lane >> 2), u = lane & 3;
                if (e < e1) {
                    const int2 en = tab[e - e0];
                    if (prefill_lane_live(en.y, e, a.n_sel, en.x, u, p)) {
                        int pi, slot;
                        page_and_slot(a.kv, en.x + u, pi, slot);
                        return row_offset(a.kv, en.y, slot, j);
                    }
                }
            }
            return -1;
        };
        run_tiles<kE4M3, kStages<kE4M3>(), decltype(offset), !kE4M3>(
            wc, rg, cs.qs, a.kv.k, a.kv.v, e0 / 4 + w, (e1 + 3) / 4, kWarps, a.G, a.scale_log2,
            lane, offset);
    }
    cta_merge<kE4M3, !kE4M3>(*cs.merge, wc, a.G, a.v_scale, out_rows, nullptr);
    raise_flag(a.err, flags);
}

// Dynamic shared-memory opt-in, once per device and instantiation.
template <bool kE4M3>
static cudaError_t prefill_smem_attr()
{
    static std::atomic<int> done[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < kMaxDevices && done[dev].load(std::memory_order_acquire))
        return cudaSuccess;
    e = cudaFuncSetAttribute(sparse_prefill_kernel<kE4M3>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SmemPlan<kE4M3>::kPrefillSmem);
    if (e == cudaSuccess && dev < kMaxDevices)
        done[dev].store(1, std::memory_order_release);
    return e;
}

cudaError_t launch_prefill(const PrefillArgs& a, bool e4m3, cudaStream_t s)
{
    cudaError_t e = e4m3 ? prefill_smem_attr<true>() : prefill_smem_attr<false>();
    if (e != cudaSuccess)
        return e;
    const dim3 grid(a.R, a.Hkv);
    if (e4m3)
        sparse_prefill_kernel<true><<<grid, kThreads, SmemPlan<true>::kPrefillSmem, s>>>(a);
    else
        sparse_prefill_kernel<false><<<grid, kThreads, SmemPlan<false>::kPrefillSmem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace pgqa
