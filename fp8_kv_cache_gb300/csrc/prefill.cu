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
// row's 16-token tiles (four block entries each) round-robin; each lane of
// 0..15 resolves one token (selected block id -> token -> page -> row
// address) so the gather is done by the same register-direct tensor-core
// pipeline as decode, then the warps merge through shared memory and the CTA
// writes the row's FP16 outputs.  No table of virtual pages is built: the
// four-token block addresses are computed inline.
#include "pgqa_internal.h"

namespace pgqa {

template <bool kE4M3>
__global__ void __launch_bounds__(kThreads, 2) sparse_prefill_kernel(PrefillArgs a)
{
    __shared__ MergeSmem sm;
    const int r = blockIdx.x, j = blockIdx.y;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int g = lane >> 2, q = lane & 3;
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
    const int n_halves = (a.n_sel + 1 + 1) / 2;  // selected entries + the tail entry, 2 per half
    const int32_t* sel_row = a.sel + (size_t)r * a.n_sel;

    using Core = WarpCore<kE4M3>;
    uint2* qs = q_stage(sm, w);
    Core::stage_q(qs, a.q + ((size_t)r * a.Hq + (size_t)j * a.G) * kD, a.G, lane);
    Core wc;
    wc.reset();
    // half-tile h = block entries 2h, 2h+1 (8 tokens); lane t < 8 resolves token t
    auto offsets = [&](int h, int64_t& ok, int64_t& o0, int64_t& o1) {
        int64_t off = -1;
        if (lane < kHalf) {
            const int t = prefill_token(sel_row, a.n_sel, own, p, 2 * h + (lane >> 2), lane & 3,
                                        flags);
            if (t >= 0)
                off = token_row_offset(a.kv, a.bt, t, j, flags);
        }
        ok = __shfl_sync(0xffffffffu, off, g);
        o0 = __shfl_sync(0xffffffffu, off, 2 * q);
        o1 = __shfl_sync(0xffffffffu, off, 2 * q + 1);
    };
    run_halves<kE4M3, kRing<kE4M3>()>(wc, qs, a.kv.k, a.kv.v, w, n_halves, kWarps, g < a.G,
                                      a.scale_log2, lane, offsets);
    cta_merge<kE4M3>(sm, wc, a.G, a.v_scale, out_rows, nullptr);
    raise_flag(a.err, flags);
}

cudaError_t launch_prefill(const PrefillArgs& a, bool e4m3, cudaStream_t s)
{
    const dim3 grid(a.R, a.Hkv);
    if (e4m3)
        sparse_prefill_kernel<true><<<grid, kThreads, 0, s>>>(a);
    else
        sparse_prefill_kernel<false><<<grid, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace pgqa
