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
// Design (ours): one CTA of 256 threads per row runs the radix selection of
// select_core.cuh over the row's candidate scores.  The scores are read as
// 32-bit patterns and keyed by IEEE totalOrder (flip the sign bit of
// non-negative values, all bits of negative ones), so every pattern has its
// place; a row's keys are staged in 64 KB of shared memory at most.
#include <atomic>

#include "select_core.cuh"

namespace pgqa {

namespace {

constexpr int kSelThreads = 256;
constexpr int kStageMax = 16384;     // keys staged in shared memory, at most (64 KB)
using SelShared = selcore::SelectShared<kSelThreads, kStageMax / 32>;

}  // namespace

__global__ void __launch_bounds__(kSelThreads, 4) qsa_select_kernel(SelectArgs a)
{
    extern __shared__ __align__(16) unsigned char sel_smem[];
    __shared__ SelShared sh;
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
        selcore::radix_select<true>(row, stage, selcore::StagedKeys{stage},
                                    selcore::TotalOrderKey{}, n, a.k, out, sh);
    } else {
        using Keys = selcore::GlobalKeys<selcore::TotalOrderKey>;
        selcore::radix_select<false>(row, nullptr, Keys{row, {}}, selcore::TotalOrderKey{}, n,
                                     a.k, out, sh);
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
