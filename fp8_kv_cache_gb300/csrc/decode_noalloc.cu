// decode_noalloc.cu -- paged_gqa_decode for callers that cannot allocate.
//
// paged_gqa_decode takes its split-KV scratch from a workspace the caller
// allocates.  Some callers cannot do that: a plugin or extension whose
// execute hook runs inside a host framework that owns all device memory and
// forbids allocations there, code on a latency-critical path where a
// cudaMalloc could synchronise the device, or a process whose device memory
// has already been handed out to another allocator.  This entry point gives
// them the same decode with the scratch held in one file-scope device array,
// so the call itself allocates nothing (no cudaMalloc, no cudaFree, no
// allocating library routine).
//
// The array costs kNoAllocScratchBytes (16 MiB) of device memory on every GPU
// where this library's device code is loaded, for the life of the process.
// With the CUDA runtime's lazy module loading (its default), that happens on
// the first call of this entry point on each device, inside the address
// lookup below: that first call is where the driver reserves the 16 MiB, so
// it can fail for lack of memory and can synchronise.  Callers should make
// one warm-up call per device at initialisation, before any stream capture
// and outside any hook where allocation is forbidden; later calls allocate
// nothing.  Every call shares the array, so calls whose kernels could
// overlap on the GPU (for example on two streams without ordering between
// them) race on it; calls on one stream, or otherwise ordered, are safe.
// Nothing in it has to start at zero: each call writes every scratch value
// it later reads (the tile prefix, the split count and the partial results
// it merges), so the contents a previous call left behind are never read.
#include <atomic>

#include "pgqa_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)16 << 20;

static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

// Device address of g_decode_scratch, looked up once per device with that
// device current (a host-side name of a __device__ variable is not a device
// address and must never be handed to a kernel).
void* scratch_address(int& status)
{
    static std::atomic<void*> addr[pgqa::kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= pgqa::kMaxDevices) {
        status = PAGED_GQA_ERR_CUDA;
        return nullptr;
    }
    void* p = addr[dev].load(std::memory_order_acquire);
    if (p != nullptr)
        return p;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) {
        status = PAGED_GQA_ERR_CUDA;
        return nullptr;
    }
    addr[dev].store(p, std::memory_order_release);
    return p;
}

}  // namespace

extern "C" int paged_gqa_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                        paged_gqa_kv_layout kv_layout, int kv_dtype,
                                        const int32_t* block_table, int64_t bt_row_stride,
                                        const int32_t* seq_lens, int B, int Hq, int Hkv, int D,
                                        int page_size, int num_pages, int max_seq_len,
                                        float kv_scale, float softmax_scale, void* out,
                                        int* err_flag, void* stream)
{
    // Shapes whose split scratch, for this KV dtype, would not fit the
    // static array are refused before anything is looked up or launched
    // (paged_gqa_decode checks the same size again before its launches).
    if (B > 0) {
        const size_t need = pgqa::decode_workspace_bytes_for(B, Hq, Hkv, D, kv_dtype);
        if (need > kNoAllocScratchBytes)
            return PAGED_GQA_ERR_WORKSPACE;
    }
    int status = PAGED_GQA_OK;
    void* scratch = scratch_address(status);
    if (scratch == nullptr)
        return status;
    paged_gqa_workspace ws{};
    ws.ptr = scratch;
    ws.bytes = kNoAllocScratchBytes;
    ws.force_splits = 0;
    ws.err_flag = err_flag;
    return paged_gqa_decode(q, k_cache, v_cache, kv_layout, kv_dtype, block_table, bt_row_stride,
                            seq_lens, B, Hq, Hkv, D, page_size, num_pages, max_seq_len, kv_scale,
                            softmax_scale, out, &ws, stream);
}
