// inspect.cu -- inspection kernels that expose the gather and dequantisation
// of the attention kernels, so tests can compare them bit for bit.
//
// They call the very device functions the attention kernels use:
// page_and_slot / table_page / row_offset (block table -> page -> row
// address), prefill_entry / prefill_lane_live (selected block entry -> tokens,
// "[Kernel][SM70] Accelerate Qwen3.8 QSA paged prefill", Changes), and the
// E4M3 converter e4m3x4_to_f16x2x2 ("[Kernel][SM70] Scale NVFP4 E4M3 decode
// batches", Purpose).
#include <atomic>

#include "pgqa_internal.h"

namespace pgqa {

// grid (ceil(T / 16), B, Hkv), one warp: rows of 16 tokens of one KV head.
template <bool kE4M3>
__global__ void __launch_bounds__(32) gather_kernel(KVGeom g, const int32_t* bt, int64_t bt_stride,
                                                    const int32_t* seq_lens, int T, int Hkv,
                                                    int max_seq_len, float kv_scale, float* out)
{
    const int tile = blockIdx.x, b = blockIdx.y, j = blockIdx.z;
    const int lane = threadIdx.x;
    int flags = 0;
    int L = __ldg(seq_lens + b);
    L = L < 0 ? 0 : (L > max_seq_len ? max_seq_len : L);
    int64_t off = -1;
    if (lane < kTile) {
        const int t = tile * kTile + lane;
        if (t < L)
            off = token_row_offset(g, bt + (int64_t)b * bt_stride, t, j, flags);
    }
    for (int i = 0; i < kTile; ++i) {
        const int t = tile * kTile + i;
        const int64_t o = __shfl_sync(0xffffffffu, off, i);
        if (t >= T)
            break;
        float* dst = out + (((int64_t)b * T + t) * Hkv + j) * kD;
        if (kE4M3) {
            // 256 codes: lanes 0..15 take 16 codes each
            if (lane < 16) {
                uint4 c = o >= 0 ? ldg_stream(g.k + o + 16 * lane) : make_uint4(0, 0, 0, 0);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    uint32_t lo, hi;
                    e4m3x4_to_f16x2x2(word(c, k), lo, hi);
                    const float2 f0 = __half22float2(*reinterpret_cast<__half2*>(&lo));
                    const float2 f1 = __half22float2(*reinterpret_cast<__half2*>(&hi));
                    float4 v = make_float4(f0.x * kv_scale, f0.y * kv_scale, f1.x * kv_scale,
                                           f1.y * kv_scale);
                    if (o < 0)
                        v = make_float4(0.f, 0.f, 0.f, 0.f);
                    reinterpret_cast<float4*>(dst + 16 * lane)[k] = v;
                }
            }
        } else {
            // 256 halves: every lane takes 8
            uint4 c = o >= 0 ? ldg_stream(g.k + o + 16 * lane) : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                uint32_t wv = word(c, k);
                const float2 f = __half22float2(*reinterpret_cast<__half2*>(&wv));
                dst[8 * lane + 2 * k] = f.x;
                dst[8 * lane + 2 * k + 1] = f.y;
            }
        }
    }
}

// grid (R), 128 threads: the token of every (entry, lane) slot of row r.
__global__ void __launch_bounds__(128) prefill_tokens_kernel(KVGeom g, const int32_t* bt, int kv_len,
                                                             const int32_t* sel, int n_sel,
                                                             const int32_t* q_pos, int32_t* out)
{
    const int r = blockIdx.x;
    const int slots = 4 * (n_sel + 1);
    int32_t* dst = out + (int64_t)r * slots;
    int p = __ldg(q_pos + r);
    int flags = 0;
    for (int s = threadIdx.x; s < slots; s += blockDim.x) {
        int t = -1;
        if (p >= 0 && kv_len > 0) {
            const int pc = p >= kv_len ? kv_len - 1 : p;
            const int e = s >> 2, u = s & 3;
            int first, page;
            prefill_entry(g, bt, sel + (int64_t)r * n_sel, n_sel, pc >> 2, e, first, page, flags);
            if (prefill_lane_live(page, e, n_sel, first, u, pc))
                t = first + u;
        }
        dst[s] = t;
    }
}

// The gather of sparse_prefill_kernel alone (grid R x Hkv, 4 warps, the same
// per-warp shared-memory rings, entry table and launch shape), with the
// attention arithmetic replaced by an XOR over every 32-bit word of the K and
// V rows the warp copied: its time is the ceiling of that gather, and the
// fold makes the copies observable (out[r * Hkv + j]).
template <bool kE4M3>
__global__ void __launch_bounds__(kThreads, kMinCtas<kE4M3>()) sparse_gather_kernel(PrefillArgs a,
                                                                                   uint32_t* out)
{
    extern __shared__ __align__(128) unsigned char smem_raw[];
    using St = Stage<kE4M3>;
    const int r = blockIdx.x, j = blockIdx.y;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    __shared__ uint32_t fold_s[kWarps];
    int flags = 0;
    int p = __ldg(a.q_pos + r);
    uint32_t fold = 0u;
    if (p >= 0 && a.kv_len > 0) {
        if (p >= a.kv_len)
            p = a.kv_len - 1;
        const int own = p >> 2;
        const int32_t* sel_row = a.sel + (size_t)r * a.n_sel;
        const CtaSmem<kE4M3> cs = CtaSmem<kE4M3>::carve(smem_raw, w);
        constexpr int kNS = kStages<kE4M3>();
        WarpRing<kE4M3, kNS> rg;
        rg.init(cs.ring, cs.masks);
        int2* tab = reinterpret_cast<int2*>(cs.tail);
        constexpr int kCap = SmemPlan<kE4M3>::kPrefillEntries;
        const int n_entries = a.n_sel + 1;
        for (int e0 = 0; e0 < n_entries; e0 += kCap) {
            const int e1 = min(n_entries, e0 + kCap);
            __syncthreads();
            for (int e = e0 + (int)threadIdx.x; e < e1; e += blockDim.x) {
                int first, page;
                prefill_entry(a.kv, a.bt, sel_row, a.n_sel, own, e, first, page, flags);
                tab[e - e0] = make_int2(first, page);
            }
            __syncthreads();
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
            // tiles first = e0/4 + w, stride kWarps, as the attention kernel's warps
            const int first = e0 / 4 + w, end = (e1 + 3) / 4;
            const int n = end > first ? (end - first + kWarps - 1) / kWarps : 0;
            const int H = 2 * n;
            auto half = [&](int jj) { return 2 * (first + (jj >> 1) * kWarps) + (jj & 1); };
            for (int jj = 0; jj < kNS; ++jj) {
                if (jj < H)
                    rg.fill(jj, offset(half(jj)), a.kv.k, a.kv.v, lane);
                else
                    rg.skip();
            }
            for (int k = 0; k < n; ++k) {
                rg.wait();
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int s = (2 * k + u) % kNS;
                    const uint32_t m = rg.masks[s];
                    // the attended rows of the stage, K then V, 16 bytes per lane at a time
                    for (int t = 0; t < kHalf; ++t) {
                        if (!((m >> t) & 1u))
                            continue;
                        for (int c = lane; c < St::kRowBytes / 16; c += 32) {
                            const uint4 kv0 = lds128(rg.addr(s) + St::k_off(t, c));
                            const uint4 kv1 = lds128(rg.addr(s) + St::v_off(t, c));
                            fold ^= kv0.x ^ kv0.y ^ kv0.z ^ kv0.w ^ kv1.x ^ kv1.y ^ kv1.z ^ kv1.w;
                        }
                    }
                }
                __syncwarp();
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int jj = 2 * k + kNS + u;
                    if (jj < H)
                        rg.fill(jj % kNS, offset(half(jj)), a.kv.k, a.kv.v, lane);
                    else
                        rg.skip();
                }
            }
            rg.drain();
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        fold ^= __shfl_xor_sync(0xffffffffu, fold, o);
    if (lane == 0)
        fold_s[w] = fold;
    __syncthreads();
    if (threadIdx.x == 0)
        out[(size_t)r * a.Hkv + j] = fold_s[0] ^ fold_s[1] ^ fold_s[2] ^ fold_s[3];
}

template <bool kE4M3>
static cudaError_t gather_probe_smem_attr()
{
    static std::atomic<int> done[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < kMaxDevices && done[dev].load(std::memory_order_acquire))
        return cudaSuccess;
    e = cudaFuncSetAttribute(sparse_gather_kernel<kE4M3>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SmemPlan<kE4M3>::kPrefillSmem);
    if (e == cudaSuccess && dev < kMaxDevices)
        done[dev].store(1, std::memory_order_release);
    return e;
}

cudaError_t launch_sparse_gather(const PrefillArgs& a, bool e4m3, uint32_t* out, cudaStream_t s)
{
    cudaError_t e = e4m3 ? gather_probe_smem_attr<true>() : gather_probe_smem_attr<false>();
    if (e != cudaSuccess)
        return e;
    const dim3 grid(a.R, a.Hkv);
    if (e4m3)
        sparse_gather_kernel<true><<<grid, kThreads, SmemPlan<true>::kPrefillSmem, s>>>(a, out);
    else
        sparse_gather_kernel<false><<<grid, kThreads, SmemPlan<false>::kPrefillSmem, s>>>(a, out);
    return cudaGetLastError();
}

cudaError_t launch_gather(const KVGeom& g, bool e4m3, const int32_t* bt, int64_t bt_stride,
                          const int32_t* seq_lens, int B, int T, int Hkv, int max_seq_len,
                          float kv_scale, float* out, cudaStream_t s)
{
    const dim3 grid((T + kTile - 1) / kTile, B, Hkv);
    if (e4m3)
        gather_kernel<true><<<grid, 32, 0, s>>>(g, bt, bt_stride, seq_lens, T, Hkv, max_seq_len,
                                                kv_scale, out);
    else
        gather_kernel<false><<<grid, 32, 0, s>>>(g, bt, bt_stride, seq_lens, T, Hkv, max_seq_len,
                                                 kv_scale, out);
    return cudaGetLastError();
}

cudaError_t launch_prefill_tokens(const KVGeom& g, const int32_t* bt, int kv_len,
                                  const int32_t* sel, int n_sel, const int32_t* q_pos, int R,
                                  int32_t* out, cudaStream_t s)
{
    prefill_tokens_kernel<<<R, 128, 0, s>>>(g, bt, kv_len, sel, n_sel, q_pos, out);
    return cudaGetLastError();
}

}  // namespace pgqa
