// inspect.cu -- inspection kernels that expose the gather and dequantisation
// of the attention kernels, so tests can compare them bit for bit.
//
// They call the very device functions the attention kernels use:
// page_and_slot / table_page / row_offset (block table -> page -> row
// address), prefill_entry / prefill_lane_live (selected block entry -> tokens,
// "[Kernel][SM70] Accelerate Qwen3.8 QSA paged prefill", Changes), and the
// E4M3 converter e4m3x4_to_f16x2x2 ("[Kernel][SM70] Scale NVFP4 E4M3 decode
// batches", Purpose).
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
