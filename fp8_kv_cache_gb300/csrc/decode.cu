// decode.cu -- batched paged GQA decode: split kernel + LSE-merge kernel.
//
// Operation: "[Kernel][SM70] Scale NVFP4 E4M3 decode batches" (1Cat-vLLM
// #282), Purpose: FP8-E4M3 (or FP16) KV, GQA-6, head dim 256 paged decode for
// batches of 1..16 including long contexts.
//
// Work decomposition (ours, not the page's V100 routing): every (sequence b,
// KV head j) is a segment of ceil(L_b / 16) tiles, preceded on the line by
// piece_cost virtual tiles that stand for the fixed cost of starting a piece;
// the segments are laid end to end and the resulting line is cut into C_eff
// equal ranges, one per CTA, so every CTA has the same amount of work (KV
// bytes plus piece starts) whatever the mix of sequence lengths.  The cut is
// computed on the device from seq_lens, so one launch shape serves every step
// of a captured CUDA graph.  A CTA that covers all real tiles of a segment
// writes the final FP16 rows; otherwise it writes an unnormalised partial
// (m, l, O) to slot (cta + segment) of the caller's workspace, and the merge
// kernel combines the pieces in a fixed order (no floating-point atomics, so
// results are reproducible run to run).
#include <atomic>

#include "pgqa_internal.h"

namespace pgqa {

namespace {

__device__ __forceinline__ int clamp_len(int L, int max_len)
{
    return L < 0 ? 0 : (L > max_len ? max_len : L);
}

// Largest b in [0, B) with Hkv * P[b] <= x (P non-decreasing, x < Hkv * P[B]).
__device__ __forceinline__ int find_seq(const int64_t* P, int B, int Hkv, int64_t x)
{
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((int64_t)Hkv * P[mid] <= x)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

// Line length of one segment of sequence b: its tiles plus the piece cost
// (0 for an empty sequence).
__device__ __forceinline__ int64_t seg_len(const DecodeArgs& a, int b)
{
    const int n = (clamp_len(__ldg(a.seq_lens + b), a.max_seq_len) + kTile - 1) / kTile;
    return n > 0 ? (int64_t)n + a.piece_cost : 0;
}

// CTAs that take part in the cut of a line of T > 0 tiles: at most the
// launched C and at most T, so every one of them gets a non-empty range; when
// min_tiles > 0, each gets at least min_tiles tiles, or twice that while the
// line still fills half the launched CTAs (longer ranges mean fewer pieces to
// merge and longer pipelines, which pays for long single sequences; short
// lines keep the parallelism).
__device__ __forceinline__ int64_t effective_ctas(const DecodeArgs& a, int64_t T)
{
    int64_t C = a.C;
    if (a.min_tiles > 0) {
        const int64_t c_long = T / (2 * a.min_tiles);
        C = min(C, c_long >= C / 2 ? c_long : (T + a.min_tiles - 1) / a.min_tiles);
    }
    return max((int64_t)1, min(C, T));
}

// The tiles [ta, te) of segment (b, j) processed by this CTA's warps
// (16-token tiles, round-robin), then merged into out_rows (final) or slot
// (partial).  CTA-uniform: every thread of the CTA calls it.
template <bool kE4M3>
__device__ void run_piece(const DecodeArgs& a, const CtaSmem<kE4M3, kDecodeWarps<kE4M3>()>& cs,
                          WarpRing<kE4M3, kStages<kE4M3>()>& rg, int b, int j, int L, int ta,
                          int te, __half* out_rows, float* slot, int& flags)
{
    constexpr int NW = kDecodeWarps<kE4M3>();
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    using Core = WarpCore<kE4M3>;
    Core::stage_q(cs.qs, a.q + ((size_t)b * a.Hq + (size_t)j * a.G) * kD, a.G, lane, w, NW);
    __syncthreads();
    Core wc;
    wc.reset();
    const int32_t* bt_row = a.bt + (int64_t)b * a.bt_stride;
    // The 8 lanes resolving a half-tile mostly share one block-table entry,
    // so the lookup is cheap; no address table is staged for decode (staging
    // one per piece measured slower than these direct lookups).
    auto offset = [&](int h) -> int64_t {
        if (lane < kHalf) {
            const int t = h * kHalf + lane;
            if (t < L)
                return token_row_offset(a.kv, bt_row, t, j, flags);
        }
        return -1;
    };
    run_tiles<kE4M3, kStages<kE4M3>()>(wc, rg, cs.qs, a.kv.k, a.kv.v, ta + w, te, NW, a.G,
                                       a.scale_log2, lane, offset);
    cta_merge<kE4M3, false, NW>(*cs.merge, wc, a.G, a.v_scale, out_rows, slot);
}

__device__ void zero_rows(__half* rows, int G)
{
    for (int i = threadIdx.x; i < G * kD; i += blockDim.x)
        rows[i] = __float2half_rn(0.f);
}

}  // namespace

template <bool kE4M3>
__global__ void __launch_bounds__(32 * kDecodeWarps<kE4M3>(), kMinCtas<kE4M3>())
    decode_split_kernel(DecodeArgs a)
{
    constexpr int NW = kDecodeWarps<kE4M3>(), NT = 32 * NW;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const CtaSmem<kE4M3, NW> cs = CtaSmem<kE4M3, NW>::carve(smem_raw, threadIdx.x >> 5);
    WarpRing<kE4M3, kStages<kE4M3>()> rg;
    rg.init(cs.ring, cs.masks);
    int flags = 0;
    // The merge kernel may be scheduled now; it waits for this grid's results.
    asm volatile("griddepcontrol.launch_dependents;");

    if (a.C == 0) {
        // ---- unsplit route: CTA = one whole segment
        const int k = blockIdx.x;
        const int b = k / a.Hkv, j = k - b * a.Hkv;
        const int raw = __ldg(a.seq_lens + b);
        const int L = clamp_len(raw, a.max_seq_len);
        __half* out_rows = a.out + ((size_t)b * a.Hq + (size_t)j * a.G) * kD;
        if (threadIdx.x == 0) {
            if (raw > a.max_seq_len) flags |= PAGED_GQA_FLAG_SEQ_CLAMPED;
            if (raw <= 0) flags |= PAGED_GQA_FLAG_EMPTY_ROW;
        }
        if (L == 0) {
            zero_rows(out_rows, a.G);
        } else {
            run_piece<kE4M3>(a, cs, rg, b, j, L, 0, (L + kTile - 1) / kTile, out_rows, nullptr,
                             flags);
        }
        raise_flag(a.err, flags);
        return;
    }

    // ---- split route: exclusive prefix P[b] of per-sequence tile counts
    int64_t* P = reinterpret_cast<int64_t*>(cs.tail);
    int64_t* wtot = P + (a.B + 1);
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int per = (a.B + NT - 1) / NT;
    const int b0 = min(a.B, tid * per), b1 = min(a.B, b0 + per);
    int64_t local = 0;
    for (int b = b0; b < b1; ++b) {
        const int raw = __ldg(a.seq_lens + b);
        if (blockIdx.x == 0) {
            if (raw > a.max_seq_len) flags |= PAGED_GQA_FLAG_SEQ_CLAMPED;
            if (raw <= 0) flags |= PAGED_GQA_FLAG_EMPTY_ROW;
        }
        local += seg_len(a, b);
    }
    int64_t incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int64_t t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) wtot[w] = incl;
    __syncthreads();
    int64_t base = 0, total = 0;
    for (int i = 0; i < NW; ++i) {
        if (i < w) base += wtot[i];
        total += wtot[i];
    }
    int64_t run = base + incl - local;
    for (int b = b0; b < b1; ++b) {
        P[b] = run;
        run += seg_len(a, b);
    }
    if (tid == 0) P[a.B] = total;
    __syncthreads();

    const int64_t T = (int64_t)a.Hkv * total;
    const int64_t C = T > 0 ? effective_ctas(a, T) : 0;
    if (blockIdx.x == 0 && a.B > kMergeScanMax) {
        for (int i = tid; i <= a.B; i += NT)
            a.hdr[2 + i] = P[i];
        if (tid == 0) {
            a.hdr[0] = T;
            a.hdr[1] = C;
        }
    }
    const int64_t c = blockIdx.x;
    if (c >= C || T == 0) {
        raise_flag(a.err, flags);
        return;
    }
    const int64_t x0 = c * T / C, x1 = (c + 1) * T / C;   // non-empty: C <= T
    int b = find_seq(P, a.B, a.Hkv, x0);
    int64_t nb = P[b + 1] - P[b];
    int j = (int)((x0 - (int64_t)a.Hkv * P[b]) / nb);
    for (;;) {
        const int64_t s0 = (int64_t)a.Hkv * P[b] + (int64_t)j * nb;
        if (s0 >= x1)
            break;
        const int64_t r0 = s0 + a.piece_cost, r1 = s0 + nb;   // the segment's real tiles
        if (max(x0, r0) < min(x1, r1)) {
            const int ta = (int)(max(x0, r0) - r0), te = (int)(min(x1, r1) - r0);
            const int L = clamp_len(__ldg(a.seq_lens + b), a.max_seq_len);
            const int64_t k = (int64_t)b * a.Hkv + j;
            const bool whole = x0 <= r0 && x1 >= r1;
            __half* out_rows = whole ? a.out + ((size_t)b * a.Hq + (size_t)j * a.G) * kD : nullptr;
            float* slot = whole ? nullptr : a.slots + (size_t)(c + k) * kSlotFloats;
            run_piece<kE4M3>(a, cs, rg, b, j, L, ta, te, out_rows, slot, flags);
        }
        // next non-empty segment
        if (++j == a.Hkv) {
            j = 0;
            do {
                ++b;
            } while (b < a.B && P[b + 1] == P[b]);
            if (b >= a.B)
                break;
            nb = P[b + 1] - P[b];
        }
    }
    raise_flag(a.err, flags);
}

// One CTA per (query head h, sequence b) (grid Hq x B, 64 threads, four
// head-dim values each): zero rows for empty sequences, nothing for segments
// one split CTA covered, else the fixed-order LSE merge of the pieces
//   M = max m_i,  O = sum_i 2^(m_i - M) O_i / sum_i 2^(m_i - M) l_i.
// Launched as a programmatic dependent of the split kernel, it is resident
// before the split kernel ends, so everything that depends only on seq_lens
// (the cut, hence which CTAs hold the segment's pieces) is done before
// griddepcontrol.wait; after it, one round of loads brings every piece's
// (m, l, O) in.  Batches above kMergeScanMax read the prefix the split kernel
// leaves in the workspace header instead, after the wait.
__global__ void __launch_bounds__(kMergeThreads * kMergeGroups) decode_merge_kernel(DecodeArgs a)
{
    constexpr int kThreadsAll = kMergeThreads * kMergeGroups;
    __shared__ int64_t red_s[kThreadsAll / 32][2];
    __shared__ float g_m[kMergeGroups], g_den[kMergeGroups];
    __shared__ float4 g_num[kMergeGroups][kMergeThreads];
    const int h = blockIdx.x, b = blockIdx.y;
    const int j = h / a.G, hh = h - j * a.G;
    const int tid = threadIdx.x, grp = tid / kMergeThreads, gt = tid % kMergeThreads;
    const int d = 4 * gt;
    __half2* out2 = reinterpret_cast<__half2*>(a.out + ((size_t)b * a.Hq + h) * kD + d);
    int64_t before, total;     // line tiles of sequences < b, of all sequences
    if (a.B <= kMergeScanMax) {
        int64_t lo = 0, all = 0;
        for (int i = tid; i < a.B; i += kThreadsAll) {
            const int64_t n = seg_len(a, i);
            all += n;
            lo += i < b ? n : 0;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            lo += __shfl_xor_sync(0xffffffffu, lo, o);
            all += __shfl_xor_sync(0xffffffffu, all, o);
        }
        if ((tid & 31) == 0) {
            red_s[tid >> 5][0] = lo;
            red_s[tid >> 5][1] = all;
        }
        __syncthreads();
        before = 0;
        total = 0;
        for (int w = 0; w < kThreadsAll / 32; ++w) {
            before += red_s[w][0];
            total += red_s[w][1];
        }
    } else {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        before = a.hdr[2 + b];
        total = a.hdr[2 + a.B];
    }
    // Every CTA waits for the split grid before it exits, so that the end of
    // this grid always implies the end of the split grid.
    const int64_t nb = seg_len(a, b);
    if (nb == 0) {                               // the split kernel never writes these rows
        if (grp == 0) {
            out2[0] = __floats2half2_rn(0.f, 0.f);
            out2[1] = __floats2half2_rn(0.f, 0.f);
        }
        asm volatile("griddepcontrol.wait;" ::: "memory");
        return;
    }
    const int64_t T = (int64_t)a.Hkv * total;
    const int64_t C = effective_ctas(a, T);
    // CTAs c_first..c_last are the ones whose ranges meet the real tiles [r0, r1)
    const int64_t s0 = (int64_t)a.Hkv * before + (int64_t)j * nb;
    const int64_t r0 = s0 + a.piece_cost, r1 = s0 + nb;
    const int64_t c_first = ((r0 + 1) * C + T - 1) / T - 1;
    const int64_t c_last = (r1 * C + T - 1) / T - 1;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (c_first == c_last)
        return;                                  // one split CTA wrote the final rows
    const int64_t k = (int64_t)b * a.Hkv + j;
    const float* base = a.slots + (size_t)(c_first + k) * kSlotFloats;
    float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
    float den = 0.f, M_run = -INFINITY;
    constexpr int kChunk = 8;
    // Chunks of kChunk pieces go to the kMergeGroups thread groups in turn;
    // a segment of one chunk is merged by group 0 alone.
    const bool grouped = c_last - c_first + 1 > kChunk;      // CTA-uniform
    if (!grouped && grp != 0)
        return;
    for (int64_t c0 = c_first + (int64_t)grp * kChunk; c0 <= c_last;
         c0 += (int64_t)(grouped ? kMergeGroups : 1) * kChunk) {
        const int np = (int)min((int64_t)kChunk, c_last - c0 + 1);
        const float* sl0 = base + (size_t)(c0 - c_first) * kSlotFloats;
        float m[kChunk], l[kChunk];
        float4 o[kChunk];
#pragma unroll
        for (int i = 0; i < kChunk; ++i) {
            m[i] = -INFINITY;
            l[i] = 0.f;
            o[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (i < np) {
                const float* sl = sl0 + (size_t)i * kSlotFloats;
                m[i] = sl[hh];
                l[i] = sl[kGMax + hh];
                o[i] = *reinterpret_cast<const float4*>(sl + 2 * kGMax + hh * kD + d);
            }
        }
        float M = M_run;
#pragma unroll
        for (int i = 0; i < kChunk; ++i)
            M = fmaxf(M, m[i]);
        if (M == -INFINITY)
            continue;                            // nothing attended so far
        const float carry = (M_run == -INFINITY) ? 0.f : ex2(M_run - M);
        num.x *= carry;
        num.y *= carry;
        num.z *= carry;
        num.w *= carry;
        den *= carry;
        M_run = M;
#pragma unroll
        for (int i = 0; i < kChunk; ++i) {
            const float e = (m[i] == -INFINITY) ? 0.f : ex2(m[i] - M);
            den += e * l[i];
            num.x += e * o[i].x;
            num.y += e * o[i].y;
            num.z += e * o[i].z;
            num.w += e * o[i].w;
        }
    }
    if (grouped) {
        // the groups' states, combined in group order
        if (gt == 0) {
            g_m[grp] = M_run;
            g_den[grp] = den;
        }
        g_num[grp][gt] = num;
        __syncthreads();
        if (grp != 0)
            return;
        float M = -INFINITY;
        for (int g = 0; g < kMergeGroups; ++g)
            M = fmaxf(M, g_m[g]);
        num = make_float4(0.f, 0.f, 0.f, 0.f);
        den = 0.f;
        if (M != -INFINITY) {
            for (int g = 0; g < kMergeGroups; ++g) {
                const float e = g_m[g] == -INFINITY ? 0.f : ex2(g_m[g] - M);
                const float4 o = g_num[g][gt];
                den += e * g_den[g];
                num.x += e * o.x;
                num.y += e * o.y;
                num.z += e * o.z;
                num.w += e * o.w;
            }
        }
    }
    const float sc = den > 0.f ? a.v_scale / den : 0.f;
    out2[0] = __floats2half2_rn(num.x * sc, num.y * sc);
    out2[1] = __floats2half2_rn(num.z * sc, num.w * sc);
}

size_t decode_split_smem(bool e4m3, int B)
{
    const size_t tail = (size_t)(B + 1) * sizeof(int64_t) +
                        (size_t)(e4m3 ? kDecodeWarps<true>() : kDecodeWarps<false>()) * sizeof(int64_t);
    return (e4m3 ? SmemPlan<true, kDecodeWarps<true>()>::kTailOff
                 : SmemPlan<false, kDecodeWarps<false>()>::kTailOff) + tail;
}

size_t workspace_bytes(int B, int Hkv, int C)
{
    size_t head = kHeaderBytes + (size_t)(B + 1) * sizeof(int64_t);
    head = (head + 255) & ~(size_t)255;
    return head + ((size_t)C + (size_t)B * Hkv) * kSlotFloats * sizeof(float);
}

// The dynamic shared-memory opt-in is a per-device function attribute; it is
// set once per device and kernel instantiation.
template <bool kE4M3>
static cudaError_t set_smem_attr()
{
    static std::atomic<int> done[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < kMaxDevices && done[dev].load(std::memory_order_acquire))
        return cudaSuccess;
    e = cudaFuncSetAttribute(decode_split_kernel<kE4M3>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)decode_split_smem(kE4M3, kMaxSplitBatch));
    if (e == cudaSuccess && dev < kMaxDevices)
        done[dev].store(1, std::memory_order_release);
    return e;
}

int split_ctas_per_sm(bool e4m3)
{
    int n = 0;
    const size_t smem = decode_split_smem(e4m3, 64);
    cudaError_t e = e4m3 ? set_smem_attr<true>() : set_smem_attr<false>();
    if (e != cudaSuccess)
        return 1;
    if (e4m3)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_split_kernel<true>,
                                                          32 * kDecodeWarps<true>(), smem);
    else
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_split_kernel<false>,
                                                          32 * kDecodeWarps<false>(), smem);
    return (e == cudaSuccess && n > 0) ? n : 1;
}

cudaError_t launch_decode(const DecodeArgs& a, bool e4m3, cudaStream_t s, void* ev0, void* ev1)
{
    cudaError_t e = e4m3 ? set_smem_attr<true>() : set_smem_attr<false>();
    if (e != cudaSuccess)
        return e;
    const int grid = a.C > 0 ? a.C : a.B * a.Hkv;
    const size_t smem = a.C > 0 ? decode_split_smem(e4m3, a.B)
                                : (e4m3 ? SmemPlan<true, kDecodeWarps<true>()>::kTailOff
                                        : SmemPlan<false, kDecodeWarps<false>()>::kTailOff);
    if (ev0 && ev1 && (e = cudaEventRecord((cudaEvent_t)ev0, s)) != cudaSuccess)
        return e;
    if (e4m3)
        decode_split_kernel<true><<<grid, 32 * kDecodeWarps<true>(), smem, s>>>(a);
    else
        decode_split_kernel<false><<<grid, 32 * kDecodeWarps<false>(), smem, s>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess)
        return e;
    if (ev0 && ev1 && (e = cudaEventRecord((cudaEvent_t)ev1, s)) != cudaSuccess)
        return e;
    if (a.C > 0) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(a.Hq, a.B);
        cfg.blockDim = dim3(kMergeThreads * kMergeGroups);
        cfg.dynamicSmemBytes = 0;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if ((e = cudaLaunchKernelEx(&cfg, decode_merge_kernel, a)) != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

}  // namespace pgqa
