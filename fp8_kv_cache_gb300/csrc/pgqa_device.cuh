// pgqa_device.cuh -- device building blocks of the paged GQA kernels (sm_103a).
//
// Data path of one warp, per tile of 16 tokens of one KV head:
//   block table -> row addresses (lanes 0..15, one token each, shared by shuffles)
//   -> 16-byte read-only global loads straight into registers
//   -> in-register E4M3 -> f16x2 conversion (hardware cvt) or FP16 as is
//   -> S = Q K^T on the tensor cores (mma.sync m16n8k16, f16 in, f32 accumulate;
//      rows = the group's query heads, padded to 16; columns = 8 tokens)
//   -> online softmax in f32 (log2 domain, 4-lane shuffles per head)
//   -> O^T += V^T P^T on the tensor cores (rows = head-dim slots, columns = the
//      8 padded heads, k = 16 tokens) plus one extra MMA against a ones matrix
//      that yields the softmax denominator from the same FP16 probabilities.
// The fragments are arranged so that no shared memory is touched on the way:
//   * the head-dim reduction order is free, so each lane loads contiguous
//     16-byte chunks and Q's fragments are permuted to match;
//   * the C fragment of S (rows heads, columns tokens 2q, 2q+1) is exactly the
//     B fragment P^T needs for the second MMA;
//   * V's token pairs are interleaved with one byte permute per register.
//
// The operation is the paged GQA attention of "[Kernel][SM70] Scale NVFP4 E4M3
// decode batches" (1Cat-vLLM #282), Purpose (decode), and of "[Kernel][SM70]
// Accelerate Qwen3.8 QSA paged prefill" (1Cat-vLLM #378), Changes (selected
// four-token blocks plus the causal tail).
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "../../include/paged_gqa.h"

namespace pgqa {

constexpr int kD = 256;        // head dim (the only one built)
constexpr int kGMax = 8;       // query heads per KV head, padded
constexpr int kTile = 16;      // tokens per tile (unit of the split partition)
constexpr int kHalf = 8;       // tokens per half-tile (unit of the warp pipeline)
constexpr int kWarps = 4;      // warps per CTA
constexpr int kThreads = kWarps * 32;

// One partial result of a split: m[8], l[8], O[8][256] (unnormalised), f32.
constexpr int kSlotFloats = 2 * kGMax + kGMax * kD;

// ------------------------------------------------------------------ PTX helpers

__device__ __forceinline__ uint4 ldg_stream(const unsigned char* p)
{
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

__device__ __forceinline__ uint32_t word(const uint4& c, int k)
{
    return k == 0 ? c.x : k == 1 ? c.y : k == 2 ? c.z : c.w;
}

// D(16x8, f32) += A(16x16, f16, row) * B(16x8, f16, col).
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Four E4M3 codes (bytes 0..3 of w) -> two f16x2: lo = (byte0, byte1),
// hi = (byte2, byte3), each byte in the matching half.  E4M3 values are all
// exactly representable in binary16, so this conversion is exact.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi)
{
    asm("{\n\t.reg .b16 a, b;\n\t"
        "mov.b32 {a, b}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, a;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi)
{
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void raise_flag(int* err, int bits)
{
    if (err != nullptr && bits != 0)
        atomicOr(err, bits);
}

// ------------------------------------------------------------------ addressing

// Byte geometry of one K/V pool pair (K and V share strides).
struct KVGeom {
    const unsigned char* k;
    const unsigned char* v;
    int64_t page_b;     // page stride, bytes
    int64_t token_b;    // token stride, bytes
    int64_t head_b;     // KV-head stride, bytes
    int page_size;
    int page_shift;     // log2(page_size) when it is a power of two, else -1
    int num_pages;
};

// Byte offset of the row of logical token t (KV head j) of the sequence whose
// block-table row is bt_row, or -1 when its page id is outside [0, num_pages)
// (then PAGED_GQA_FLAG_BAD_PAGE is added to *flags).
__device__ __forceinline__ int64_t token_row_offset(const KVGeom& g, const int32_t* bt_row,
                                                    int t, int j, int& flags)
{
    int pi, slot;
    if (g.page_shift >= 0) {
        pi = t >> g.page_shift;
        slot = t & ((1 << g.page_shift) - 1);
    } else {
        pi = t / g.page_size;
        slot = t - pi * g.page_size;
    }
    const int page = __ldg(bt_row + pi);
    if (page < 0 || page >= g.num_pages) {
        flags |= PAGED_GQA_FLAG_BAD_PAGE;
        return -1;
    }
    return (int64_t)page * g.page_b + (int64_t)slot * g.token_b + (int64_t)j * g.head_b;
}

// Logical token of lane u (0..3) of block entry `entry` of a sparse-prefill
// row: entries 0..n_sel-1 are the selected four-token blocks, entry n_sel is
// the row's own causal block, cut after position p.  -1 = not attended.
__device__ __forceinline__ int prefill_token(const int32_t* sel_row, int n_sel, int own,
                                             int p, int entry, int u, int& flags)
{
    if (entry < n_sel) {
        const int b = __ldg(sel_row + entry);
        if (b < 0)
            return -1;                        // padding
        if (b >= own) {
            flags |= PAGED_GQA_FLAG_BAD_SEL;  // not strictly before the tail block
            return -1;
        }
        return 4 * b + u;
    }
    if (entry == n_sel) {
        const int t = 4 * own + u;
        return t <= p ? t : -1;
    }
    return -1;
}

// ------------------------------------------------------------------ warp core

// D(16x8, f32) += A(16x8, f16, row) * B(8x8, f16, col).
__device__ __forceinline__ void mma16808(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t b0)
{
    asm("mma.sync.aligned.m16n8k8.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5}, {%6}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(b0));
}

// Raw K/V registers of one half-tile (8 tokens) as lane (g, q) holds them:
// the K row of token g and the V rows of tokens 2q and 2q+1.
template <bool kE4M3>
struct HalfTile {
    static constexpr int kKCh = kE4M3 ? 4 : 8;   // 16-byte chunks of the K row
    static constexpr int kVCh = kE4M3 ? 2 : 4;   // 16-byte chunks of each V row
    uint4 k[kKCh];
    uint4 v[2][kVCh];
    bool valid[2];                               // tokens 2q, 2q+1 attended
};

// Register-resident attention state of one warp for one (sequence or row,
// KV head): O^T accumulators, the softmax denominators and the running max of
// head g (= lane / 4).  The Q fragments live in shared memory (qs), laid out
// [k-step][lane] as uint2 so each lane reads 8 contiguous bytes.
template <bool kE4M3>
struct WarpCore {
    float acc[17][4];     // [0..15]: O^T fragments, [16]: denominators
    float m;              // running max of head g, log2 domain

    // Head-dim index of element n (0..63) of the K-row chunks lane q holds
    // (chunk c = q + 4i is 16 bytes at byte offset 16c of the row).
    __device__ static int k_dim(int q, int n)
    {
        return kE4M3 ? 16 * (q + 4 * (n >> 4)) + (n & 15) : 8 * (q + 4 * (n >> 3)) + (n & 7);
    }
    // Head-dim index of output slot n (0..31) of lane group g (V chunk i is
    // 16 bytes at byte offset 16g + 128i of the row).
    __device__ static int v_dim(int g, int n)
    {
        return kE4M3 ? 16 * g + 128 * (n >> 4) + (n & 15) : 8 * g + 64 * (n >> 3) + (n & 7);
    }

    // Writes this lane's Q fragments (heads g < G of the group, binary16
    // [G][256] rows at qg) into qs[16][32] (uint2), then syncs the warp.
    __device__ static void stage_q(uint2* qs, const __half* qg, int G, int lane)
    {
        const int g = lane >> 2, q = lane & 3;
        const uint32_t* row = reinterpret_cast<const uint32_t*>(qg + (size_t)g * kD);
#pragma unroll
        for (int s = 0; s < 16; ++s) {
            uint2 f = make_uint2(0u, 0u);
            if (g < G) {
                f.x = __ldg(row + (k_dim(q, 4 * s) >> 1));
                f.y = __ldg(row + (k_dim(q, 4 * s + 2) >> 1));
            }
            qs[s * 32 + lane] = f;
        }
        __syncwarp();
    }

    __device__ void reset()
    {
#pragma unroll
        for (int i = 0; i < 17; ++i)
#pragma unroll
            for (int c = 0; c < 4; ++c)
                acc[i][c] = 0.f;
        m = -INFINITY;
    }

    // One half-tile of 8 tokens: S = Q K^T (m16n8k16, rows = heads), online
    // softmax of head g, then O^T += V^T P^T and l += 1^T P^T (m16n8k8).
    __device__ void step(const HalfTile<kE4M3>& t, const uint2* qs, bool head_ok, float scale_log2,
                         int lane)
    {
        const int q = lane & 3;
        // four independent accumulation chains over the 16 k-steps
        float sc[4][4];
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                sc[c][e] = 0.f;
#pragma unroll
        for (int s = 0; s < 16; ++s) {
            const uint2 a = qs[s * 32 + lane];
            uint32_t b0, b1;
            if (kE4M3) {
                e4m3x4_to_f16x2x2(word(t.k[s >> 2], s & 3), b0, b1);
            } else {
                b0 = word(t.k[s >> 1], 2 * (s & 1));
                b1 = word(t.k[s >> 1], 2 * (s & 1) + 1);
            }
            mma16816(sc[s & 3], a.x, 0u, a.y, 0u, b0, b1);
        }
        // scores of head g for tokens 2q, 2q+1
        const float s0 = (sc[0][0] + sc[1][0]) + (sc[2][0] + sc[3][0]);
        const float s1 = (sc[0][1] + sc[1][1]) + (sc[2][1] + sc[3][1]);
        float x0 = (t.valid[0] && head_ok) ? s0 * scale_log2 : -INFINITY;
        float x1 = (t.valid[1] && head_ok) ? s1 * scale_log2 : -INFINITY;
        float mx = fmaxf(x0, x1);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float m_new = fmaxf(m, mx);
        float alpha = 1.f, p0 = 0.f, p1 = 0.f;
        if (m_new != -INFINITY) {
            alpha = ex2(m - m_new);
            p0 = ex2(x0 - m_new);
            p1 = ex2(x1 - m_new);
        }
        m = m_new;
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
            const float a_lo = __shfl_sync(0xffffffffu, alpha, 8 * q);
            const float a_hi = __shfl_sync(0xffffffffu, alpha, 8 * q + 4);
#pragma unroll
            for (int i = 0; i < 17; ++i) {
                acc[i][0] *= a_lo;
                acc[i][2] *= a_lo;
                acc[i][1] *= a_hi;
                acc[i][3] *= a_hi;
            }
        }
        const uint32_t pb = pack_half2(p0, p1);
#pragma unroll
        for (int mt = 0; mt < 16; ++mt) {
            uint32_t a0, a1;
            if (kE4M3) {
                const int i = mt >> 3, w = (mt & 7) >> 1;
                const uint32_t sel = (mt & 1) ? 0x7362u : 0x5140u;
                e4m3x4_to_f16x2x2(__byte_perm(word(t.v[0][i], w), word(t.v[1][i], w), sel), a0, a1);
            } else {
                const int i = mt >> 2, w = mt & 3;
                a0 = __byte_perm(word(t.v[0][i], w), word(t.v[1][i], w), 0x5410u);
                a1 = __byte_perm(word(t.v[0][i], w), word(t.v[1][i], w), 0x7632u);
            }
            mma16808(acc[mt], a0, a1, pb);
        }
        const uint32_t one2 = 0x3C003C00u;   // half2(1, 1)
        mma16808(acc[16], one2, one2, pb);
    }
};

// ------------------------------------------------------------------ async ring

// One stage of a warp's shared-memory ring holds one half-tile: the K rows of
// its 8 tokens, then their V rows.  Row strides are padded so that the
// fragment reads below are free of bank conflicts: a K row is read by lanes
// (g, q) as chunks q + 4i (8 rows x 4 chunks per quarter-warp phase -> the
// stride must be 64 mod 128 bytes); a V row pair 2q, 2q+1 is read at chunk
// g + 8i (stride 16 mod 64 bytes).
template <bool kE4M3>
struct Stage {
    static constexpr int kRowBytes = kE4M3 ? 256 : 512;
    static constexpr int kKStride = kRowBytes + 64;
    static constexpr int kVStride = kRowBytes + 16;
    static constexpr int kKBytes = kHalf * kKStride;
    static constexpr int kBytes = kHalf * (kKStride + kVStride);
};

// Ring depth (stages per warp): kNS - 1 half-tiles stay in flight while one
// is read.  With the CTAs per SM below, an SM keeps 96 KB (E4M3: 12 warps x
// 2 x 4 KB) or 70 KB (FP16: 8 warps x 1 x 8.6 KB) of KV in flight, and the
// shared memory of those CTAs fits in 228 KB.
template <bool kE4M3>
__host__ __device__ constexpr int kStages()
{
    return kE4M3 ? 3 : 2;
}

// Resident CTAs per SM the attention kernels are compiled for (registers:
// 65536 / (128 threads x CTAs)).
template <bool kE4M3>
__host__ __device__ constexpr int kMinCtas()
{
    return kE4M3 ? 3 : 2;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint4 lds128(uint32_t addr)
{
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "r"(addr));
    return r;
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const unsigned char* src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_commit()
{
    asm volatile("cp.async.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// A warp's private ring of kNS stages filled by 16-byte asynchronous copies
// (global -> shared, bypassing L1).  Each fill is one commit group per lane;
// a stage is ready once every lane's group for it has completed and the warp
// has synchronised.  The same warp produces and consumes, so no CTA-wide
// synchronisation is involved, and completion needs no waiting loop.
template <bool kE4M3, int kNS>
struct WarpRing {
    uint32_t ring;        // shared address of stage 0
    uint32_t* masks;      // kNS words: bit t = token t of the stage is valid

    __device__ void init(unsigned char* ring_ptr, uint32_t* mask_ptr)
    {
        ring = smem_u32(ring_ptr);
        masks = mask_ptr;
    }

    // Starts filling stage s and commits one group.  Lane t < 8 passes the
    // byte offset of token t's rows (K and V share it), or < 0 when the token
    // is not attended.  Chunk c of a row is copied by lane c (FP16 rows are
    // 32 chunks) or lane c + 16 * (row parity) (E4M3 rows are 16 chunks), so
    // every copy instruction reads whole 512-byte row pieces.
    __device__ void fill(int s, int64_t off, const unsigned char* kb, const unsigned char* vb,
                         int lane)
    {
        using St = Stage<kE4M3>;
        const uint32_t mask = __ballot_sync(0xffffffffu, lane < kHalf && off >= 0) & 0xFFu;
        if (lane == 0)
            masks[s] = mask;
        const uint32_t base = ring + s * St::kBytes;
        if (kE4M3) {
            // instruction k: token 2(k % 4) + lane / 16, chunk lane % 16, K for k < 4
            const int half = lane >> 4, c = lane & 15;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int t = 2 * k + half;
                const int64_t o = __shfl_sync(0xffffffffu, off, t);
                if ((mask >> t) & 1u) {
                    cp_async16(base + t * St::kKStride + 16 * c, kb + o + 16 * c);
                    cp_async16(base + St::kKBytes + t * St::kVStride + 16 * c, vb + o + 16 * c);
                }
            }
        } else {
            // instruction k: token k, chunk lane
#pragma unroll
            for (int t = 0; t < kHalf; ++t) {
                const int64_t o = __shfl_sync(0xffffffffu, off, t);
                if ((mask >> t) & 1u) {
                    cp_async16(base + t * St::kKStride + 16 * lane, kb + o + 16 * lane);
                    cp_async16(base + St::kKBytes + t * St::kVStride + 16 * lane, vb + o + 16 * lane);
                }
            }
        }
        cp_async_commit();
    }

    // Commits an empty group (keeps one group per ring slot).
    __device__ void skip() const
    {
        cp_async_commit();
    }

    // The oldest of the kNS - 1 committed fills is complete for every lane
    // (at most kNS - 2 groups may still be pending).
    __device__ void wait() const
    {
        static_assert(kNS >= 2, "the ring needs at least two stages");
        cp_async_wait<kNS - 2>();
        __syncwarp();
    }

    __device__ void drain() const
    {
        asm volatile("cp.async.wait_all;" ::: "memory");
        __syncwarp();
    }

    // The fragments lane (g, q) needs from stage s: K row g, V rows 2q, 2q+1
    // (zeros for tokens that are not attended).
    __device__ void read(int s, HalfTile<kE4M3>& t, int g, int q) const
    {
        using St = Stage<kE4M3>;
        const uint32_t mask = masks[s];
        const uint32_t base = ring + s * St::kBytes;
        const bool kv = (mask >> g) & 1u;
#pragma unroll
        for (int i = 0; i < HalfTile<kE4M3>::kKCh; ++i)
            t.k[i] = kv ? lds128(base + g * St::kKStride + 16 * (q + 4 * i)) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int row = 2 * q + u;
            const bool vv = (mask >> row) & 1u;
            t.valid[u] = vv;
#pragma unroll
            for (int i = 0; i < HalfTile<kE4M3>::kVCh; ++i)
                t.v[u][i] = vv ? lds128(base + St::kKBytes + row * St::kVStride + 16 * g + 128 * i)
                               : make_uint4(0, 0, 0, 0);
        }
    }
};

// Runs a warp over half-tiles h = first, first + stride, ... < end through
// its ring: kNS - 1 fills in flight; per half-tile: wait for the oldest fill,
// read its fragments, refill that stage kNS - 1 half-tiles ahead, compute.
// offset(h) returns, on lanes t < 8, the byte offset of token t of half-tile h
// (or -1), and -1 on the other lanes.
template <bool kE4M3, int kNS, class Offset>
__device__ __forceinline__ void run_halves(WarpCore<kE4M3>& wc, WarpRing<kE4M3, kNS>& rg,
                                           const uint2* qs, const unsigned char* kb,
                                           const unsigned char* vb, int first, int end, int stride,
                                           bool head_ok, float scale_log2, int lane, Offset offset)
{
    const int g = lane >> 2, q = lane & 3;
    const int n = end > first ? (end - first + stride - 1) / stride : 0;
    if (n == 0)
        return;
    for (int i = 0; i < kNS - 1; ++i) {
        if (i < n)
            rg.fill(i, offset(first + i * stride), kb, vb, lane);
        else
            rg.skip();
    }
    for (int i = 0; i < n; ++i) {
        const int s = i % kNS;
        HalfTile<kE4M3> t;
        rg.wait();
        rg.read(s, t, g, q);
        __syncwarp();
        const int nf = i + kNS - 1;
        if (nf < n)
            rg.fill(nf % kNS, offset(first + nf * stride), kb, vb, lane);
        else
            rg.skip();
        wc.step(t, qs, head_ok, scale_log2, lane);
    }
    rg.drain();
}

// Shared-memory carve-up of a CTA of the attention kernels:
//   [Q fragments of 4 warps][rings of 4 warps (the merge buffer aliases them)]
//   [stage masks][kernel-specific tail]
template <bool kE4M3>
struct SmemPlan {
    static constexpr int kNS = kStages<kE4M3>();
    static constexpr size_t kQBytes = (size_t)kWarps * 16 * 32 * sizeof(uint2);
    static constexpr size_t kRingBytes = (size_t)kWarps * kNS * Stage<kE4M3>::kBytes;
    static constexpr size_t kRingOrMerge = kRingBytes;   // asserted >= sizeof(MergeSmem) below
    static constexpr size_t kMaskOff = kQBytes + kRingOrMerge;
    static constexpr size_t kTailOff = (kMaskOff + (size_t)kWarps * kNS * 4 + 15) & ~(size_t)15;
};

// ------------------------------------------------------------------ CTA merge

// Combines the kWarps warps' states of one (row, KV head) through shared
// memory.  Writes either the final binary16 output rows (out_rows != nullptr,
// rows of the G heads at stride kD) or a partial slot (m, l, O).
struct MergeSmem {
    float m[kWarps][kGMax];
    float l[kWarps][kGMax];
    float o[kWarps][kGMax][kD];
};

// The pieces of a CTA's shared memory for one attention kernel instance.
template <bool kE4M3>
struct CtaSmem {
    uint2* qs;            // this warp's Q fragments
    MergeSmem* merge;     // aliases the rings; used only after every ring is drained
    unsigned char* ring;  // this warp's ring
    uint32_t* masks;      // this warp's stage masks
    unsigned char* tail;  // kernel-specific tail

    __device__ static CtaSmem carve(unsigned char* base, int w)
    {
        using Pl = SmemPlan<kE4M3>;
        static_assert(Pl::kRingBytes >= sizeof(MergeSmem), "merge buffer must fit in the rings");
        CtaSmem c;
        c.qs = reinterpret_cast<uint2*>(base) + w * 16 * 32;
        c.merge = reinterpret_cast<MergeSmem*>(base + Pl::kQBytes);
        c.ring = base + Pl::kQBytes + (size_t)w * Pl::kNS * Stage<kE4M3>::kBytes;
        c.masks = reinterpret_cast<uint32_t*>(base + Pl::kMaskOff) + w * Pl::kNS;
        c.tail = base + Pl::kTailOff;
        return c;
    }
};

template <bool kE4M3>
__device__ void cta_merge(MergeSmem& sm, const WarpCore<kE4M3>& wc, int G, float v_scale,
                          __half* out_rows, float* slot)
{
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int g = lane >> 2, q = lane & 3;
    __syncthreads();   // previous use of sm finished
    if (q == 0)
        sm.m[w][g] = wc.m;
    if (g == 0) {
        sm.l[w][2 * q] = wc.acc[16][0];
        sm.l[w][2 * q + 1] = wc.acc[16][1];
    }
#pragma unroll
    for (int mt = 0; mt < 16; ++mt) {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int d = WarpCore<kE4M3>::v_dim(g, 2 * mt + r);
            sm.o[w][2 * q][d] = wc.acc[mt][2 * r];
            sm.o[w][2 * q + 1][d] = wc.acc[mt][2 * r + 1];
        }
    }
    __syncthreads();
    for (int h = 0; h < G; ++h) {
        float M = -INFINITY;
#pragma unroll
        for (int i = 0; i < kWarps; ++i)
            M = fmaxf(M, sm.m[i][h]);
        float sc[kWarps];
        float den = 0.f;
#pragma unroll
        for (int i = 0; i < kWarps; ++i) {
            sc[i] = (M == -INFINITY) ? 0.f : ex2(sm.m[i][h] - M);
            den += sc[i] * sm.l[i][h];
        }
        for (int d = tid; d < kD; d += kThreads) {
            float num = 0.f;
#pragma unroll
            for (int i = 0; i < kWarps; ++i)
                num += sc[i] * sm.o[i][h][d];
            if (out_rows != nullptr) {
                const float v = den > 0.f ? num / den * v_scale : 0.f;
                out_rows[(size_t)h * kD + d] = __float2half_rn(v);
            } else {
                slot[2 * kGMax + h * kD + d] = num;
            }
        }
        if (out_rows == nullptr && tid == 0) {
            slot[h] = M;
            slot[kGMax + h] = den;
        }
    }
    __syncthreads();   // sm is free again (its Q-staging area is reused next)
}

}  // namespace pgqa
