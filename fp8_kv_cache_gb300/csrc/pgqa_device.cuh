// pgqa_device.cuh -- device building blocks of the paged GQA kernels (sm_103a).
//
// Data path of one warp, per tile of 16 tokens of one KV head:
//   block table -> row addresses (lanes 0..7 resolve one token each of a
//   half-tile of 8; the offsets are shared by shuffles)
//   -> 16-byte cp.async.cg copies (global -> shared, bypassing L1) into the
//      warp's private ring of half-tile stages (WarpRing below), kNS - 2
//      half-tiles in flight while the current tile is computed; chunks are
//      XOR-swizzled in the stage so the fragment reads are conflict-free
//   -> 16-byte shared-memory loads of the K and V rows into registers
//   -> in-register E4M3 -> f16x2 conversion (hardware cvt) or FP16 as is
//   -> S^T = K Q^T on the tensor cores (mma.sync m16n8k16, f16 in, f32
//      accumulate; rows = the 16 tokens, columns = the group's query heads,
//      padded to 8; Q's fragments are staged once per piece in shared memory)
//   -> online softmax in f32 (log2 domain, shuffles across the 8 lane groups)
//   -> O^T += V^T P^T on the tensor cores (rows = head-dim slots, columns = the
//      8 padded heads, k = 16 tokens) plus one extra MMA against a ones matrix
//      that yields the softmax denominator from the same FP16 probabilities.
// The fragments are arranged so that no data moves between lanes on the way:
//   * the head-dim reduction order is free, so each lane reads contiguous
//     16-byte chunks of a row and Q's fragments are permuted to match;
//   * two movmatrix transposes turn the probabilities of S^T's C fragment
//     into the B fragment P^T the second MMA needs;
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
constexpr int kWarps = 4;      // warps per CTA of the prefill kernels
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

// Block-table index and slot of logical token t.
__device__ __forceinline__ void page_and_slot(const KVGeom& g, int t, int& pi, int& slot)
{
    if (g.page_shift >= 0) {
        pi = t >> g.page_shift;
        slot = t & ((1 << g.page_shift) - 1);
    } else {
        pi = t / g.page_size;
        slot = t - pi * g.page_size;
    }
}

// Physical page named by entry pi of the block-table row bt_row, or -1 when it
// is outside [0, num_pages) (then PAGED_GQA_FLAG_BAD_PAGE is added to flags).
__device__ __forceinline__ int table_page(const KVGeom& g, const int32_t* bt_row, int pi,
                                          int& flags)
{
    const int page = __ldg(bt_row + pi);
    if (page < 0 || page >= g.num_pages) {
        flags |= PAGED_GQA_FLAG_BAD_PAGE;
        return -1;
    }
    return page;
}

// Byte offset of the row at (page, slot, KV head j).
__device__ __forceinline__ int64_t row_offset(const KVGeom& g, int page, int slot, int j)
{
    return (int64_t)page * g.page_b + (int64_t)slot * g.token_b + (int64_t)j * g.head_b;
}

// Byte offset of the row of logical token t (KV head j) of the sequence whose
// block-table row is bt_row, or -1 when its page id is invalid.
__device__ __forceinline__ int64_t token_row_offset(const KVGeom& g, const int32_t* bt_row,
                                                    int t, int j, int& flags)
{
    int pi, slot;
    page_and_slot(g, t, pi, slot);
    const int page = table_page(g, bt_row, pi, flags);
    return page < 0 ? -1 : row_offset(g, page, slot, j);
}

// Block entry e of a sparse-prefill row: entries 0..n_sel-1 are the selected
// four-token blocks, entry n_sel is the row's own causal block.  Sets first
// (the block's first logical token) and page (its physical page, or -1 when
// the entry is not attended: padding, a block not strictly before the row's
// own block (PAGED_GQA_FLAG_BAD_SEL), or an invalid page id).  A block never
// straddles pages because page_size is a multiple of 4.
__device__ __forceinline__ void prefill_entry(const KVGeom& g, const int32_t* bt,
                                              const int32_t* sel_row, int n_sel, int own, int e,
                                              int& first, int& page, int& flags)
{
    page = -1;
    first = 0;
    if (e < n_sel) {
        const int b = __ldg(sel_row + e);
        if (b < 0)
            return;                           // padding
        if (b >= own) {
            flags |= PAGED_GQA_FLAG_BAD_SEL;  // not strictly before the tail block
            return;
        }
        first = 4 * b;
    } else if (e == n_sel) {
        first = 4 * own;
    } else {
        return;
    }
    int pi, slot;
    page_and_slot(g, first, pi, slot);
    page = table_page(g, bt, pi, flags);
}

// Whether lane u (0..3) of entry e is attended, given its page: every token
// of a selected block, and the tail block's tokens up to the row's position p.
__device__ __forceinline__ bool prefill_lane_live(int page, int e, int n_sel, int first, int u,
                                                  int p)
{
    return page >= 0 && (e < n_sel || first + u <= p);
}

// ------------------------------------------------------------------ async ring

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

// One stage of a warp's shared-memory ring holds one half-tile: the K rows of
// its 8 tokens, then their V rows, unpadded.  16-byte chunks are placed with
// an XOR swizzle so that the fragment reads of the tile step are free of bank
// conflicts: chunk c of K row t sits at chunk c ^ 4(t & 1) (a quarter-warp
// reads chunks q + 4i of rows g, g+1), chunk c of V row t at c ^ 2((t >> 1) & 3)
// (a quarter-warp reads chunk g of rows 2q + u for four q).
template <bool kE4M3>
struct Stage {
    static constexpr int kRowBytes = kE4M3 ? 256 : 512;
    static constexpr int kKBytes = kHalf * kRowBytes;
    static constexpr int kBytes = 2 * kKBytes;
    __device__ static uint32_t k_off(int t, int c) { return t * kRowBytes + ((16 * c) ^ (64 * (t & 1))); }
    __device__ static uint32_t v_off(int t, int c)
    {
        return kKBytes + t * kRowBytes + ((16 * c) ^ (32 * ((t >> 1) & 3)));
    }
};

// Ring depth in half-tiles per warp.  A 16-token tile consumes two stages, so
// kNS - 2 half-tiles stay in flight while a tile is computed: E4M3 keeps
// 2 x 4 KB per warp (12 warps per SM: 96 KB in flight), FP16 1 x 8 KB (8 warps
// per SM: 64 KB in flight), and the CTAs' shared memory fits in 228 KB.
template <bool kE4M3>
__host__ __device__ constexpr int kStages()
{
    return kE4M3 ? 4 : 3;
}

// Resident CTAs per SM the attention kernels are compiled for (registers:
// 65536 / (128 threads x CTAs)).
template <bool kE4M3>
__host__ __device__ constexpr int kMinCtas()
{
    return kE4M3 ? 3 : 2;
}

// A warp's private ring of kNS stages filled by 16-byte asynchronous copies
// (global -> shared, bypassing L1).  Each fill is one commit group per lane;
// a stage is ready once every lane's group for it has completed and the warp
// has synchronised.  The same warp produces and consumes, so no CTA-wide
// synchronisation is involved, and completion needs no waiting loop.
template <bool kE4M3, int kNS>
struct WarpRing {
    uint32_t ring;        // shared address of stage 0
    uint32_t* masks;      // kNS words: bit t = token t of the stage is attended

    __device__ void init(unsigned char* ring_ptr, uint32_t* mask_ptr)
    {
        ring = smem_u32(ring_ptr);
        masks = mask_ptr;
    }

    __device__ uint32_t addr(int s) const
    {
        return ring + s * Stage<kE4M3>::kBytes;
    }

    // Starts filling stage s and commits one group.  Lane t < 8 passes the
    // byte offset of token t's rows (K and V share it), or < 0 when the token
    // is not attended.  Each copy instruction moves whole 512-byte pieces of
    // rows: FP16 row chunks go to lanes 0..31, E4M3 rows are 16 chunks, so
    // lanes 0..15 take one row and lanes 16..31 the next.
    __device__ void fill(int s, int64_t off, const unsigned char* kb, const unsigned char* vb,
                         int lane)
    {
        using St = Stage<kE4M3>;
        const uint32_t mask = __ballot_sync(0xffffffffu, lane < kHalf && off >= 0) & 0xFFu;
        if (lane == 0)
            masks[s] = mask;
        const uint32_t base = addr(s);
        if (kE4M3) {
            const int c = lane & 15;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int t = 2 * k + (lane >> 4);
                const int64_t o = __shfl_sync(0xffffffffu, off, t);
                if ((mask >> t) & 1u) {
                    cp_async16(base + St::k_off(t, c), kb + o + 16 * c);
                    cp_async16(base + St::v_off(t, c), vb + o + 16 * c);
                }
            }
        } else {
#pragma unroll
            for (int t = 0; t < kHalf; ++t) {
                const int64_t o = __shfl_sync(0xffffffffu, off, t);
                if ((mask >> t) & 1u) {
                    cp_async16(base + St::k_off(t, lane), kb + o + 16 * lane);
                    cp_async16(base + St::v_off(t, lane), vb + o + 16 * lane);
                }
            }
        }
        cp_async_commit();
    }

    // Commits an empty group (one group per ring slot keeps the counts fixed).
    __device__ void skip() const
    {
        cp_async_commit();
    }

    // With kNS fills committed ahead of the current tile, the tile's two
    // stages are complete once at most kNS - 2 groups remain pending.
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
};

// ------------------------------------------------------------------ warp core

// Register-resident attention state of one warp for one (sequence or row,
// KV head): O^T accumulators, the softmax denominators and the running maxima
// of heads 2q and 2q+1 (q = lane & 3).  The Q fragments live in shared
// memory (qs, [k-step][lane] as uint2), shared by the CTA's warps.
//
// Per 16-token tile (two ring stages):
//   S^T = K Q^T   m16n8k16, rows = the 16 tokens, columns = 8 (padded) heads,
//                 K straight from the stage (E4M3 -> f16 in registers);
//   softmax       per head over the tile's 16 tokens (3 shuffles per head);
//   P^T -> P      two movmatrix transposes turn the probabilities of the C
//                 fragment into the B fragment of the next product;
//   O^T += V^T P^T and l += 1^T P^T   m16n8k16 over the 16 tokens.
template <bool kE4M3, bool kQRegs = false>
struct WarpCore {
    static constexpr int kKCh = kE4M3 ? 4 : 8;   // 16-byte chunks of a K row per lane
    static constexpr int kVCh = kE4M3 ? 2 : 4;   // 16-byte chunks of a V row per lane

    float acc[17][4];     // [0..15]: O^T fragments, [16]: denominators
    float m0, m1;         // running max of heads 2q, 2q+1, log2 domain
    uint2 qf[kQRegs ? 16 : 1];   // the lane's Q fragments, when held in registers

    // With kQRegs, copies the lane's Q fragments out of qs (after staging).
    __device__ void load_q(const uint2* qs, int lane)
    {
        if constexpr (kQRegs) {
#pragma unroll
            for (int s = 0; s < 16; ++s)
                qf[s] = qs[s * 32 + lane];
        }
    }

    // Head-dim index of element n (0..63) of the K-row chunks lane q holds
    // (logical chunk c = q + 4i is the 16 bytes at byte 16c of the row).
    __device__ static int k_dim(int q, int n)
    {
        return kE4M3 ? 16 * (q + 4 * (n >> 4)) + (n & 15) : 8 * (q + 4 * (n >> 3)) + (n & 7);
    }
    // Head-dim index of output slot n (0..31) of lane group g (logical V
    // chunk g + 8i).
    __device__ static int v_dim(int g, int n)
    {
        return kE4M3 ? 16 * g + 128 * (n >> 4) + (n & 15) : 8 * g + 64 * (n >> 3) + (n & 7);
    }

    // The CTA's nw warps write the Q fragments of heads g < G (binary16
    // [G][256] rows at qg) into qs[16][32] (uint2), the k-steps dealt to the
    // warps in turn; the caller synchronises the CTA before use.
    __device__ static void stage_q(uint2* qs, const __half* qg, int G, int lane, int w, int nw)
    {
        const int g = lane >> 2, q = lane & 3;
        const uint32_t* row = reinterpret_cast<const uint32_t*>(qg + (size_t)g * kD);
        for (int s = w; s < 16; s += nw) {
            uint2 f = make_uint2(0u, 0u);
            if (g < G) {
                f.x = __ldg(row + (k_dim(q, 4 * s) >> 1));
                f.y = __ldg(row + (k_dim(q, 4 * s + 2) >> 1));
            }
            qs[s * 32 + lane] = f;
        }
    }

    __device__ void reset()
    {
#pragma unroll
        for (int i = 0; i < 17; ++i)
#pragma unroll
            for (int c = 0; c < 4; ++c)
                acc[i][c] = 0.f;
        m0 = m1 = -INFINITY;
    }

    // One 16-token tile whose first 8 tokens are in stage st0 and last 8 in
    // st1; bit t of mask says whether token t is attended.
    __device__ void tile(uint32_t st0, uint32_t st1, uint32_t mask, const uint2* qs, int G,
                         float scale_log2, int lane)
    {
        using St = Stage<kE4M3>;
        const int g = lane >> 2, q = lane & 3;
        const uint4 zero = make_uint4(0, 0, 0, 0);
        // ---- S^T = K Q^T over the 16 k-steps, four accumulation chains
        float sc[4][4];
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                sc[c][e] = 0.f;
        const bool kv0 = (mask >> g) & 1u, kv1 = (mask >> (g + 8)) & 1u;
#pragma unroll
        for (int i = 0; i < kKCh; ++i) {
            const uint4 k0 = kv0 ? lds128(st0 + St::k_off(g, q + 4 * i)) : zero;   // token g
            const uint4 k1 = kv1 ? lds128(st1 + St::k_off(g, q + 4 * i)) : zero;   // token g + 8
#pragma unroll
            for (int w = 0; w < (kE4M3 ? 4 : 2); ++w) {
                const int s = kE4M3 ? 4 * i + w : 2 * i + w;
                uint2 b;
                if constexpr (kQRegs)
                    b = qf[s];
                else
                    b = qs[s * 32 + lane];
                uint32_t a0, a1, a2, a3;
                if (kE4M3) {
                    e4m3x4_to_f16x2x2(word(k0, w), a0, a2);
                    e4m3x4_to_f16x2x2(word(k1, w), a1, a3);
                } else {
                    a0 = word(k0, 2 * w);
                    a2 = word(k0, 2 * w + 1);
                    a1 = word(k1, 2 * w);
                    a3 = word(k1, 2 * w + 1);
                }
                mma16816(sc[s & 3], a0, a1, a2, a3, b.x, b.y);
            }
        }
        // ---- online softmax: lane holds tokens g, g+8 of heads 2q, 2q+1
        const bool h0 = 2 * q < G, h1 = 2 * q + 1 < G;
        float x[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
            x[e] = (sc[0][e] + sc[1][e]) + (sc[2][e] + sc[3][e]);
        x[0] = (kv0 && h0) ? x[0] * scale_log2 : -INFINITY;   // token g,     head 2q
        x[1] = (kv0 && h1) ? x[1] * scale_log2 : -INFINITY;   // token g,     head 2q+1
        x[2] = (kv1 && h0) ? x[2] * scale_log2 : -INFINITY;   // token g + 8, head 2q
        x[3] = (kv1 && h1) ? x[3] * scale_log2 : -INFINITY;   // token g + 8, head 2q+1
        float mx0 = fmaxf(x[0], x[2]), mx1 = fmaxf(x[1], x[3]);
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
        }
        const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
        const float al0 = n0 == -INFINITY ? 1.f : ex2(m0 - n0);
        const float al1 = n1 == -INFINITY ? 1.f : ex2(m1 - n1);
        float p[4];
        p[0] = n0 == -INFINITY ? 0.f : ex2(x[0] - n0);
        p[2] = n0 == -INFINITY ? 0.f : ex2(x[2] - n0);
        p[1] = n1 == -INFINITY ? 0.f : ex2(x[1] - n1);
        p[3] = n1 == -INFINITY ? 0.f : ex2(x[3] - n1);
        m0 = n0;
        m1 = n1;
        if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
            for (int i = 0; i < 17; ++i) {
                acc[i][0] *= al0;
                acc[i][2] *= al0;
                acc[i][1] *= al1;
                acc[i][3] *= al1;
            }
        }
        // ---- P fragments: transpose the two 8x8 blocks [token][head] -> [head][token]
        uint32_t pb0, pb1;
        asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(pb0) : "r"(pack_half2(p[0], p[1])));
        asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(pb1) : "r"(pack_half2(p[2], p[3])));
        // ---- O^T += V^T P^T: V rows 2q, 2q+1 (stage 0) and 2q+8, 2q+9 (stage 1)
        const bool v0 = (mask >> (2 * q)) & 1u, v1 = (mask >> (2 * q + 1)) & 1u;
        const bool v2 = (mask >> (2 * q + 8)) & 1u, v3 = (mask >> (2 * q + 9)) & 1u;
#pragma unroll
        for (int i = 0; i < kVCh; ++i) {
            const int c = g + 8 * i;
            const uint4 r0 = v0 ? lds128(st0 + St::v_off(2 * q, c)) : zero;
            const uint4 r1 = v1 ? lds128(st0 + St::v_off(2 * q + 1, c)) : zero;
            const uint4 r2 = v2 ? lds128(st1 + St::v_off(2 * q, c)) : zero;
            const uint4 r3 = v3 ? lds128(st1 + St::v_off(2 * q + 1, c)) : zero;
#pragma unroll
            for (int j = 0; j < (kE4M3 ? 8 : 4); ++j) {
                const int mt = (kE4M3 ? 8 : 4) * i + j;
                uint32_t a0, a1, a2, a3;
                if (kE4M3) {
                    const int w = j >> 1;
                    const uint32_t sel = (j & 1) ? 0x7362u : 0x5140u;
                    e4m3x4_to_f16x2x2(__byte_perm(word(r0, w), word(r1, w), sel), a0, a1);
                    e4m3x4_to_f16x2x2(__byte_perm(word(r2, w), word(r3, w), sel), a2, a3);
                } else {
                    a0 = __byte_perm(word(r0, j), word(r1, j), 0x5410u);
                    a1 = __byte_perm(word(r0, j), word(r1, j), 0x7632u);
                    a2 = __byte_perm(word(r2, j), word(r3, j), 0x5410u);
                    a3 = __byte_perm(word(r2, j), word(r3, j), 0x7632u);
                }
                mma16816(acc[mt], a0, a1, a2, a3, pb0, pb1);
            }
        }
        const uint32_t one2 = 0x3C003C00u;   // half2(1, 1)
        mma16816(acc[16], one2, one2, one2, one2, pb0, pb1);
    }
};

// Runs a warp over 16-token tiles k = first, first + stride, ... < end.  Tile
// k is half-tiles 2k and 2k+1; offset(h) returns, on lanes t < 8, the byte
// offset of token t of half-tile h (or -1), and -1 on the other lanes.  The
// ring keeps kNS half-tiles committed ahead of the tile being computed.
template <bool kE4M3, int kNS, class Offset, bool kQRegs = false>
__device__ __forceinline__ void run_tiles(WarpCore<kE4M3, kQRegs>& wc, WarpRing<kE4M3, kNS>& rg,
                                          const uint2* qs, const unsigned char* kb,
                                          const unsigned char* vb, int first, int end, int stride,
                                          int G, float scale_log2, int lane, Offset offset)
{
    const int n = end > first ? (end - first + stride - 1) / stride : 0;
    if (n == 0)
        return;
    const int H = 2 * n;                        // half-tiles of this warp, in order
    auto half = [&](int j) { return 2 * (first + (j >> 1) * stride) + (j & 1); };
    for (int j = 0; j < kNS; ++j) {
        if (j < H)
            rg.fill(j, offset(half(j)), kb, vb, lane);
        else
            rg.skip();
    }
    for (int k = 0; k < n; ++k) {
        const int s0 = (2 * k) % kNS, s1 = (2 * k + 1) % kNS;
        rg.wait();
        const uint32_t mask = rg.masks[s0] | (rg.masks[s1] << 8);
        wc.tile(rg.addr(s0), rg.addr(s1), mask, qs, G, scale_log2, lane);
        __syncwarp();
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int j = 2 * k + kNS + u;
            if (j < H)
                rg.fill(j % kNS, offset(half(j)), kb, vb, lane);
            else
                rg.skip();
        }
    }
    rg.drain();
}

// Shared-memory carve-up of a CTA of the attention kernels:
//   [Q fragments (4 KB, shared)][rings of 4 warps (the merge buffer aliases them)]
//   [stage masks]
//   [kernel-specific tail]
// The sparse-prefill kernel keeps its address table in the tail: a chunk's
// resolved block entries (int2 {first token, page} each), so that its ring
// fills issue their copies without the two dependent global loads
// (selection index, then block-table entry) in front of them.
template <bool kE4M3, int NW = kWarps>
struct SmemPlan {
    static constexpr int kNS = kStages<kE4M3>();
    static constexpr size_t kQBytes = (size_t)16 * 32 * sizeof(uint2);
    static constexpr size_t kRingBytes = (size_t)NW * kNS * Stage<kE4M3>::kBytes;
    static constexpr size_t kMaskOff = kQBytes + kRingBytes;
    static constexpr size_t kTailOff = (kMaskOff + (size_t)NW * kNS * 4 + 15) & ~(size_t)15;
    static constexpr int kPrefillEntries = kE4M3 ? 520 : 1024; // block entries per prefill chunk
    static constexpr size_t kPrefillSmem = kTailOff + (size_t)kPrefillEntries * sizeof(int2);
};

// ------------------------------------------------------------------ CTA merge

// Combines the NW warps' states of one (row, KV head) through shared memory.
// Writes either the final binary16 output rows (out_rows != nullptr, rows of
// the G heads at stride kD) or a partial slot (m, l, O).
template <int NW = kWarps>
struct MergeSmem {
    float m[NW][kGMax];
    float l[NW][kGMax];
    float o[NW][kGMax][kD];
};

// The pieces of a CTA's shared memory for one attention kernel instance.
template <bool kE4M3, int NW = kWarps>
struct CtaSmem {
    uint2* qs;              // the CTA's Q fragments
    MergeSmem<NW>* merge;   // aliases the rings; used only after every ring is drained
    unsigned char* ring;    // this warp's ring
    uint32_t* masks;        // this warp's stage masks
    unsigned char* tail;    // kernel-specific tail

    __device__ static CtaSmem carve(unsigned char* base, int w)
    {
        using Pl = SmemPlan<kE4M3, NW>;
        static_assert(Pl::kRingBytes >= sizeof(MergeSmem<NW>), "merge buffer must fit in the rings");
        CtaSmem c;
        c.qs = reinterpret_cast<uint2*>(base);
        c.merge = reinterpret_cast<MergeSmem<NW>*>(base + Pl::kQBytes);
        c.ring = base + Pl::kQBytes + (size_t)w * Pl::kNS * Stage<kE4M3>::kBytes;
        c.masks = reinterpret_cast<uint32_t*>(base + Pl::kMaskOff) + w * Pl::kNS;
        c.tail = base + Pl::kTailOff;
        return c;
    }
};

template <bool kE4M3, bool kQRegs = false, int NW = kWarps>
__device__ void cta_merge(MergeSmem<NW>& sm, const WarpCore<kE4M3, kQRegs>& wc, int G,
                          float v_scale, __half* out_rows, float* slot)
{
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int g = lane >> 2, q = lane & 3;
    __syncthreads();   // previous use of sm finished
    if (g == 0) {
        sm.m[w][2 * q] = wc.m0;
        sm.m[w][2 * q + 1] = wc.m1;
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
        for (int i = 0; i < NW; ++i)
            M = fmaxf(M, sm.m[i][h]);
        float sc[NW];
        float den = 0.f;
#pragma unroll
        for (int i = 0; i < NW; ++i) {
            sc[i] = (M == -INFINITY) ? 0.f : ex2(sm.m[i][h] - M);
            den += sc[i] * sm.l[i][h];
        }
        for (int d = tid; d < kD; d += NW * 32) {
            float num = 0.f;
#pragma unroll
            for (int i = 0; i < NW; ++i)
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
