// pgqa_internal.h -- argument blocks and launch wrappers shared between the
// host entry points (api.cu) and the kernel translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "pgqa_device.cuh"

namespace pgqa {

constexpr int kMaxSplitBatch = 4096;   // split route keeps a (B+1) prefix in shared memory
constexpr int kMergeThreads = 64;     // threads of a merge group: 4 head-dim values each
constexpr int kMergeGroups = 4;       // groups of a merge CTA, taking chunks of pieces in turn
constexpr int kMergeScanMax = 512;    // merge recomputes the cut from seq_lens up to this batch
constexpr int kHeaderBytes = 64;       // workspace header: T, C_eff
constexpr int kMaxDevices = 64;        // per-device caches
// Warps of a decode CTA.  Four warps, with kMinCtas CTAs resident per SM
// (3 for E4M3, 2 for FP16): one CTA per SM with all 12 (E4M3) or 8 (FP16)
// warps measured within 2 % on the long decode and 3 to 6 % slower on short
// ones, where more independent CTAs start more loads at once.
template <bool kE4M3>
__host__ __device__ constexpr int kDecodeWarps()
{
    return kWarps;
}

// Virtual tiles charged at the start of every non-empty segment when the tile
// line is cut among the split CTAs: a CTA whose range takes in a segment start
// runs one more piece (Q staging, pipeline start, CTA merge, about 5 us at
// full load against 0.56 us per tile per CTA), so such CTAs get that much less
// real work.  8 to 20 were measured; 12 to 20 tie and beat 0 by about 4%.
constexpr int kPieceCostTiles = 12;

struct DecodeArgs {
    const __half* q;
    KVGeom kv;
    const int32_t* bt;
    int64_t bt_stride;
    const int32_t* seq_lens;
    int B, Hq, Hkv, G, max_seq_len;
    float scale_log2;    // softmax_scale * kv_scale(K) * log2(e)
    float v_scale;       // kv_scale for E4M3 V, 1 for FP16
    __half* out;
    // split route only
    int64_t* hdr;        // [0] = T (line length), [1] = C_eff, then prefix[B + 1]
    float* slots;        // (C + B * Hkv) partial slots
    int C;               // CTAs launched on the split route; 0 = unsplit route
    int min_tiles;       // minimum tiles per CTA when choosing C_eff
    int piece_cost;      // virtual tiles at the start of each non-empty segment
    int* err;
};

struct PrefillArgs {
    const __half* q;
    KVGeom kv;
    const int32_t* bt;
    int kv_len;
    const int32_t* sel;
    int n_sel;
    const int32_t* q_pos;
    int R, Hq, Hkv, G;
    float scale_log2, v_scale;
    __half* out;
    int* err;
};

// Grouped sparse prefill (prefill_grouped.cu): a union bitmap over the
// sequence's four-token blocks of at most kGroupMaxWords words.
constexpr int kGroupMaxWords = 1024;
constexpr int kGroupSlots = 128;      // query-head slots of a group: the M of one MMA

struct GroupArgs {
    PrefillArgs a;
    int Rg;              // query rows per group (unit = group x KV head)
    int n_units;
    int nbw;             // words of the union bitmap
    long spin_limit;     // polls of a bounded wait before it gives up
    int stall_stage;     // test hook: ring stage never published (-1: none)
};

struct SelectArgs {
    const float* scores;
    int64_t stride;
    int n_blocks;
    const int32_t* q_pos;
    int R, kv_len, k;
    int stage_keys;      // keys a CTA stages in shared memory (select_stage_keys)
    int32_t* out;
    int* err;
};

struct MaskArgs {
    const float* x;
    int64_t x_stride;
    float* out;
    int64_t out_stride;
    int B, V, k;
    int slice;           // columns per CTA of a row's cluster (mask_slice)
    float p;
    int* err;
};

size_t decode_split_smem(bool e4m3, int B);
size_t workspace_bytes(int B, int Hkv, int C);
size_t decode_workspace_bytes_for(int B, int Hq, int Hkv, int D, int kv_dtype);
int split_ctas_per_sm(bool e4m3);

cudaError_t launch_decode(const DecodeArgs& a, bool e4m3, cudaStream_t s, void* ev0, void* ev1);
cudaError_t launch_prefill(const PrefillArgs& a, bool e4m3, cudaStream_t s);
bool grouped_prefill_supported(const PrefillArgs& a);
int grouped_prefill_rows(const PrefillArgs& a, int clusters, int rows_per_group);
cudaError_t grouped_prefill_clusters(int& clusters);
cudaError_t launch_prefill_grouped(const PrefillArgs& a, bool e4m3, int rows_per_group,
                                   cudaStream_t s, long spin_limit = 0, int stall_stage = -1);
cudaError_t launch_gather(const KVGeom& g, bool e4m3, const int32_t* bt, int64_t bt_stride,
                          const int32_t* seq_lens, int B, int T, int Hkv, int max_seq_len,
                          float kv_scale, float* out, cudaStream_t s);
int select_stage_keys(int n_blocks);
int mask_slice(int V);
bool mask_supported(int V, int k);
cudaError_t launch_topk_topp(const MaskArgs& a, cudaStream_t s);
cudaError_t launch_select(const SelectArgs& a, cudaStream_t s);
cudaError_t launch_sparse_gather(const PrefillArgs& a, bool e4m3, uint32_t* out, cudaStream_t s);
cudaError_t launch_prefill_tokens(const KVGeom& g, const int32_t* bt, int kv_len,
                                  const int32_t* sel, int n_sel, const int32_t* q_pos, int R,
                                  int32_t* out, cudaStream_t s);

}  // namespace pgqa
