// api.cu -- the extern "C" entry points declared in include/paged_gqa.h:
// host-side validation, the split-count choice and the launches.  Nothing
// here allocates memory or synchronises the host.
#include <atomic>
#include <cmath>

#include "pgqa_internal.h"

using namespace pgqa;

namespace {

constexpr double kLog2e = 1.4426950408889634;

bool aligned16(const void* p)
{
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

int elem_bytes(int kv_dtype)
{
    return kv_dtype == PAGED_GQA_KV_E4M3 ? 1 : 2;
}

int log2_if_pow2(int x)
{
    if (x <= 0 || (x & (x - 1)) != 0)
        return -1;
    int s = 0;
    while ((1 << s) < x)
        ++s;
    return s;
}

// Common checks of the KV pools and layout.
int check_kv(const void* k, const void* v, const paged_gqa_kv_layout& L, int kv_dtype)
{
    if (kv_dtype != PAGED_GQA_KV_FP16 && kv_dtype != PAGED_GQA_KV_E4M3)
        return PAGED_GQA_ERR_UNSUPPORTED;
    if (k == nullptr || v == nullptr)
        return PAGED_GQA_ERR_NULL_POINTER;
    if (!aligned16(k) || !aligned16(v))
        return PAGED_GQA_ERR_ALIGNMENT;
    if (L.page_stride < 0 || L.token_stride < 0 || L.head_stride < 0)
        return PAGED_GQA_ERR_SHAPE;
    const int64_t e = elem_bytes(kv_dtype);
    if ((L.page_stride * e) % 16 || (L.token_stride * e) % 16 || (L.head_stride * e) % 16)
        return PAGED_GQA_ERR_ALIGNMENT;
    return PAGED_GQA_OK;
}

KVGeom make_geom(const void* k, const void* v, const paged_gqa_kv_layout& L, int kv_dtype,
                 int page_size, int num_pages)
{
    const int64_t e = elem_bytes(kv_dtype);
    KVGeom g;
    g.k = static_cast<const unsigned char*>(k);
    g.v = static_cast<const unsigned char*>(v);
    g.page_b = L.page_stride * e;
    g.token_b = L.token_stride * e;
    g.head_b = L.head_stride * e;
    g.page_size = page_size;
    g.page_shift = log2_if_pow2(page_size);
    g.num_pages = num_pages;
    return g;
}

// Per-device cache of the SM count and of the split kernel's CTAs per SM.
struct DeviceInfo {
    int sms;
    int ctas_fp16;
    int ctas_e4m3;
};

int device_info(DeviceInfo& out)
{
    static std::atomic<int> sms[kMaxDevices], c16[kMaxDevices], c8[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return PAGED_GQA_ERR_CUDA;
    if (dev < kMaxDevices && sms[dev].load(std::memory_order_acquire) > 0) {
        out.sms = sms[dev].load(std::memory_order_acquire);
        out.ctas_fp16 = c16[dev].load(std::memory_order_relaxed);
        out.ctas_e4m3 = c8[dev].load(std::memory_order_relaxed);
        return PAGED_GQA_OK;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        return PAGED_GQA_ERR_CUDA;
    out.sms = n;
    out.ctas_fp16 = split_ctas_per_sm(false);
    out.ctas_e4m3 = split_ctas_per_sm(true);
    if (dev < kMaxDevices) {
        c16[dev].store(out.ctas_fp16, std::memory_order_relaxed);
        c8[dev].store(out.ctas_e4m3, std::memory_order_relaxed);
        sms[dev].store(n, std::memory_order_release);
    }
    return PAGED_GQA_OK;
}

int check_decode_shape(int B, int Hq, int Hkv, int D, int max_seq_len)
{
    if (B < 0 || Hq < 1 || Hkv < 1 || max_seq_len < 0)
        return PAGED_GQA_ERR_SHAPE;
    if (Hq % Hkv != 0 || (int64_t)B * Hq > INT32_MAX)   // one CTA per (b, KV head) at most
        return PAGED_GQA_ERR_SHAPE;
    if (D != kD || Hq / Hkv > kGMax)
        return PAGED_GQA_ERR_UNSUPPORTED;
    return PAGED_GQA_OK;
}

int prefill_route_impl(const void* q, const void* k_cache, const void* v_cache,
                       paged_gqa_kv_layout kv_layout, int kv_dtype, const int32_t* block_table,
                       int num_pages, int kv_len, const int32_t* sel_idx, int n_sel,
                       const int32_t* q_pos, int R, int Hq, int Hkv, int D, int page_size,
                       float kv_scale, float softmax_scale, void* out, int* err_flag,
                       void* stream, int route, int rows_per_group, long spin_limit,
                       int stall_stage);

// Automatic route choice (the grouped route must also support the shape).
// The grouped kernel pays a fixed cost per call (a unit's setup and the
// pair exchange, ~20 us) and then gathers each row group's union of blocks
// once; the per-row kernel gathers every row's blocks for that row alone.
// Measured over 32768 tokens (L2 flushed before each call):
//  * FP16, 4096 rows: grouped is faster at every density measured, from 16
//    selections (0.087 vs 0.133 ms) through 512 (0.552 vs 0.820 ms) to 2048
//    (0.871 vs 2.974 ms); from 1024 rows on it is faster from 16 selections
//    (33 vs 42 us at 1024 rows);
//  * FP16, 1 to 512 rows: per row is faster up to 128 selections (15 vs
//    27 us at 128 rows x 16, 48 vs 52 us at 512 rows x 128), grouped from
//    512 (46 vs 60 us at 1 row, 111 vs 128 us at 512 rows: a unit's
//    half-tiles are split over two SMs);
//  * E4M3, 4096 rows: the per-row gather moves half the bytes while the
//    grouped route converts them to binary16 as it gathers; they cross over
//    between 768 selections (0.898 vs 0.850 ms) and 1024 (0.954 vs
//    1.103 ms), near 850; at 1 to 512 rows per row is as fast or faster
//    through 512 selections.
// Rule, with rows x KV heads = the per-row kernel's CTAs: FP16 grouped when
// 64 n_sel >= kv_len, or when rows x KV heads >= 1024 and 2048 n_sel >=
// kv_len; E4M3 grouped when rows x KV heads >= 1024 and 36 n_sel >= kv_len.
bool auto_picks_grouped(int R, int Hkv, int n_sel, int kv_len, bool e4m3)
{
    const int64_t ctas = (int64_t)R * Hkv, sel = n_sel;
    if (e4m3)
        return ctas >= 1024 && 36 * sel >= (int64_t)kv_len;
    return 64 * sel >= (int64_t)kv_len || (ctas >= 1024 && 2048 * sel >= (int64_t)kv_len);
}

}  // namespace

extern "C" {

int paged_gqa_version(void)
{
    return PAGED_GQA_VERSION;
}

const char* paged_gqa_status_string(int status)
{
    switch (status) {
    case PAGED_GQA_OK: return "ok";
    case PAGED_GQA_ERR_NULL_POINTER: return "a required pointer is NULL";
    case PAGED_GQA_ERR_ALIGNMENT: return "a pointer or stride is not 16-byte aligned";
    case PAGED_GQA_ERR_SHAPE: return "inconsistent or out-of-range sizes";
    case PAGED_GQA_ERR_UNSUPPORTED: return "unsupported head dim, group size or KV dtype";
    case PAGED_GQA_ERR_WORKSPACE: return "workspace too small or misaligned";
    case PAGED_GQA_ERR_CUDA: return "a CUDA runtime call or launch failed";
    default: return "unknown status";
    }
}

size_t paged_gqa_decode_workspace_size(int B, int Hq, int Hkv, int D, int max_seq_len)
{
    if (check_decode_shape(B, Hq, Hkv, D, max_seq_len) != PAGED_GQA_OK)
        return 0;
    if (B > kMaxSplitBatch)
        return 0;   // such batches take the unsplit route
    DeviceInfo di;
    if (device_info(di) != PAGED_GQA_OK)
        return 0;
    const int per = di.ctas_fp16 > di.ctas_e4m3 ? di.ctas_fp16 : di.ctas_e4m3;
    return workspace_bytes(B, Hkv, di.sms * per);
}

size_t paged_gqa_decode_workspace_size_splits(int B, int Hq, int Hkv, int D, int splits)
{
    if (check_decode_shape(B, Hq, Hkv, D, 0) != PAGED_GQA_OK || splits < 1 || B > kMaxSplitBatch)
        return 0;
    return workspace_bytes(B, Hkv, splits);
}

int paged_gqa_decode(const void* q, const void* k_cache, const void* v_cache,
                     paged_gqa_kv_layout kv_layout, int kv_dtype, const int32_t* block_table,
                     int64_t bt_row_stride, const int32_t* seq_lens, int B, int Hq, int Hkv, int D,
                     int page_size, int num_pages, int max_seq_len, float kv_scale,
                     float softmax_scale, void* out, const paged_gqa_workspace* ws, void* stream)
{
    int st = check_decode_shape(B, Hq, Hkv, D, max_seq_len);
    if (st != PAGED_GQA_OK)
        return st;
    if (page_size < 1 || num_pages < 1 || bt_row_stride < 0)
        return PAGED_GQA_ERR_SHAPE;
    if (B > 1 && bt_row_stride < (int64_t)((max_seq_len + page_size - 1) / page_size))
        return PAGED_GQA_ERR_SHAPE;
    if ((st = check_kv(k_cache, v_cache, kv_layout, kv_dtype)) != PAGED_GQA_OK)
        return st;
    if (q == nullptr || block_table == nullptr || seq_lens == nullptr || out == nullptr)
        return PAGED_GQA_ERR_NULL_POINTER;
    if (!aligned16(q) || !aligned16(out))
        return PAGED_GQA_ERR_ALIGNMENT;
    if (B == 0)
        return PAGED_GQA_OK;

    const bool e4m3 = kv_dtype == PAGED_GQA_KV_E4M3;
    DecodeArgs a{};
    a.q = static_cast<const __half*>(q);
    a.kv = make_geom(k_cache, v_cache, kv_layout, kv_dtype, page_size, num_pages);
    a.bt = block_table;
    a.bt_stride = bt_row_stride;
    a.seq_lens = seq_lens;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.G = Hq / Hkv;
    a.max_seq_len = max_seq_len;
    a.scale_log2 = (float)((double)softmax_scale * (e4m3 ? (double)kv_scale : 1.0) * kLog2e);
    a.v_scale = e4m3 ? kv_scale : 1.f;
    a.out = static_cast<__half*>(out);
    a.err = ws ? ws->err_flag : nullptr;
    a.C = 0;

    const bool split = ws != nullptr && ws->ptr != nullptr && B <= kMaxSplitBatch;
    if (split) {
        if ((reinterpret_cast<uintptr_t>(ws->ptr) & 255u) != 0)
            return PAGED_GQA_ERR_WORKSPACE;
        DeviceInfo di;
        if (device_info(di) != PAGED_GQA_OK)
            return PAGED_GQA_ERR_CUDA;
        int C = ws->force_splits > 0 ? ws->force_splits
                                     : di.sms * (e4m3 ? di.ctas_e4m3 : di.ctas_fp16);
        if (workspace_bytes(B, Hkv, C) > ws->bytes)
            return PAGED_GQA_ERR_WORKSPACE;
        size_t head = kHeaderBytes + (size_t)(B + 1) * sizeof(int64_t);
        head = (head + 255) & ~(size_t)255;
        a.hdr = static_cast<int64_t*>(ws->ptr);
        a.slots = reinterpret_cast<float*>(static_cast<unsigned char*>(ws->ptr) + head);
        a.C = C;
        a.min_tiles = ws->force_splits > 0 ? 0 : 8;
        a.piece_cost = kPieceCostTiles;
    }
    void* ev0 = ws ? ws->split_events[0] : nullptr;
    void* ev1 = ws ? ws->split_events[1] : nullptr;
    const cudaError_t e = launch_decode(a, e4m3, static_cast<cudaStream_t>(stream), ev0, ev1);
    return e == cudaSuccess ? PAGED_GQA_OK : PAGED_GQA_ERR_CUDA;
}

int paged_gqa_sparse_prefill(const void* q, const void* k_cache, const void* v_cache,
                             paged_gqa_kv_layout kv_layout, int kv_dtype,
                             const int32_t* block_table, int num_pages, int kv_len,
                             const int32_t* sel_idx, int n_sel, const int32_t* q_pos, int R,
                             int Hq, int Hkv, int D, int page_size, float kv_scale,
                             float softmax_scale, void* out, int* err_flag, void* stream)
{
    return paged_gqa_sparse_prefill_route(q, k_cache, v_cache, kv_layout, kv_dtype, block_table,
                                          num_pages, kv_len, sel_idx, n_sel, q_pos, R, Hq, Hkv,
                                          D, page_size, kv_scale, softmax_scale, out, err_flag,
                                          stream, PAGED_GQA_PREFILL_AUTO, 0);
}

int paged_gqa_sparse_prefill_route(const void* q, const void* k_cache, const void* v_cache,
                                   paged_gqa_kv_layout kv_layout, int kv_dtype,
                                   const int32_t* block_table, int num_pages, int kv_len,
                                   const int32_t* sel_idx, int n_sel, const int32_t* q_pos,
                                   int R, int Hq, int Hkv, int D, int page_size, float kv_scale,
                                   float softmax_scale, void* out, int* err_flag, void* stream,
                                   int route, int rows_per_group)
{
    return prefill_route_impl(q, k_cache, v_cache, kv_layout, kv_dtype, block_table, num_pages,
                              kv_len, sel_idx, n_sel, q_pos, R, Hq, Hkv, D, page_size, kv_scale,
                              softmax_scale, out, err_flag, stream, route, rows_per_group, 0, -1);
}

int paged_gqa_debug_grouped_prefill_stall(const void* q, const void* k_cache, const void* v_cache,
                                          paged_gqa_kv_layout kv_layout, int kv_dtype,
                                          const int32_t* block_table, int num_pages, int kv_len,
                                          const int32_t* sel_idx, int n_sel, const int32_t* q_pos,
                                          int R, int Hq, int Hkv, int D, int page_size,
                                          float kv_scale, float softmax_scale, void* out,
                                          int* err_flag, void* stream, long long spin_limit,
                                          int stall_stage)
{
    if (spin_limit < 0 || spin_limit > (1LL << 30) || stall_stage < -1)
        return PAGED_GQA_ERR_SHAPE;
    return prefill_route_impl(q, k_cache, v_cache, kv_layout, kv_dtype, block_table, num_pages,
                              kv_len, sel_idx, n_sel, q_pos, R, Hq, Hkv, D, page_size, kv_scale,
                              softmax_scale, out, err_flag, stream, PAGED_GQA_PREFILL_GROUPED, 0,
                              (long)spin_limit, stall_stage);
}

}  // extern "C"

namespace {

int prefill_route_impl(const void* q, const void* k_cache, const void* v_cache,
                       paged_gqa_kv_layout kv_layout, int kv_dtype, const int32_t* block_table,
                       int num_pages, int kv_len, const int32_t* sel_idx, int n_sel,
                       const int32_t* q_pos, int R, int Hq, int Hkv, int D, int page_size,
                       float kv_scale, float softmax_scale, void* out, int* err_flag,
                       void* stream, int route, int rows_per_group, long spin_limit,
                       int stall_stage)
{
    if (route < PAGED_GQA_PREFILL_AUTO || route > PAGED_GQA_PREFILL_GROUPED ||
        rows_per_group < 0)
        return PAGED_GQA_ERR_SHAPE;
    if (R < 0 || n_sel < 0 || Hq < 1 || Hkv < 1 || kv_len < 0 || Hq % Hkv != 0)
        return PAGED_GQA_ERR_SHAPE;
    if (D != kD || Hq / Hkv > kGMax)
        return PAGED_GQA_ERR_UNSUPPORTED;
    if (page_size < 4 || page_size % 4 != 0 || num_pages < 1 || Hkv > 65535)
        return PAGED_GQA_ERR_SHAPE;
    if (n_sel > (1 << 28))
        return PAGED_GQA_ERR_SHAPE;
    int st = check_kv(k_cache, v_cache, kv_layout, kv_dtype);
    if (st != PAGED_GQA_OK)
        return st;
    if (q == nullptr || block_table == nullptr || q_pos == nullptr || out == nullptr ||
        (n_sel > 0 && sel_idx == nullptr))
        return PAGED_GQA_ERR_NULL_POINTER;
    if (!aligned16(q) || !aligned16(out))
        return PAGED_GQA_ERR_ALIGNMENT;
    if (R == 0)
        return PAGED_GQA_OK;
    const bool e4m3 = kv_dtype == PAGED_GQA_KV_E4M3;
    PrefillArgs a{};
    a.q = static_cast<const __half*>(q);
    a.kv = make_geom(k_cache, v_cache, kv_layout, kv_dtype, page_size, num_pages);
    a.bt = block_table;
    a.kv_len = kv_len;
    a.sel = sel_idx;
    a.n_sel = n_sel;
    a.q_pos = q_pos;
    a.R = R;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.G = Hq / Hkv;
    a.scale_log2 = (float)((double)softmax_scale * (e4m3 ? (double)kv_scale : 1.0) * kLog2e);
    a.v_scale = e4m3 ? kv_scale : 1.f;
    a.out = static_cast<__half*>(out);
    a.err = err_flag;
    const bool grouped_ok = grouped_prefill_supported(a);
    if (route == PAGED_GQA_PREFILL_GROUPED && !grouped_ok)
        return PAGED_GQA_ERR_UNSUPPORTED;
    if (rows_per_group > kGroupSlots / a.G)
        return PAGED_GQA_ERR_SHAPE;
    const bool grouped = route == PAGED_GQA_PREFILL_GROUPED ||
                         (route == PAGED_GQA_PREFILL_AUTO && grouped_ok &&
                          auto_picks_grouped(R, Hkv, n_sel, kv_len, e4m3));
    const cudaError_t e =
        grouped ? launch_prefill_grouped(a, e4m3, rows_per_group, static_cast<cudaStream_t>(stream),
                                         spin_limit, stall_stage)
                : launch_prefill(a, e4m3, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PAGED_GQA_OK : PAGED_GQA_ERR_CUDA;
}

}  // namespace

extern "C" {

int paged_gqa_sparse_prefill_auto_route(int R, int Hq, int Hkv, int kv_len, int n_sel,
                                        int kv_dtype)
{
    if (R < 0 || n_sel < 0 || Hq < 1 || Hkv < 1 || kv_len < 0 || Hq % Hkv != 0)
        return PAGED_GQA_ERR_SHAPE;
    if (Hq / Hkv > kGMax || (kv_dtype != PAGED_GQA_KV_FP16 && kv_dtype != PAGED_GQA_KV_E4M3))
        return PAGED_GQA_ERR_UNSUPPORTED;
    PrefillArgs a{};
    a.R = R;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.G = Hq / Hkv;
    a.kv_len = kv_len;
    return grouped_prefill_supported(a) && auto_picks_grouped(R, Hkv, n_sel, kv_len,
                                                               kv_dtype == PAGED_GQA_KV_E4M3)
               ? PAGED_GQA_PREFILL_GROUPED
               : PAGED_GQA_PREFILL_ROWWISE;
}

int paged_gqa_sparse_prefill_group_rows(int R, int Hq, int Hkv, int rows_per_group)
{
    if (R < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || rows_per_group < 0)
        return PAGED_GQA_ERR_SHAPE;
    if (Hq / Hkv > kGMax)
        return PAGED_GQA_ERR_UNSUPPORTED;
    if (rows_per_group > kGroupSlots / (Hq / Hkv))
        return PAGED_GQA_ERR_SHAPE;
    int clusters = 0;
    if (grouped_prefill_clusters(clusters) != cudaSuccess || clusters <= 0)
        return PAGED_GQA_ERR_CUDA;
    PrefillArgs a{};
    a.R = R;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.G = Hq / Hkv;
    return grouped_prefill_rows(a, clusters, rows_per_group);
}

int paged_gqa_gather_dequant(const void* cache, paged_gqa_kv_layout kv_layout, int kv_dtype,
                             const int32_t* block_table, int64_t bt_row_stride,
                             const int32_t* seq_lens, int B, int T, int Hkv, int D, int page_size,
                             int num_pages, int max_seq_len, float kv_scale, float* out,
                             void* stream)
{
    if (B < 0 || T < 0 || Hkv < 1 || page_size < 1 || num_pages < 1 || max_seq_len < 0 ||
        bt_row_stride < 0 || B > 65535 || Hkv > 65535)
        return PAGED_GQA_ERR_SHAPE;
    if (D != kD)
        return PAGED_GQA_ERR_UNSUPPORTED;
    int st = check_kv(cache, cache, kv_layout, kv_dtype);
    if (st != PAGED_GQA_OK)
        return st;
    if (block_table == nullptr || seq_lens == nullptr || out == nullptr)
        return PAGED_GQA_ERR_NULL_POINTER;
    if (!aligned16(out))
        return PAGED_GQA_ERR_ALIGNMENT;
    if (B == 0 || T == 0)
        return PAGED_GQA_OK;
    const KVGeom g = make_geom(cache, cache, kv_layout, kv_dtype, page_size, num_pages);
    const cudaError_t e = launch_gather(g, kv_dtype == PAGED_GQA_KV_E4M3, block_table,
                                       bt_row_stride, seq_lens, B, T, Hkv, max_seq_len, kv_scale,
                                       out, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PAGED_GQA_OK : PAGED_GQA_ERR_CUDA;
}

int paged_gqa_sparse_gather_probe(const void* k_cache, const void* v_cache,
                                  paged_gqa_kv_layout kv_layout, int kv_dtype,
                                  const int32_t* block_table, int num_pages, int kv_len,
                                  const int32_t* sel_idx, int n_sel, const int32_t* q_pos, int R,
                                  int Hkv, int D, int page_size, uint32_t* out, void* stream)
{
    if (R < 0 || n_sel < 0 || kv_len < 0 || Hkv < 1 || Hkv > 65535 || num_pages < 1 ||
        page_size < 4 || page_size % 4 != 0 || n_sel > (1 << 28))
        return PAGED_GQA_ERR_SHAPE;
    if (D != kD)
        return PAGED_GQA_ERR_UNSUPPORTED;
    int st = check_kv(k_cache, v_cache, kv_layout, kv_dtype);
    if (st != PAGED_GQA_OK)
        return st;
    if (block_table == nullptr || q_pos == nullptr || out == nullptr ||
        (n_sel > 0 && sel_idx == nullptr))
        return PAGED_GQA_ERR_NULL_POINTER;
    if ((reinterpret_cast<uintptr_t>(out) & 3u) != 0)
        return PAGED_GQA_ERR_ALIGNMENT;
    if (R == 0)
        return PAGED_GQA_OK;
    PrefillArgs a{};
    a.kv = make_geom(k_cache, v_cache, kv_layout, kv_dtype, page_size, num_pages);
    a.bt = block_table;
    a.kv_len = kv_len;
    a.sel = sel_idx;
    a.n_sel = n_sel;
    a.q_pos = q_pos;
    a.R = R;
    a.Hkv = Hkv;
    a.Hq = Hkv;
    a.G = 1;
    const cudaError_t e = launch_sparse_gather(a, kv_dtype == PAGED_GQA_KV_E4M3, out,
                                               static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PAGED_GQA_OK : PAGED_GQA_ERR_CUDA;
}

int paged_gqa_sparse_prefill_tokens(const int32_t* block_table, int num_pages, int kv_len,
                                    const int32_t* sel_idx, int n_sel, const int32_t* q_pos,
                                    int R, int page_size, int32_t* out, void* stream)
{
    if (R < 0 || n_sel < 0 || kv_len < 0 || num_pages < 1 || page_size < 4 ||
        page_size % 4 != 0 || n_sel > (1 << 28))
        return PAGED_GQA_ERR_SHAPE;
    if (block_table == nullptr || q_pos == nullptr || out == nullptr ||
        (n_sel > 0 && sel_idx == nullptr))
        return PAGED_GQA_ERR_NULL_POINTER;
    if (R == 0)
        return PAGED_GQA_OK;
    paged_gqa_kv_layout L{0, 0, 0};
    const KVGeom g = make_geom(nullptr, nullptr, L, PAGED_GQA_KV_FP16, page_size, num_pages);
    const cudaError_t e = launch_prefill_tokens(g, block_table, kv_len, sel_idx, n_sel, q_pos, R,
                                                out, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PAGED_GQA_OK : PAGED_GQA_ERR_CUDA;
}

int paged_gqa_select_blocks(const float* scores, int64_t score_stride, int n_blocks,
                            const int32_t* q_pos, int R, int kv_len, int k,
                            int32_t* sel_out, int* err_flag, void* stream)
{
    if (R < 0 || k < 0 || n_blocks < 0 || score_stride < n_blocks)
        return PAGED_GQA_ERR_SHAPE;
    if (q_pos == nullptr || (k > 0 && sel_out == nullptr) || (n_blocks > 0 && scores == nullptr))
        return PAGED_GQA_ERR_NULL_POINTER;
    if (R == 0 || k == 0)
        return PAGED_GQA_OK;
    SelectArgs a{};
    a.scores = scores;
    a.stride = score_stride;
    a.n_blocks = n_blocks;
    a.q_pos = q_pos;
    a.R = R;
    a.kv_len = kv_len;
    a.k = k;
    a.stage_keys = select_stage_keys(n_blocks);
    a.out = sel_out;
    a.err = err_flag;
    const cudaError_t e = launch_select(a, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PAGED_GQA_OK : PAGED_GQA_ERR_CUDA;
}

int paged_gqa_topk_topp_mask(const float* logits, int64_t logits_stride, float* out,
                             int64_t out_stride, int B, int V, int k, float p, int* err_flag,
                             void* stream)
{
    if (B < 0 || B > (1 << 27) || V < 1 || logits_stride < V || out_stride < V ||
        !(p > 0.f && p <= 1.f))
        return PAGED_GQA_ERR_SHAPE;
    if (!mask_supported(V, k))
        return k < 1 ? PAGED_GQA_ERR_SHAPE : PAGED_GQA_ERR_UNSUPPORTED;
    if (logits == nullptr || out == nullptr)
        return PAGED_GQA_ERR_NULL_POINTER;
    if (out == logits && out_stride != logits_stride)
        return PAGED_GQA_ERR_SHAPE;
    if (B == 0)
        return PAGED_GQA_OK;
    MaskArgs a{};
    a.x = logits;
    a.x_stride = logits_stride;
    a.out = out;
    a.out_stride = out_stride;
    a.B = B;
    a.V = V;
    a.k = k;
    a.slice = mask_slice(V);
    a.p = p;
    a.err = err_flag;
    const cudaError_t e = launch_topk_topp(a, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PAGED_GQA_OK : PAGED_GQA_ERR_CUDA;
}

}  // extern "C"

namespace pgqa {

// Workspace bytes paged_gqa_decode needs for this shape with its automatic
// split count on the current device for the given KV dtype (0 when the shape
// is invalid or takes the unsplit route).
size_t decode_workspace_bytes_for(int B, int Hq, int Hkv, int D, int kv_dtype)
{
    if (check_decode_shape(B, Hq, Hkv, D, 0) != PAGED_GQA_OK || B > kMaxSplitBatch)
        return 0;
    DeviceInfo di;
    if (device_info(di) != PAGED_GQA_OK)
        return 0;
    const int per = kv_dtype == PAGED_GQA_KV_E4M3 ? di.ctas_e4m3 : di.ctas_fp16;
    return workspace_bytes(B, Hkv, di.sms * per);
}

}  // namespace pgqa
