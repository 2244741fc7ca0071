"""Paged grouped-query attention on GB300 (sm_103a): Python binding.

A thin ctypes layer over ``libpaged_gqa.so`` (the C ABI declared in
``include/paged_gqa.h``).  It only marshals arguments: torch tensors supply
device pointers, strides and the current CUDA stream; every step of the
computation runs in the library's CUDA kernels.  There is no fallback: if the
library has not been built, every call raises.

Entry points keep the C names:

* ``paged_gqa_decode`` -- batched paged decode over FP16 or FP8-E4M3 KV
  ("[Kernel][SM70] Scale NVFP4 E4M3 decode batches", Purpose);
* ``paged_gqa_sparse_prefill`` -- selected-sparse prefill over four-token
  blocks ("[Kernel][SM70] Accelerate Qwen3.8 QSA paged prefill", Changes);
* ``paged_gqa_gather_dequant`` / ``paged_gqa_sparse_prefill_tokens`` --
  inspection of the kernels' gather and dequantisation;
* ``paged_gqa_decode_workspace_size``, ``paged_gqa_status_string``,
  ``paged_gqa_version``.
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "PagedGQAError", "library_path", "lib", "KV_FP16", "KV_E4M3",
    "FLAG_BAD_PAGE", "FLAG_SEQ_CLAMPED", "FLAG_EMPTY_ROW", "FLAG_QPOS_CLAMPED", "FLAG_BAD_SEL",
    "paged_gqa_decode", "paged_gqa_decode_noalloc", "paged_gqa_sparse_prefill",
    "paged_gqa_sparse_prefill_route", "paged_gqa_sparse_prefill_group_rows", "PREFILL_AUTO",
    "PREFILL_ROWWISE", "PREFILL_GROUPED", "paged_gqa_debug_grouped_prefill_stall",
    "paged_gqa_sparse_prefill_auto_route",
    "paged_gqa_gather_dequant", "paged_gqa_sparse_gather_probe",
    "paged_gqa_sparse_prefill_tokens", "paged_gqa_decode_workspace_size",
    "paged_gqa_decode_workspace_size_splits",
    "paged_gqa_status_string", "paged_gqa_version", "Workspace",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_HERE, "libpaged_gqa.so")

KV_FP16 = 0
KV_E4M3 = 1
FLAG_BAD_PAGE = 1
FLAG_SEQ_CLAMPED = 2
FLAG_EMPTY_ROW = 4
FLAG_QPOS_CLAMPED = 8
FLAG_BAD_SEL = 16
FLAG_SCORES_SHORT = 32
FLAG_BAD_LOGIT = 64
FLAG_TIMEOUT = 128


class PagedGQAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: status {status} ({paged_gqa_status_string(status)})")


class KVLayout(ctypes.Structure):
    _fields_ = [("page_stride", ctypes.c_int64), ("token_stride", ctypes.c_int64),
                ("head_stride", ctypes.c_int64)]


class Workspace(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p), ("bytes", ctypes.c_size_t),
                ("force_splits", ctypes.c_int), ("err_flag", ctypes.c_void_p),
                ("split_events", ctypes.c_void_p * 2)]


_lock = threading.Lock()
_lib = None


def lib():
    """The loaded C library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(library_path):
                raise RuntimeError(
                    f"{library_path} is missing: build it with "
                    "`python -m fp8_kv_cache_gb300.build` (there is no fallback path)")
            L = ctypes.CDLL(library_path)
            i32, i64, f32, vp, sz = (ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                                     ctypes.c_void_p, ctypes.c_size_t)
            L.paged_gqa_version.argtypes = []
            L.paged_gqa_version.restype = i32
            L.paged_gqa_status_string.argtypes = [i32]
            L.paged_gqa_status_string.restype = ctypes.c_char_p
            L.paged_gqa_decode_workspace_size.argtypes = [i32, i32, i32, i32, i32]
            L.paged_gqa_decode_workspace_size.restype = sz
            L.paged_gqa_decode_workspace_size_splits.argtypes = [i32, i32, i32, i32, i32]
            L.paged_gqa_decode_workspace_size_splits.restype = sz
            L.paged_gqa_decode.argtypes = [vp, vp, vp, KVLayout, i32, vp, i64, vp,
                                           i32, i32, i32, i32, i32, i32, i32, f32, f32,
                                           vp, ctypes.POINTER(Workspace), vp]
            L.paged_gqa_decode.restype = i32
            L.paged_gqa_decode_noalloc.argtypes = [vp, vp, vp, KVLayout, i32, vp, i64, vp,
                                                   i32, i32, i32, i32, i32, i32, i32, f32, f32,
                                                   vp, vp, vp]
            L.paged_gqa_decode_noalloc.restype = i32
            L.paged_gqa_sparse_prefill.argtypes = [vp, vp, vp, KVLayout, i32, vp, i32, i32,
                                                   vp, i32, vp, i32, i32, i32, i32, i32, f32, f32,
                                                   vp, vp, vp]
            L.paged_gqa_sparse_prefill.restype = i32
            L.paged_gqa_sparse_prefill_route.argtypes = [vp, vp, vp, KVLayout, i32, vp, i32, i32,
                                                         vp, i32, vp, i32, i32, i32, i32, i32,
                                                         f32, f32, vp, vp, vp, i32, i32]
            L.paged_gqa_sparse_prefill_route.restype = i32
            L.paged_gqa_debug_grouped_prefill_stall.argtypes = [
                vp, vp, vp, KVLayout, i32, vp, i32, i32, vp, i32, vp, i32, i32, i32, i32, i32,
                f32, f32, vp, vp, vp, ctypes.c_longlong, i32]
            L.paged_gqa_debug_grouped_prefill_stall.restype = i32
            L.paged_gqa_sparse_prefill_auto_route.argtypes = [i32, i32, i32, i32, i32, i32]
            L.paged_gqa_sparse_prefill_auto_route.restype = i32
            L.paged_gqa_sparse_prefill_group_rows.argtypes = [i32, i32, i32, i32]
            L.paged_gqa_sparse_prefill_group_rows.restype = i32
            L.paged_gqa_gather_dequant.argtypes = [vp, KVLayout, i32, vp, i64, vp, i32, i32, i32,
                                                   i32, i32, i32, i32, f32, vp, vp]
            L.paged_gqa_gather_dequant.restype = i32
            L.paged_gqa_sparse_prefill_tokens.argtypes = [vp, i32, i32, vp, i32, vp, i32, i32,
                                                          vp, vp]
            L.paged_gqa_sparse_prefill_tokens.restype = i32
            L.paged_gqa_sparse_gather_probe.argtypes = [vp, vp, KVLayout, i32, vp, i32, i32, vp,
                                                        i32, vp, i32, i32, i32, i32, vp, vp]
            L.paged_gqa_sparse_gather_probe.restype = i32
            L.paged_gqa_select_blocks.argtypes = [vp, i64, i32, vp, i32, i32, i32, vp, vp, vp]
            L.paged_gqa_select_blocks.restype = i32
            L.paged_gqa_topk_topp_mask.argtypes = [vp, i64, vp, i64, i32, i32, i32, f32, vp, vp]
            L.paged_gqa_topk_topp_mask.restype = i32
            _lib = L
    return _lib


def paged_gqa_version() -> int:
    return lib().paged_gqa_version()


def paged_gqa_status_string(status: int) -> str:
    return lib().paged_gqa_status_string(int(status)).decode()


def paged_gqa_decode_workspace_size(B, Hq, Hkv, D, max_seq_len) -> int:
    return int(lib().paged_gqa_decode_workspace_size(B, Hq, Hkv, D, max_seq_len))


def paged_gqa_decode_workspace_size_splits(B, Hq, Hkv, D, splits) -> int:
    return int(lib().paged_gqa_decode_workspace_size_splits(B, Hq, Hkv, D, splits))


# ------------------------------------------------------------------ helpers

def _torch():
    import torch
    return torch


def _kv_dtype(t) -> int:
    torch = _torch()
    if t.dtype == torch.float16:
        return KV_FP16
    if t.dtype in (torch.uint8, torch.float8_e4m3fn):
        return KV_E4M3
    raise TypeError(f"KV cache dtype {t.dtype} is neither float16 nor E4M3 (uint8/float8_e4m3fn)")


def _layout(k, v) -> KVLayout:
    """Element strides of 4-D K/V views [num_pages, page_size, Hkv, D]."""
    if k.dim() != 4 or v.dim() != 4 or k.shape != v.shape:
        raise ValueError("k_cache and v_cache must be 4-D [num_pages, page_size, Hkv, D] views")
    if k.stride() != v.stride() or k.stride(3) != 1:
        raise ValueError("k_cache and v_cache must share strides with unit head-dim stride")
    return KVLayout(k.stride(0), k.stride(1), k.stride(2))


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(_torch().cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check(status, where):
    if status != 0:
        raise PagedGQAError(status, where)


# ------------------------------------------------------------------ entry points

def paged_gqa_decode(q, k_cache, v_cache, block_table, seq_lens, page_size, kv_scale,
                     softmax_scale, out=None, *, max_seq_len, num_pages=None, workspace=None,
                     force_splits=0, err_flag=None, split_events=None, stream=None):
    """Batched paged GQA decode.

    q [B, Hq, 256] float16; k_cache/v_cache [num_pages, page_size, Hkv, 256]
    views (float16, or uint8/float8_e4m3fn codes); block_table int32 [B, >=
    ceil(max_seq_len/page_size)]; seq_lens int32 [B].  ``workspace``: a CUDA
    uint8 tensor of at least ``paged_gqa_decode_workspace_size`` bytes, None
    to allocate one, or False for the unsplit route.  ``err_flag``: optional
    CUDA int32 [1] receiving FLAG_* bits.  ``split_events``: optional pair of
    torch.cuda.Event recorded around the split kernel.  Returns ``out``."""
    torch = _torch()
    B, Hq, D = q.shape
    Hkv = k_cache.shape[2]
    if out is None:
        out = torch.empty_like(q)
    if num_pages is None:
        num_pages = k_cache.shape[0]
    ws = Workspace()
    ws.force_splits = int(force_splits)
    ws.err_flag = None if err_flag is None else err_flag.data_ptr()
    if split_events is not None:
        ws.split_events[0] = split_events[0].cuda_event
        ws.split_events[1] = split_events[1].cuda_event
    if workspace is None:
        nbytes = paged_gqa_decode_workspace_size(B, Hq, Hkv, D, max_seq_len)
        if force_splits:
            nbytes = max(nbytes, paged_gqa_decode_workspace_size_splits(B, Hq, Hkv, D,
                                                                        force_splits))
        workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=q.device)
    if workspace is not False:
        ws.ptr = workspace.data_ptr()
        ws.bytes = workspace.numel() * workspace.element_size()
    st = lib().paged_gqa_decode(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _layout(k_cache, v_cache), _kv_dtype(k_cache),
        _ptr(block_table), block_table.stride(0), _ptr(seq_lens),
        B, Hq, Hkv, D, page_size, num_pages, max_seq_len, float(kv_scale), float(softmax_scale),
        _ptr(out), ctypes.byref(ws), _stream(stream))
    _check(st, "paged_gqa_decode")
    return out


def paged_gqa_decode_noalloc(q, k_cache, v_cache, block_table, seq_lens, page_size, kv_scale,
                             softmax_scale, out=None, *, max_seq_len, num_pages=None,
                             err_flag=None, stream=None):
    """paged_gqa_decode for callers that cannot allocate device memory: the
    split scratch is the library's own 16 MiB static device array, so the
    call allocates nothing (``out`` is allocated here only when not given).
    Calls that may overlap on the GPU share that array and race; the first
    call on a device should precede any stream capture."""
    torch = _torch()
    B, Hq, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    if num_pages is None:
        num_pages = k_cache.shape[0]
    st = lib().paged_gqa_decode_noalloc(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _layout(k_cache, v_cache), _kv_dtype(k_cache),
        _ptr(block_table), block_table.stride(0), _ptr(seq_lens),
        B, Hq, k_cache.shape[2], D, page_size, num_pages, max_seq_len, float(kv_scale),
        float(softmax_scale), _ptr(out), _ptr(err_flag), _stream(stream))
    _check(st, "paged_gqa_decode_noalloc")
    return out


PREFILL_AUTO, PREFILL_ROWWISE, PREFILL_GROUPED = 0, 1, 2


def paged_gqa_sparse_prefill(q, k_cache, v_cache, block_table, kv_len, sel_idx, q_pos, page_size,
                             softmax_scale, kv_scale=1.0, out=None, *, num_pages=None,
                             err_flag=None, stream=None):
    """Selected-sparse prefill of one sequence.  q [R, Hq, 256] float16;
    sel_idx int32 [R, n_sel] four-token block ids; q_pos int32 [R]."""
    args, out = _prefill_args(q, k_cache, v_cache, block_table, kv_len, sel_idx, q_pos,
                              page_size, softmax_scale, kv_scale, out, num_pages, err_flag, stream)
    _check(lib().paged_gqa_sparse_prefill(*args), "paged_gqa_sparse_prefill")
    return out


def paged_gqa_sparse_prefill_route(q, k_cache, v_cache, block_table, kv_len, sel_idx, q_pos,
                                   page_size, softmax_scale, kv_scale=1.0, out=None, *,
                                   route=PREFILL_AUTO, rows_per_group=0, num_pages=None,
                                   err_flag=None, stream=None):
    """paged_gqa_sparse_prefill on a chosen kernel route (PREFILL_ROWWISE or
    PREFILL_GROUPED; rows_per_group 0 = automatic group size)."""
    args, out = _prefill_args(q, k_cache, v_cache, block_table, kv_len, sel_idx, q_pos,
                              page_size, softmax_scale, kv_scale, out, num_pages, err_flag, stream)
    _check(lib().paged_gqa_sparse_prefill_route(*args, int(route), int(rows_per_group)),
           "paged_gqa_sparse_prefill_route")
    return out


def paged_gqa_debug_grouped_prefill_stall(q, k_cache, v_cache, block_table, kv_len, sel_idx,
                                          q_pos, page_size, softmax_scale, kv_scale=1.0,
                                          out=None, *, spin_limit, stall_stage, num_pages=None,
                                          err_flag=None, stream=None):
    """Test hook of the grouped route's time-out path: every bounded wait
    gives up after ``spin_limit`` polls and each CTA leaves ring stage
    ``stall_stage`` unpublished (-1: none), so the kernel sets FLAG_TIMEOUT
    and leaves ``out`` undefined.  For tests of that path only."""
    args, out = _prefill_args(q, k_cache, v_cache, block_table, kv_len, sel_idx, q_pos,
                              page_size, softmax_scale, kv_scale, out, num_pages, err_flag, stream)
    _check(lib().paged_gqa_debug_grouped_prefill_stall(*args, int(spin_limit), int(stall_stage)),
           "paged_gqa_debug_grouped_prefill_stall")
    return out


def paged_gqa_sparse_prefill_auto_route(R, Hq, Hkv, kv_len, n_sel, kv_dtype=KV_FP16) -> int:
    """The route (PREFILL_ROWWISE or PREFILL_GROUPED) the automatic rule takes."""
    n = lib().paged_gqa_sparse_prefill_auto_route(int(R), int(Hq), int(Hkv), int(kv_len),
                                                  int(n_sel), int(kv_dtype))
    _check(min(n, 0), "paged_gqa_sparse_prefill_auto_route")
    return n


def paged_gqa_sparse_prefill_group_rows(R, Hq, Hkv, rows_per_group=0) -> int:
    """Rows per group of the grouped prefill route on the current device."""
    n = lib().paged_gqa_sparse_prefill_group_rows(int(R), int(Hq), int(Hkv), int(rows_per_group))
    _check(min(n, 0), "paged_gqa_sparse_prefill_group_rows")
    return n


def _prefill_args(q, k_cache, v_cache, block_table, kv_len, sel_idx, q_pos, page_size,
                  softmax_scale, kv_scale, out, num_pages, err_flag, stream):
    torch = _torch()
    R, Hq, D = q.shape
    Hkv = k_cache.shape[2]
    if out is None:
        out = torch.empty_like(q)
    if num_pages is None:
        num_pages = k_cache.shape[0]
    n_sel = sel_idx.shape[1] if sel_idx.dim() == 2 else 0
    return (_ptr(q), _ptr(k_cache), _ptr(v_cache), _layout(k_cache, v_cache),
            _kv_dtype(k_cache), _ptr(block_table), num_pages, kv_len,
            _ptr(sel_idx) if n_sel else None, n_sel, _ptr(q_pos), R, Hq, Hkv, D, page_size,
            float(kv_scale), float(softmax_scale), _ptr(out), _ptr(err_flag),
            _stream(stream)), out


def paged_gqa_gather_dequant(cache, block_table, seq_lens, page_size, max_seq_len, kv_scale=1.0,
                             T=None, *, num_pages=None, stream=None):
    """The rows the decode kernels gather, dequantised: float32 [B, T, Hkv, 256]."""
    torch = _torch()
    B = seq_lens.shape[0]
    T = max_seq_len if T is None else T
    Hkv, D = cache.shape[2], cache.shape[3]
    if num_pages is None:
        num_pages = cache.shape[0]
    out = torch.empty((B, T, Hkv, D), dtype=torch.float32, device=cache.device)
    st = lib().paged_gqa_gather_dequant(
        _ptr(cache), _layout(cache, cache), _kv_dtype(cache), _ptr(block_table),
        block_table.stride(0), _ptr(seq_lens), B, T, Hkv, D, page_size, num_pages, max_seq_len,
        float(kv_scale), _ptr(out), _stream(stream))
    _check(st, "paged_gqa_gather_dequant")
    return out


def paged_gqa_sparse_prefill_tokens(block_table, num_pages, kv_len, sel_idx, q_pos, page_size,
                                    *, stream=None):
    """Per-row token slots of the sparse-prefill kernel: int32 [R, 4*(n_sel+1)], -1 = unused."""
    torch = _torch()
    R = q_pos.shape[0]
    n_sel = sel_idx.shape[1] if sel_idx.dim() == 2 else 0
    out = torch.empty((R, 4 * (n_sel + 1)), dtype=torch.int32, device=q_pos.device)
    st = lib().paged_gqa_sparse_prefill_tokens(
        _ptr(block_table), num_pages, kv_len, _ptr(sel_idx) if n_sel else None, n_sel,
        _ptr(q_pos), R, page_size, _ptr(out), _stream(stream))
    _check(st, "paged_gqa_sparse_prefill_tokens")
    return out


def paged_gqa_sparse_gather_probe(k_cache, v_cache, block_table, kv_len, sel_idx, q_pos,
                                  page_size, *, num_pages=None, out=None, stream=None):
    """The per-row prefill route's gather alone (a measurement helper):
    returns uint32 [R, Hkv], per row and KV head the XOR of every 32-bit word
    of the K and V rows it attends."""
    torch = _torch()
    R = q_pos.shape[0]
    Hkv, D = k_cache.shape[2], k_cache.shape[3]
    n_sel = sel_idx.shape[1] if sel_idx.dim() == 2 else 0
    if num_pages is None:
        num_pages = k_cache.shape[0]
    if out is None:
        out = torch.empty((R, Hkv), dtype=torch.int32, device=k_cache.device)
    st = lib().paged_gqa_sparse_gather_probe(
        _ptr(k_cache), _ptr(v_cache), _layout(k_cache, v_cache), _kv_dtype(k_cache),
        _ptr(block_table), num_pages, kv_len, _ptr(sel_idx) if n_sel else None, n_sel,
        _ptr(q_pos), R, Hkv, D, page_size, _ptr(out), _stream(stream))
    _check(st, "paged_gqa_sparse_gather_probe")
    return out


def paged_gqa_select_blocks(scores, q_pos, kv_len, k, *, n_blocks=None, out=None, err_flag=None,
                            stream=None):
    """QSA block selection: for each row the min(k, n) best of its causal
    blocks by score (ties to the lower index), ascending, padded with -1.
    scores float32 [R, >= n_blocks] on the GPU (unit column stride, any row
    stride); q_pos int32 [R].  Returns int32 [R, k]."""
    torch = _torch()
    if scores.dtype != torch.float32 or scores.dim() != 2 or scores.stride(1) != 1:
        raise ValueError("scores must be a 2-D float32 tensor with unit column stride")
    R = scores.shape[0]
    n_blocks = scores.shape[1] if n_blocks is None else int(n_blocks)
    if out is None:
        out = torch.empty((R, int(k)), dtype=torch.int32, device=scores.device)
    st = lib().paged_gqa_select_blocks(_ptr(scores), scores.stride(0), n_blocks, _ptr(q_pos), R,
                                       int(kv_len), int(k), _ptr(out), _ptr(err_flag),
                                       _stream(stream))
    _check(st, "paged_gqa_select_blocks")
    return out


def paged_gqa_topk_topp_mask(logits, k, p, *, out=None, err_flag=None, stream=None):
    """Combined top-k/top-p masking: the kept logits unchanged, -inf
    elsewhere.  logits float32 [B, V] on the GPU (unit column stride);
    ``out=logits`` masks in place.  Returns out."""
    torch = _torch()
    if logits.dtype != torch.float32 or logits.dim() != 2 or logits.stride(1) != 1:
        raise ValueError("logits must be a 2-D float32 tensor with unit column stride")
    B, V = logits.shape
    if out is None:
        out = torch.empty_like(logits)
    if out.shape != logits.shape or out.dtype != torch.float32 or out.stride(1) != 1:
        raise ValueError("out must match logits")
    st = lib().paged_gqa_topk_topp_mask(_ptr(logits), logits.stride(0), _ptr(out), out.stride(0),
                                        B, V, int(k), float(p), _ptr(err_flag), _stream(stream))
    _check(st, "paged_gqa_topk_topp_mask")
    return out
