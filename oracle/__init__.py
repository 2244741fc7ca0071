"""FP64 CPU oracle for paged grouped-query attention (TEST INFRASTRUCTURE).

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product package never imports it and shares
no code with it.

The arithmetic lives in ``paged_gqa_oracle.c`` (plain C, FP64).  This module
compiles it with gcc and marshals numpy arrays into it.  The passages it
follows (1Cat-vLLM pull requests):

* decode: "[Kernel][SM70] Scale NVFP4 E4M3 decode batches" (#282), Purpose;
* sparse prefill and the inert-input rules: "[Kernel][SM70] Accelerate Qwen3.8
  QSA paged prefill" (#378), Changes;
* QSA block selection (top-k of block scores, ties to the lower index):
  "[Kernel][SM70] Accelerate exact Qwen3.8 decode" (#415), Implementation;
* the combined top-k/top-p masking of the decode step's logits: "[Kernel]
  [SM70] Scale NVFP4 E4M3 decode batches" (#282), Purpose.

``Oracle(path)`` loads any compiled copy of the source (the tests use this to
check that deliberately broken copies fail the pins); the module-level
functions use the default build next to this file.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "paged_gqa_oracle.c")
LIBRARY = os.path.join(HERE, "libpaged_gqa_oracle.so")

# Status bits the oracle ORs into its flag word.
FLAG_BAD_PAGE = 1
FLAG_SEQ_CLAMPED = 2
FLAG_EMPTY_ROW = 4
FLAG_QPOS_CLAMPED = 8
FLAG_BAD_SEL = 16
FLAG_SCORES_SHORT = 32


def compile_source(src: str, out: str) -> str:
    """gcc -O2 with OpenMP and no floating-point contraction, so that x86 and
    Arm hosts produce the same results."""
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile the default oracle library if it is missing or stale."""
    if force or not os.path.exists(LIBRARY) or os.path.getmtime(LIBRARY) < os.path.getmtime(SOURCE):
        compile_source(SOURCE, LIBRARY)
    return LIBRARY


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)))


def _ptr(a):
    return None if a is None else a.ctypes.data


def _kv_strides(k: np.ndarray, v: np.ndarray):
    """Element strides (page, token, head) of 4-D K and V views
    [num_pages, page_size, Hkv, D]; K and V must share them and have unit
    stride along D."""
    if k.ndim != 4 or v.ndim != 4 or k.shape != v.shape or k.dtype != v.dtype:
        raise ValueError("k and v must be 4-D views of the same shape and dtype")
    if k.strides != v.strides:
        raise ValueError("k and v must share strides")
    es = k.itemsize
    st = [s // es for s in k.strides]
    if st[3] != 1:
        raise ValueError("the head-dim stride must be 1")
    return st[0], st[1], st[2]


def _kv_kind(k: np.ndarray) -> int:
    if k.dtype == np.uint8:
        return 1
    if k.dtype == np.float16:
        return 0
    raise ValueError("k/v must be uint8 E4M3 codes or float16")


class Oracle:
    """ctypes view of one compiled copy of the oracle source."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        i32, i64, dbl, vp = ctypes.c_int, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
        lib.orc_f16_to_f64.argtypes = [ctypes.c_uint16]
        lib.orc_f16_to_f64.restype = dbl
        lib.orc_f64_to_f16.argtypes = [dbl]
        lib.orc_f64_to_f16.restype = ctypes.c_uint16
        lib.orc_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        lib.orc_e4m3_to_f64.restype = dbl
        lib.orc_decode.argtypes = [vp, vp, vp, i32, i64, i64, i64, vp, i64, vp,
                                   i32, i32, i32, i32, i32, i32, i32, dbl, dbl,
                                   vp, i32, vp, vp, vp, i32]
        lib.orc_decode.restype = i32
        lib.orc_sparse_prefill.argtypes = [vp, vp, vp, i32, i64, i64, i64, vp, i32, i32,
                                           vp, i32, vp, i32, i32, i32, i32, i32, dbl, dbl,
                                           vp, i32, vp, vp, vp, i32]
        lib.orc_sparse_prefill.restype = i32
        lib.orc_gather_rows.argtypes = [vp, i32, i64, i64, i64, vp, i64, vp,
                                        i32, i32, i32, i32, i32, i32, i32, dbl, vp, i32]
        lib.orc_gather_rows.restype = i32
        lib.orc_sparse_row_tokens.argtypes = [vp, i32, i32, vp, i32, ctypes.c_int32, i32, vp, i64]
        lib.orc_sparse_row_tokens.restype = i64
        lib.orc_select_blocks.argtypes = [vp, i64, i32, vp, i32, i32, i32, vp, vp, i32]
        lib.orc_select_blocks.restype = i32
        lib.orc_topk_topp_mask.argtypes = [vp, i64, i32, i32, i32, dbl, vp, i64, vp, i32]
        lib.orc_topk_topp_mask.restype = i32
        self.lib = lib
        self.path = path

    # -- number formats ---------------------------------------------------
    def f16_to_f64(self, bits: int) -> float:
        """binary16 bit pattern -> float."""
        return self.lib.orc_f16_to_f64(int(bits))

    def f64_to_f16(self, x: float) -> int:
        """float -> binary16 bit pattern, nearest-even."""
        return int(self.lib.orc_f64_to_f16(float(x)))

    def e4m3_to_f64(self, code: int) -> float:
        """E4M3FN code -> float."""
        return self.lib.orc_e4m3_to_f64(int(code))

    # -- attention ---------------------------------------------------------
    def decode(self, q, k, v, block_table, seq_lens, page_size, num_pages, max_seq_len,
               kv_scale, softmax_scale, pairs=None, want_f64=False, threads=None):
        """Paged GQA decode.  q float16 [B, Hq, D]; k, v 4-D views
        [pages, P, Hkv, D] (uint8 E4M3 codes or float16); block_table int32
        [B, >= ceil(max_seq_len / P)]; seq_lens int32 [B].  ``pairs``: optional
        int32 [n, 2] (b, h) subset.  Returns (out float16 [B, Hq, D],
        out_f64 or None, flags)."""
        q = np.ascontiguousarray(q, dtype=np.float16)
        B, Hq, D = q.shape
        Hkv = k.shape[2]
        ps, ts, hs = _kv_strides(k, v)
        bt = np.ascontiguousarray(block_table, dtype=np.int32).reshape(B, -1)
        sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
        out = np.zeros((B, Hq, D), dtype=np.float16)
        o64 = np.zeros((B, Hq, D), dtype=np.float64) if want_f64 else None
        pr = None if pairs is None else np.ascontiguousarray(pairs, dtype=np.int32).reshape(-1, 2)
        flags = ctypes.c_int(0)
        rc = self.lib.orc_decode(_ptr(q), k.ctypes.data, v.ctypes.data, _kv_kind(k), ps, ts, hs,
                                 _ptr(bt), bt.shape[1], _ptr(sl), B, Hq, Hkv, D, page_size,
                                 num_pages, max_seq_len, float(kv_scale), float(softmax_scale),
                                 _ptr(pr), 0 if pr is None else pr.shape[0],
                                 out.ctypes.data, _ptr(o64), ctypes.addressof(flags),
                                 threads or default_threads())
        if rc != 0:
            raise ValueError("oracle rejected the decode shapes")
        return out, o64, flags.value

    def sparse_prefill(self, q, k, v, block_table, num_pages, kv_len, sel_idx, q_pos,
                       page_size, softmax_scale, kv_scale=1.0, rows=None, want_f64=False,
                       threads=None):
        """Selected-sparse prefill over four-token blocks of one sequence.
        q float16 [R, Hq, D]; sel_idx int32 [R, n_sel]; q_pos int32 [R].
        ``rows``: optional int32 subset of row indices.
        Returns (out float16 [R, Hq, D], out_f64 or None, flags)."""
        q = np.ascontiguousarray(q, dtype=np.float16)
        R, Hq, D = q.shape
        Hkv = k.shape[2]
        ps, ts, hs = _kv_strides(k, v)
        bt = np.ascontiguousarray(block_table, dtype=np.int32).reshape(-1)
        sel = np.ascontiguousarray(sel_idx, dtype=np.int32)
        if sel.ndim != 2 or sel.shape[0] != R:
            raise ValueError("sel_idx must be [R, n_sel]")
        qp = np.ascontiguousarray(q_pos, dtype=np.int32)
        out = np.zeros((R, Hq, D), dtype=np.float16)
        o64 = np.zeros((R, Hq, D), dtype=np.float64) if want_f64 else None
        rw = None if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
        flags = ctypes.c_int(0)
        rc = self.lib.orc_sparse_prefill(_ptr(q), k.ctypes.data, v.ctypes.data, _kv_kind(k),
                                         ps, ts, hs, _ptr(bt), num_pages, kv_len, _ptr(sel),
                                         sel.shape[1], _ptr(qp), R, Hq, Hkv, D, page_size,
                                         float(kv_scale), float(softmax_scale),
                                         _ptr(rw), 0 if rw is None else rw.shape[0],
                                         out.ctypes.data, _ptr(o64), ctypes.addressof(flags),
                                         threads or default_threads())
        if rc != 0:
            raise ValueError("oracle rejected the sparse-prefill shapes")
        return out, o64, flags.value

    def sparse_row_tokens(self, block_table, num_pages, kv_len, sel_row, q_pos, page_size):
        """Logical tokens one prefill row attends to, in order (int64 array)."""
        bt = np.ascontiguousarray(block_table, dtype=np.int32).reshape(-1)
        sel = np.ascontiguousarray(sel_row, dtype=np.int32).reshape(-1)
        cap = 4 * sel.shape[0] + 4
        buf = np.empty(cap, dtype=np.int64)
        n = self.lib.orc_sparse_row_tokens(_ptr(bt), num_pages, kv_len, _ptr(sel), sel.shape[0],
                                           int(q_pos), page_size, buf.ctypes.data, cap)
        if n < 0:
            raise ValueError("token buffer too small")
        return buf[:n].copy()

    def select_blocks(self, scores, q_pos, kv_len, k, n_blocks=None, threads=None):
        """QSA block selection.  scores float32 [R, >= n_blocks] (row stride
        taken from the array); q_pos int32 [R].  Returns (sel int32 [R, k],
        flags)."""
        sc = np.asarray(scores, dtype=np.float32)
        if sc.ndim != 2 or sc.strides[1] != 4:
            raise ValueError("scores must be 2-D float32 with unit column stride")
        R = sc.shape[0]
        n_blocks = sc.shape[1] if n_blocks is None else int(n_blocks)
        qp = np.ascontiguousarray(q_pos, dtype=np.int32).reshape(R)
        sel = np.empty((R, int(k)), dtype=np.int32)
        flags = ctypes.c_int(0)
        rc = self.lib.orc_select_blocks(sc.ctypes.data, sc.strides[0] // 4, n_blocks, _ptr(qp), R,
                                        int(kv_len), int(k), sel.ctypes.data,
                                        ctypes.addressof(flags), threads or default_threads())
        if rc != 0:
            raise ValueError("oracle rejected the selection shapes" if rc == -1 else "out of memory")
        return sel, flags.value

    def topk_topp_mask(self, logits, k, p, threads=None):
        """Combined top-k/top-p masking.  logits float32 [B, V] (unit column
        stride).  Returns (masked float32 [B, V], margin float64 [B])."""
        x = np.asarray(logits, dtype=np.float32)
        if x.ndim != 2 or x.strides[1] != 4:
            raise ValueError("logits must be 2-D float32 with unit column stride")
        B, V = x.shape
        out = np.empty((B, V), dtype=np.float32)
        margin = np.empty(B, dtype=np.float64)
        rc = self.lib.orc_topk_topp_mask(x.ctypes.data, x.strides[0] // 4, B, V, int(k),
                                         float(np.float32(p)), out.ctypes.data, V,
                                         margin.ctypes.data, threads or default_threads())
        if rc != 0:
            raise ValueError({-1: "bad arguments", -2: "out of memory",
                              -3: "NaN or +inf logit"}.get(rc, str(rc)))
        return out, margin

    def gather_rows(self, cache, block_table, seq_lens, page_size, num_pages, max_seq_len,
                    kv_scale=1.0, T=None, threads=None):
        """Gathered, dequantised rows [B, T, Hkv, D] float32 of one K or V pool
        (zeros past each sequence's length and on invalid pages)."""
        ps, ts, hs = _kv_strides(cache, cache)
        sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
        B = sl.shape[0]
        bt = np.ascontiguousarray(block_table, dtype=np.int32).reshape(B, -1)
        T = max_seq_len if T is None else T
        Hkv, D = cache.shape[2], cache.shape[3]
        out = np.empty((B, T, Hkv, D), dtype=np.float32)
        rc = self.lib.orc_gather_rows(cache.ctypes.data, _kv_kind(cache), ps, ts, hs, _ptr(bt),
                                      bt.shape[1], _ptr(sl), B, T, Hkv, D, page_size, num_pages,
                                      max_seq_len, float(kv_scale), out.ctypes.data,
                                      threads or default_threads())
        if rc != 0:
            raise ValueError("oracle rejected the gather shapes")
        return out


_default = None
_lock = threading.Lock()


def default() -> Oracle:
    """The oracle compiled from the committed source."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def decode(*args, **kwargs):
    return default().decode(*args, **kwargs)


def sparse_prefill(*args, **kwargs):
    return default().sparse_prefill(*args, **kwargs)


def sparse_row_tokens(*args, **kwargs):
    return default().sparse_row_tokens(*args, **kwargs)


def gather_rows(*args, **kwargs):
    return default().gather_rows(*args, **kwargs)


def select_blocks(*args, **kwargs):
    return default().select_blocks(*args, **kwargs)


def topk_topp_mask(*args, **kwargs):
    return default().topk_topp_mask(*args, **kwargs)
