"""Independent numpy references used to pin the oracle (test-side only).

These never call the oracle's C code: values are decoded with library
routines (numpy's float16 view, torch's float8_e4m3fn view), pages are
gathered with numpy fancy indexing, and attention is the textbook dense
softmax(s * q K^T) V in float64 via numpy.
"""
from __future__ import annotations

import numpy as np


def lib_decode(view: np.ndarray, kv_scale: float) -> np.ndarray:
    """Values of a K or V view as float64, decoded by library routines."""
    if view.dtype == np.float16:
        return view.astype(np.float64)
    import torch
    t = torch.from_numpy(np.ascontiguousarray(view)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy() * float(np.float32(kv_scale))


def unroll(view_vals: np.ndarray, bt_row: np.ndarray, tokens: np.ndarray, page_size: int,
           num_pages: int):
    """Rows of the listed logical tokens (invalid pages dropped).
    view_vals [pages, P, Hkv, D] -> [n, Hkv, D], and the kept tokens."""
    tokens = np.asarray(tokens, dtype=np.int64)
    pages = bt_row[tokens // page_size].astype(np.int64)
    keep = (pages >= 0) & (pages < num_pages)
    return view_vals[pages[keep], tokens[keep] % page_size], tokens[keep]


def softmax_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    """Dense softmax(scale * q K^T) V for one query vector (float64)."""
    if K.shape[0] == 0:
        return np.zeros(V.shape[-1])
    x = scale * (K @ q)
    w = np.exp(x - x.max())
    w /= w.sum()
    return w @ V


def dense_decode(case, max_seq_len=None) -> np.ndarray:
    """[B, Hq, D] float64 decode output of a DecodeCase via the dense route."""
    Kd = lib_decode(case.k, case.kv_scale if case.kv_dtype == "e4m3" else 1.0)
    Vd = lib_decode(case.v, case.kv_scale if case.kv_dtype == "e4m3" else 1.0)
    msl = case.max_seq_len if max_seq_len is None else max_seq_len
    B, Hq, D = case.q.shape
    G = Hq // case.Hkv
    out = np.zeros((B, Hq, D))
    for b in range(B):
        L = int(min(case.seq_lens[b], msl))
        if L <= 0:
            continue
        Kb, _ = unroll(Kd, case.block_table[b], np.arange(L), case.page_size, case.num_pages)
        Vb, _ = unroll(Vd, case.block_table[b], np.arange(L), case.page_size, case.num_pages)
        for h in range(Hq):
            j = h // G
            out[b, h] = softmax_attention(case.q[b, h].astype(np.float64), Kb[:, j], Vb[:, j],
                                          case.softmax_scale)
    return out


def prefill_tokens(sel_row: np.ndarray, q_pos: int, kv_len: int) -> np.ndarray:
    """Token list of one prefill row written from the page's description:
    the selected four-token blocks before the row's own block, then its
    causal partial block up to and including the row's position."""
    if q_pos < 0:
        return np.zeros(0, dtype=np.int64)
    p = min(int(q_pos), kv_len - 1)
    own = p // 4
    blocks = [int(b) for b in sel_row if 0 <= b < own]
    toks = [4 * b + i for b in blocks for i in range(4)]
    toks += list(range(4 * own, p + 1))
    return np.asarray(toks, dtype=np.int64)


def dense_prefill_row(case, r: int) -> np.ndarray:
    """[Hq, D] float64 output of one prefill row via the dense route."""
    Kd = lib_decode(case.k, case.kv_scale if case.kv_dtype == "e4m3" else 1.0)
    Vd = lib_decode(case.v, case.kv_scale if case.kv_dtype == "e4m3" else 1.0)
    toks = prefill_tokens(case.sel_idx[r], int(case.q_pos[r]), case.kv_len)
    Kr, _ = unroll(Kd, case.block_table, toks, case.page_size, case.num_pages)
    Vr, _ = unroll(Vd, case.block_table, toks, case.page_size, case.num_pages)
    G = case.Hq // case.Hkv
    out = np.zeros((case.Hq, case.D))
    for h in range(case.Hq):
        out[h] = softmax_attention(case.q[r, h].astype(np.float64), Kr[:, h // G], Vr[:, h // G],
                                   case.softmax_scale)
    return out


def lse_partial(q, K, V, scale):
    """(m, l, o_unnormalised) of softmax attention over one token chunk."""
    x = scale * (K @ q)
    m = x.max()
    w = np.exp(x - m)
    return m, w.sum(), w @ V


def lse_merge(parts):
    """Merge (m, l, o) partials: M = max m_i, o = sum e^{m_i-M} o_i / sum e^{m_i-M} l_i."""
    M = max(p[0] for p in parts)
    num = sum(np.exp(m - M) * o for m, _, o in parts)
    den = sum(np.exp(m - M) * l for m, l, _ in parts)
    return num / den
