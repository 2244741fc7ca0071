"""Helpers of the GPU parity tests: device copies of generated cases, calls
through the binding, and the tolerance check against the oracle.

Tolerances: the outputs must match the oracle's FP16-rounded results within
max |err| <= 2e-3 and relative L2 <= 5e-4 (the accuracy bar set for this
path); gathers, dequantised values and token lists must match bit for bit.
Where |oracle| >= 4 one FP16 step (2^-8 and up) is itself wider than 2e-3, so
two correct FP16 roundings of nearly equal values may differ by one step; the
per-element bound there is one FP16 ULP of the oracle's value.  Such elements
only occur in short-context edge cases (a few tokens of N(0,1)*2 values), and
the check reports how many there were.
"""
from __future__ import annotations

import numpy as np

MAX_ABS = 2e-3
REL_L2 = 5e-4


def torch():
    import torch as t
    return t


def dev_kv(case, device="cuda"):
    """(backing buffer, k view, v view) on the device with the case's strides."""
    t = torch()
    buf = t.from_numpy(np.ascontiguousarray(case.kv)).to(device)
    item = case.kv.itemsize

    def view(a):
        off = (a.ctypes.data - case.kv.ctypes.data) // item
        return t.as_strided(buf, size=a.shape, stride=[s // item for s in a.strides],
                            storage_offset=off)
    return buf, view(case.k), view(case.v)


def dev(a, device="cuda"):
    return torch().from_numpy(np.ascontiguousarray(a)).to(device)


def run_decode(case, kv=None, **kw):
    """The library's decode on a DecodeCase; returns (out numpy float16, flags)."""
    import fp8_kv_cache_gb300 as P
    t = torch()
    if kv is None:
        kv = dev_kv(case)
    _, k, v = kv
    err = t.zeros(1, dtype=t.int32, device="cuda")
    out = P.paged_gqa_decode(dev(case.q), k, v, dev(case.block_table), dev(case.seq_lens),
                             case.page_size, case.kv_scale, case.softmax_scale,
                             max_seq_len=kw.pop("max_seq_len", case.max_seq_len),
                             num_pages=kw.pop("num_pages", case.num_pages), err_flag=err, **kw)
    t.cuda.synchronize()
    return out.cpu().numpy(), int(err.item())


def run_prefill(case, kv=None, **kw):
    import fp8_kv_cache_gb300 as P
    t = torch()
    if kv is None:
        kv = dev_kv(case)
    _, k, v = kv
    err = t.zeros(1, dtype=t.int32, device="cuda")
    route, rows = kw.pop("route", None), kw.pop("rows_per_group", 0)
    args = (dev(case.q), k, v, dev(case.block_table), case.kv_len, dev(case.sel_idx),
            dev(kw.pop("q_pos", case.q_pos)), case.page_size, case.softmax_scale, case.kv_scale)
    num_pages = kw.pop("num_pages", case.num_pages)
    if route is None:
        out = P.paged_gqa_sparse_prefill(*args, num_pages=num_pages, err_flag=err, **kw)
    else:
        out = P.paged_gqa_sparse_prefill_route(*args, route=route, rows_per_group=rows,
                                               num_pages=num_pages, err_flag=err, **kw)
    t.cuda.synchronize()
    return out.cpu().numpy(), int(err.item())


def oracle_decode(case, pairs=None, **kw):
    import oracle
    return oracle.decode(case.q, case.k, case.v, case.block_table, case.seq_lens, case.page_size,
                         kw.pop("num_pages", case.num_pages),
                         kw.pop("max_seq_len", case.max_seq_len), case.kv_scale,
                         case.softmax_scale, pairs=pairs, **kw)


def oracle_prefill(case, rows=None, **kw):
    import oracle
    return oracle.sparse_prefill(case.q, case.k, case.v, case.block_table,
                                 kw.pop("num_pages", case.num_pages), case.kv_len, case.sel_idx,
                                 kw.pop("q_pos", case.q_pos), case.page_size, case.softmax_scale,
                                 case.kv_scale, rows=rows, **kw)


def ulp16(x):
    """Spacing of the FP16 grid at |x| (normal range; 2^-24 below it)."""
    ax = np.maximum(np.abs(np.asarray(x, dtype=np.float64)), 2.0 ** -14)
    return 2.0 ** (np.floor(np.log2(ax)) - 10)


def assert_close(got, want, what="", max_abs=MAX_ABS, rel_l2=REL_L2):
    """Element-wise comparison of FP16 outputs (as float64): |err| <=
    max(max_abs, 1 FP16 ULP of the oracle value) and rel L2 <= rel_l2.
    Returns (max abs err, rel L2, elements that needed the ULP allowance)."""
    a = np.asarray(got, dtype=np.float64)
    b = np.asarray(want, dtype=np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} != {b.shape}"
    assert np.all(np.isfinite(a)), f"{what}: non-finite output"
    diff = np.abs(a - b)
    worst = float(diff.max()) if diff.size else 0.0
    nb = float(np.linalg.norm(b))
    rl2 = float(np.linalg.norm(a - b)) / nb if nb > 0 else float(np.linalg.norm(a - b))
    bound = np.maximum(max_abs, ulp16(b))
    bad = diff > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} elements beyond max(2e-3, 1 ulp); "
                           f"worst {worst:.3e}")
    wide = int((diff > max_abs).sum())
    if wide:
        print(f"[tolerance] {what}: {wide} element(s) with |oracle| >= 4 differ by one FP16 "
              f"ULP (<= {float(ulp16(b[diff > max_abs]).max()):.3e})")
    assert rl2 <= rel_l2, f"{what}: rel L2 {rl2:.3e} > {rel_l2:.1e}"
    return worst, rl2, wide


def sample_pairs(B, Hq, per_seq=2, seed=0):
    """(b, h) pairs: every sequence, ``per_seq`` heads each, covering all groups."""
    rng = np.random.default_rng(seed)
    pairs = []
    for b in range(B):
        for h in rng.choice(Hq, size=min(per_seq, Hq), replace=False):
            pairs.append((b, int(h)))
    return np.asarray(pairs, dtype=np.int32)
