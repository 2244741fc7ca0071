"""The C ABI on the host (no GPU needed): the library builds and loads, exports
every function include/paged_gqa.h declares, and rejects bad arguments with
its status codes before launching anything.  Pointers passed here are fake
non-NULL addresses; every case fails a host check that runs before any CUDA
call, so nothing is ever dereferenced."""
import ctypes
import os
import re

import pytest

import oracle
import fp8_kv_cache_gb300 as P
from fp8_kv_cache_gb300 import build as B

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "paged_gqa.h")


@pytest.fixture(scope="module")
def L():
    B.build()
    return P.lib()


def _header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(paged_gqa_\w+)\s*\(", text)))


def test_header_declares_entry_points():
    names = _header_functions()
    for n in ("paged_gqa_decode", "paged_gqa_sparse_prefill", "paged_gqa_decode_workspace_size",
              "paged_gqa_gather_dequant", "paged_gqa_sparse_prefill_tokens",
              "paged_gqa_select_blocks", "paged_gqa_topk_topp_mask", "paged_gqa_status_string",
              "paged_gqa_version"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for name in _header_functions():
        assert hasattr(L, name), f"{name} is declared but not exported"


def test_version_and_status_strings(L):
    text = open(HEADER).read()
    ver = int(re.search(r"#define PAGED_GQA_VERSION (\d+)", text).group(1))
    assert P.paged_gqa_version() == ver
    for st in range(-6, 1):
        assert P.paged_gqa_status_string(st) not in ("", "unknown status")
    assert P.paged_gqa_status_string(-99) == "unknown status"


def test_flag_bits_match_header_and_oracle():
    text = open(HEADER).read()
    bits = {m.group(1): int(m.group(2))
            for m in re.finditer(r"#define PAGED_GQA_FLAG_(\w+)\s+(\d+)", text)}
    assert bits == {"BAD_PAGE": 1, "SEQ_CLAMPED": 2, "EMPTY_ROW": 4, "QPOS_CLAMPED": 8,
                    "BAD_SEL": 16, "SCORES_SHORT": 32, "BAD_LOGIT": 64, "TIMEOUT": 128}
    assert (oracle.FLAG_BAD_PAGE, oracle.FLAG_SEQ_CLAMPED, oracle.FLAG_EMPTY_ROW,
            oracle.FLAG_QPOS_CLAMPED, oracle.FLAG_BAD_SEL) == (1, 2, 4, 8, 16)
    assert (P.FLAG_BAD_PAGE, P.FLAG_SEQ_CLAMPED, P.FLAG_EMPTY_ROW, P.FLAG_QPOS_CLAMPED,
            P.FLAG_BAD_SEL) == (1, 2, 4, 8, 16)
    assert oracle.FLAG_SCORES_SHORT == P.FLAG_SCORES_SHORT == 32
    assert P.FLAG_BAD_LOGIT == 64
    assert P.FLAG_TIMEOUT == 128


A = 0x10000   # a fake, 16-byte aligned, non-NULL address (never dereferenced)


def _no_device():
    try:
        import torch
        return not torch.cuda.is_available()
    except Exception:  # pragma: no cover
        return True


# Calls with fake addresses only run where no CUDA device exists, so that a
# case that wrongly passed validation could never launch a kernel on a GPU.
host_only = pytest.mark.skipif(not _no_device(), reason="fake-pointer calls run only without a GPU")


def _decode(L, **kw):
    args = dict(q=A, k=A, v=A, layout=(16 * 4 * 256, 4 * 256, 256), dtype=1, bt=A, bt_stride=1024,
                sl=A, B=2, Hq=24, Hkv=4, D=256, P=16, num_pages=100, max_seq_len=16384,
                kv_scale=1.0, s=0.0625, out=A, ws=None)
    args.update(kw)
    ws = args["ws"]
    return L.paged_gqa_decode(args["q"], args["k"], args["v"], P.KVLayout(*args["layout"]),
                              args["dtype"], args["bt"], args["bt_stride"], args["sl"], args["B"],
                              args["Hq"], args["Hkv"], args["D"], args["P"], args["num_pages"],
                              args["max_seq_len"], args["kv_scale"], args["s"], args["out"],
                              None if ws is None else ctypes.byref(ws), None)


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), -1), (dict(k=None), -1), (dict(v=None), -1), (dict(bt=None), -1),
    (dict(sl=None), -1), (dict(out=None), -1),
    (dict(q=A + 8), -2), (dict(out=A + 4), -2), (dict(k=A + 1), -2),
    (dict(layout=(16 * 4 * 256, 4 * 256, 200)), -2),          # 200 B head stride (E4M3)
    (dict(dtype=0, layout=(16 * 4 * 256, 4 * 256, 260)), -2),  # 520 B head stride (FP16)
    (dict(B=-1), -3), (dict(Hq=0), -3), (dict(Hkv=0), -3), (dict(Hq=25), -3),
    (dict(P=0), -3), (dict(num_pages=0), -3), (dict(max_seq_len=-1), -3),
    (dict(bt_stride=100), -3), (dict(layout=(-1, 256, 256)), -3),
    (dict(B=(1 << 27), Hq=24, Hkv=4), -3),                   # B * Hq beyond one launch
    (dict(D=128), -4), (dict(Hq=36, Hkv=4), -4), (dict(dtype=2), -4),
])
@host_only
def test_decode_rejects_bad_arguments(L, kw, status):
    assert _decode(L, **kw) == status


@host_only
def test_decode_batch_zero_is_a_no_op(L):
    assert _decode(L, B=0) == 0


@host_only
def test_decode_rejects_misaligned_workspace(L):
    ws = P.Workspace()
    ws.ptr = A + 64
    ws.bytes = 1 << 30
    assert _decode(L, ws=ws) == -5


def _prefill(L, **kw):
    args = dict(q=A, k=A, v=A, layout=(16 * 512, 512, 256), dtype=0, bt=A, num_pages=2048,
                kv_len=32768, sel=A, n_sel=512, qp=A, R=4096, Hq=6, Hkv=1, D=256, P=16,
                kv_scale=1.0, s=0.0625, out=A, err=None)
    args.update(kw)
    return L.paged_gqa_sparse_prefill(args["q"], args["k"], args["v"], P.KVLayout(*args["layout"]),
                                      args["dtype"], args["bt"], args["num_pages"], args["kv_len"],
                                      args["sel"], args["n_sel"], args["qp"], args["R"], args["Hq"],
                                      args["Hkv"], args["D"], args["P"], args["kv_scale"], args["s"],
                                      args["out"], args["err"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), -1), (dict(sel=None), -1), (dict(qp=None), -1), (dict(out=None), -1),
    (dict(bt=None), -1), (dict(k=None), -1),
    (dict(q=A + 2), -2), (dict(out=A + 8), -2), (dict(layout=(16 * 512, 516, 256)), -2),
    (dict(R=-1), -3), (dict(n_sel=-1), -3), (dict(P=6), -3), (dict(P=2), -3), (dict(kv_len=-1), -3),
    (dict(num_pages=0), -3), (dict(Hq=7, Hkv=2), -3),
    (dict(D=64), -4), (dict(Hq=12, Hkv=1), -4), (dict(dtype=7), -4),
])
@host_only
def test_prefill_rejects_bad_arguments(L, kw, status):
    assert _prefill(L, **kw) == status


def _prefill_route(L, route, rows, **kw):
    args = dict(q=A, k=A, v=A, layout=(16 * 512, 512, 256), dtype=0, bt=A, num_pages=2048,
                kv_len=32768, sel=A, n_sel=512, qp=A, R=4096, Hq=6, Hkv=1, D=256, P=16,
                kv_scale=1.0, s=0.0625, out=A, err=None)
    args.update(kw)
    return L.paged_gqa_sparse_prefill_route(
        args["q"], args["k"], args["v"], P.KVLayout(*args["layout"]), args["dtype"], args["bt"],
        args["num_pages"], args["kv_len"], args["sel"], args["n_sel"], args["qp"], args["R"],
        args["Hq"], args["Hkv"], args["D"], args["P"], args["kv_scale"], args["s"], args["out"],
        args["err"], None, route, rows)


@pytest.mark.parametrize("route,rows,kw,status", [
    (3, 0, {}, -3), (-1, 0, {}, -3), (2, -1, {}, -3),
    (2, 22, {}, -3),                               # 22 rows x 6 heads > 128 slots
    (2, 0, dict(kv_len=131076, num_pages=8193), -4),   # beyond the union bitmap
    (1, 0, dict(q=None), -1), (2, 0, dict(D=64), -4),
])
@host_only
def test_prefill_route_rejects_bad_arguments(L, route, rows, kw, status):
    assert _prefill_route(L, route, rows, **kw) == status


@pytest.mark.parametrize("args,status", [
    ((0, 6, 1, 0), -3), ((10, 7, 2, 0), -3), ((10, 6, 1, -1), -3), ((10, 6, 1, 22), -3),
    ((10, 12, 1, 0), -4),
])
def test_group_rows_rejects_bad_arguments(L, args, status):
    assert L.paged_gqa_sparse_prefill_group_rows(*args) == status


@host_only
def test_prefill_empty_cases_are_no_ops(L):
    assert _prefill(L, R=0) == 0
    # n_sel == 0 needs no selection pointer; R == 0 keeps it a host-only call
    assert _prefill(L, n_sel=0, sel=None, R=0) == 0


@host_only
def test_inspection_entry_points_validate(L):
    lay = P.KVLayout(16 * 4 * 256, 4 * 256, 256)
    assert L.paged_gqa_gather_dequant(None, lay, 1, A, 64, A, 2, 16, 4, 256, 16, 8, 16, 1.0, A,
                                      None) == -1
    assert L.paged_gqa_gather_dequant(A, lay, 1, A, 64, A, 2, 16, 4, 128, 16, 8, 16, 1.0, A,
                                      None) == -4
    assert L.paged_gqa_gather_dequant(A, lay, 1, A, 64, A, 2, 16, 4, 256, 16, 8, 16, 1.0, A + 4,
                                      None) == -2
    assert L.paged_gqa_sparse_prefill_tokens(A, 8, 64, A, 4, A, 3, 6, A, None) == -3
    assert L.paged_gqa_sparse_prefill_tokens(None, 8, 64, A, 4, A, 3, 16, A, None) == -1
    assert L.paged_gqa_sparse_prefill_tokens(A, 8, 64, A, 4, A, 0, 16, A, None) == 0


@host_only
def test_select_blocks_validates(L):
    # (scores, score_stride, n_blocks, q_pos, R, kv_len, k, sel_out, err_flag, stream)
    assert L.paged_gqa_select_blocks(A, 8, 16, A, 4, 64, 4, A, None, None) == -3   # stride < n
    assert L.paged_gqa_select_blocks(A, 16, 16, A, -1, 64, 4, A, None, None) == -3
    assert L.paged_gqa_select_blocks(A, 16, 16, A, 4, 64, -2, A, None, None) == -3
    assert L.paged_gqa_select_blocks(None, 16, 16, A, 4, 64, 4, A, None, None) == -1
    assert L.paged_gqa_select_blocks(A, 16, 16, None, 4, 64, 4, A, None, None) == -1
    assert L.paged_gqa_select_blocks(A, 16, 16, A, 4, 64, 4, None, None, None) == -1
    assert L.paged_gqa_select_blocks(A, 16, 16, A, 0, 64, 4, A, None, None) == 0
    assert L.paged_gqa_select_blocks(A, 16, 16, A, 4, 64, 0, None, None, None) == 0


@host_only
def test_topk_topp_mask_validates(L):
    # (logits, logits_stride, out, out_stride, B, V, k, p, err_flag, stream)
    ok = (A, 1000, A + 4096, 1000, 4, 1000, 20, 0.95)
    assert L.paged_gqa_topk_topp_mask(None, *ok[1:], None, None) == -1
    assert L.paged_gqa_topk_topp_mask(A, 1000, None, 1000, 4, 1000, 20, 0.95, None, None) == -1
    assert L.paged_gqa_topk_topp_mask(A, 999, A + 4096, 1000, 4, 1000, 20, 0.95, None, None) == -3
    assert L.paged_gqa_topk_topp_mask(A, 1000, A + 4096, 1000, -1, 1000, 20, 0.95, None, None) == -3
    assert L.paged_gqa_topk_topp_mask(A, 1000, A + 4096, 1000, 4, 1000, 0, 0.95, None, None) == -3
    assert L.paged_gqa_topk_topp_mask(A, 1000, A + 4096, 1000, 4, 1000, 129, 0.95, None, None) == -4
    assert L.paged_gqa_topk_topp_mask(A, 400000, A, 400000, 4, 400000, 20, 0.95, None, None) == -4
    for p in (0.0, -0.5, 1.5, float("nan")):
        assert L.paged_gqa_topk_topp_mask(A, 1000, A + 4096, 1000, 4, 1000, 20, p, None, None) == -3
    assert L.paged_gqa_topk_topp_mask(A, 1000, A, 1024, 4, 1000, 20, 0.95, None, None) == -3
    assert L.paged_gqa_topk_topp_mask(A, 1000, A + 4096, 1000, (1 << 27) + 1, 1000, 20, 0.95,
                                      None, None) == -3
    assert L.paged_gqa_topk_topp_mask(A, 1000, A + 4096, 1000, 0, 1000, 20, 0.95, None, None) == 0


def test_workspace_size_for_forced_splits(L):
    n1 = P.paged_gqa_decode_workspace_size_splits(16, 24, 4, 256, 1)
    n2 = P.paged_gqa_decode_workspace_size_splits(16, 24, 4, 256, 2)
    assert n2 - n1 == (2 * 8 + 8 * 256) * 4     # one more partial slot
    assert P.paged_gqa_decode_workspace_size_splits(16, 24, 4, 128, 2) == 0
    assert P.paged_gqa_decode_workspace_size_splits(16, 24, 4, 256, 0) == 0


def test_binding_fails_loudly_without_library(monkeypatch):
    monkeypatch.setattr(P, "_lib", None)
    monkeypatch.setattr(P, "library_path", "/nonexistent/libpaged_gqa.so")
    with pytest.raises(RuntimeError, match="no fallback"):
        P.lib()


def test_auto_route_follows_the_documented_rule(L):
    """PAGED_GQA_PREFILL_AUTO, with C = R * Hkv: FP16 grouped when
    64 n_sel >= kv_len, or C >= 1024 and 2048 n_sel >= kv_len; E4M3 grouped
    when C >= 1024 and 36 n_sel >= kv_len; always only where the grouped
    route supports the shape."""
    f = L.paged_gqa_sparse_prefill_auto_route
    assert f(4096, 6, 1, 32768, 16, 0) == 2            # FP16, C >= 1024, 2048 * 16 = 32768
    assert f(4096, 6, 1, 32768, 15, 0) == 1
    assert f(1024, 6, 1, 32768, 16, 0) == 2
    assert f(1023, 6, 1, 32768, 16, 0) == 1            # C < 1024: the dense rule only
    assert f(512, 12, 2, 32768, 16, 0) == 2            # C = 1024 over two KV heads
    assert f(1, 6, 1, 32768, 512, 0) == 2              # 64 * 512 = 32768
    assert f(512, 6, 1, 32768, 511, 0) == 1
    assert f(4096, 6, 1, 32768, 911, 1) == 2           # E4M3, 36 * 911 >= 32768
    assert f(4096, 6, 1, 32768, 910, 1) == 1
    assert f(1023, 6, 1, 32768, 4096, 1) == 1          # E4M3 needs C >= 1024
    assert f(4096, 6, 1, 131076, 4096, 0) == 1         # beyond the grouped route's bitmap
    assert f(-1, 6, 1, 32768, 512, 0) == -3
    assert f(10, 7, 2, 32768, 512, 0) == -3
    assert f(10, 12, 1, 32768, 512, 0) == -4           # 12 query heads per KV head
    assert f(10, 6, 1, 32768, 512, 5) == -4            # unknown KV dtype


@host_only
def test_gather_probe_and_stall_hook_validate(L):
    lay = P.KVLayout(16 * 512, 512, 256)
    # (k, v, layout, dtype, bt, num_pages, kv_len, sel, n_sel, q_pos, R, Hkv, D, page, out, stream)
    ok = [A, A, lay, 0, A, 2048, 32768, A, 512, A, 4096, 1, 256, 16, A, None]

    def probe(**kw):
        a = list(ok)
        names = ["k", "v", "lay", "dtype", "bt", "num_pages", "kv_len", "sel", "n_sel", "qp", "R",
                 "Hkv", "D", "P", "out", "stream"]
        for k_, v_ in kw.items():
            a[names.index(k_)] = v_
        return L.paged_gqa_sparse_gather_probe(*a)

    assert probe(k=None) == -1 and probe(out=None) == -1 and probe(sel=None) == -1
    assert probe(out=A + 2) == -2 and probe(k=A + 8) == -2
    assert probe(R=-1) == -3 and probe(P=6) == -3 and probe(Hkv=0) == -3
    assert probe(D=128) == -4 and probe(dtype=3) == -4
    assert probe(R=0) == 0
    # the stall hook: its own limits, then the route's validation
    args = [A, A, A, lay, 0, A, 2048, 32768, A, 512, A, 4096, 6, 1, 256, 16, 1.0, 0.0625, A,
            None, None]
    stall = L.paged_gqa_debug_grouped_prefill_stall
    assert stall(*args, -1, 0) == -3
    assert stall(*args, (1 << 30) + 1, 0) == -3
    assert stall(*args, 1000, -2) == -3
    bad_q = list(args)
    bad_q[0] = None
    assert stall(*bad_q, 1000, 3) == -1
    zero_r = list(args)
    zero_r[11] = 0
    assert stall(*zero_r, 1000, 3) == 0
