"""paged_gqa_decode_noalloc: the decode entry point for callers that cannot
allocate device memory (its split scratch is a static device array inside the
library).  Two calls in a row through the C ABI, each with different inputs,
must match the FP64 oracle within the parity tolerance and the regular
paged_gqa_decode (with a caller-allocated workspace and the same automatic
split) bit for bit; a batch above 512 (where the merge kernel reads the tile
prefix the split kernel leaves in the scratch header) goes through the Python
wrapper.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest

import fp8_kv_cache_gb300 as P
from fp8_kv_cache_gb300 import workloads as W
from tests import gpu_util as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _noalloc_via_c_abi(case, kv):
    """Direct ctypes call of the extern "C" symbol (no Python wrapper)."""
    import torch
    _, k, v = kv
    q, bt, sl = U.dev(case.q), U.dev(case.block_table), U.dev(case.seq_lens)
    out = torch.full_like(q, float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    lay = P.KVLayout(k.stride(0), k.stride(1), k.stride(2))
    st = P.lib().paged_gqa_decode_noalloc(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
        ctypes.c_void_p(v.data_ptr()), lay, P.KV_E4M3 if case.kv_dtype == "e4m3" else P.KV_FP16,
        ctypes.c_void_p(bt.data_ptr()), bt.stride(0), ctypes.c_void_p(sl.data_ptr()),
        case.B, case.Hq, case.Hkv, case.D, case.page_size, case.num_pages, case.max_seq_len,
        case.kv_scale, case.softmax_scale, ctypes.c_void_p(out.data_ptr()),
        ctypes.c_void_p(err.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, P.paged_gqa_status_string(st)
    torch.cuda.synchronize()
    return out.cpu().numpy(), int(err.item())


def _check(case, got, flags, kv):
    want, _, oflags = U.oracle_decode(case)
    U.assert_close(got, want, f"{case.name}: noalloc vs oracle")
    ref, ref_flags = U.run_decode(case, kv=kv)     # workspace route, same automatic split
    np.testing.assert_array_equal(got.view(np.uint16), ref.view(np.uint16),
                                  err_msg=f"{case.name}: noalloc vs workspace entry point")
    assert flags == ref_flags == oflags


def test_two_calls_in_a_row_match_the_oracle_and_the_workspace_entry_point():
    first = W.decode_case("noalloc_a", B=8, Hq=24, Hkv=4, seq_lens=[1024, 5, 700, 33, 1024,
                                                                     300, 17, 999],
                          kv_dtype="e4m3", seed=301)
    second = W.decode_case("noalloc_b", B=3, Hq=12, Hkv=2, seq_lens=[4000, 64, 1],
                           kv_dtype="fp16", seed=302)
    for case in (first, second):
        kv = U.dev_kv(case)
        got, flags = _noalloc_via_c_abi(case, kv)
        _check(case, got, flags, kv)


def test_batch_above_512_through_the_python_wrapper():
    """B = 600 > 512: the split kernel writes the per-sequence tile prefix and
    the split count into the scratch header and the merge kernel reads them;
    short ragged lengths (with empty rows) keep the scratch within 16 MiB."""
    import torch
    rng = np.random.default_rng(303)
    lens = rng.integers(-1, 120, size=600).astype(np.int32)
    case = W.decode_case("noalloc_b600", B=600, Hq=6, Hkv=1, seq_lens=lens, kv_dtype="e4m3",
                         seed=303, max_seq_len=128)
    kv = U.dev_kv(case)
    _, k, v = kv
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(2):                                   # twice: the scratch keeps old contents
        out = P.paged_gqa_decode_noalloc(U.dev(case.q), k, v, U.dev(case.block_table),
                                         U.dev(case.seq_lens), case.page_size, case.kv_scale,
                                         case.softmax_scale, max_seq_len=case.max_seq_len,
                                         num_pages=case.num_pages, err_flag=err)
        torch.cuda.synchronize()
        _check(case, out.cpu().numpy(), int(err.item()), kv)
        err.zero_()


def test_shapes_beyond_the_static_scratch_are_refused():
    """Every buffer is sized for the shape (zero lengths, a zero block table,
    a real KV pool), so even a call that got past the size check could only
    write zero rows inside its own output."""
    import torch
    B, Hq, Hkv, max_len, page = 3000, 64, 8, 1024, 16     # far more partial slots than 16 MiB
    need = P.paged_gqa_decode_workspace_size(B, Hq, Hkv, 256, max_len)
    assert need > 16 << 20
    num_pages = 8
    q = torch.zeros((B, Hq, 256), dtype=torch.float16, device="cuda")
    out = torch.full((B, Hq, 256), 3.0, dtype=torch.float16, device="cuda")
    sl = torch.zeros(B, dtype=torch.int32, device="cuda")
    bt = torch.zeros((B, max_len // page), dtype=torch.int32, device="cuda")
    kv = torch.zeros((num_pages, page, Hkv, 256), dtype=torch.float16, device="cuda")
    with pytest.raises(P.PagedGQAError) as ei:
        P.paged_gqa_decode_noalloc(q, kv, kv, bt, sl, page, 1.0, 0.0625, out,
                                   max_seq_len=max_len, num_pages=num_pages)
    assert ei.value.status == -5                         # PAGED_GQA_ERR_WORKSPACE, nothing launched
    torch.cuda.synchronize()
    assert bool((out == 3.0).all())
