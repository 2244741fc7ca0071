"""paged_gqa_decode_noalloc: the decode entry point for callers that cannot
allocate device memory (its split scratch is a static device array inside the
library).  Two calls in a row through the C ABI, each with different inputs,
must match the regular paged_gqa_decode (with a caller-allocated workspace)
within the parity tolerance.  This file is collected last on purpose."""
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


def test_two_calls_in_a_row_match_the_workspace_entry_point():
    first = W.decode_case("noalloc_a", B=8, Hq=24, Hkv=4, seq_lens=[1024, 5, 700, 33, 1024,
                                                                     300, 17, 999],
                          kv_dtype="e4m3", seed=301)
    second = W.decode_case("noalloc_b", B=3, Hq=12, Hkv=2, seq_lens=[4000, 64, 1],
                           kv_dtype="fp16", seed=302)
    for case in (first, second):
        kv = U.dev_kv(case)
        got, flags = _noalloc_via_c_abi(case, kv)
        ref, ref_flags = U.run_decode(case, kv=kv)
        U.assert_close(got, ref, f"{case.name}: noalloc vs workspace")
        assert flags == ref_flags == 0


def test_shapes_beyond_the_static_scratch_are_refused():
    import torch
    B, Hq, Hkv = 4096, 64, 8            # far more partial slots than 16 MiB holds
    need = P.paged_gqa_decode_workspace_size(B, Hq, Hkv, 256, 1024)
    assert need > 16 << 20
    x = torch.zeros(16, dtype=torch.float16, device="cuda")
    lay = P.KVLayout(16 * Hkv * 256, Hkv * 256, 256)
    ptr = ctypes.c_void_p(x.data_ptr())
    st = P.lib().paged_gqa_decode_noalloc(ptr, ptr, ptr, lay, P.KV_FP16, ptr, 64, ptr, B, Hq, Hkv,
                                          256, 16, 8, 1024, 1.0, 0.0625, ptr, None, None)
    assert st == -5                      # PAGED_GQA_ERR_WORKSPACE, nothing launched
    np.testing.assert_array_equal(x.cpu().numpy(), 0)
