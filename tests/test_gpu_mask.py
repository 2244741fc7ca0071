"""GPU parity of the combined top-k/top-p masking against the oracle.

The kept logits must be the oracle's, bit for bit, and every other logit
-inf.  The top-p decision is taken in FP64 on both sides ("[Kernel][SM70]
Scale NVFP4 E4M3 decode batches", Purpose: combined top-k/top-p masking;
compared bitwise in its Test plan and result); exp may differ by an ulp
between the two libraries, so a row whose decision lies within 1e-12 of its
threshold (the oracle's margin) may differ there, and the test reports it."""
import numpy as np
import pytest

import oracle
from fp8_kv_cache_gb300 import workloads as W

pytestmark = pytest.mark.gpu

MARGIN = 1e-12


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _run(x, k, p, in_place=False, stride=None):
    import torch
    import fp8_kv_cache_gb300 as P
    B, V = x.shape
    if stride is None:
        xd = torch.from_numpy(np.ascontiguousarray(x)).cuda()
    else:
        full = torch.full((B, stride), 7.0, dtype=torch.float32, device="cuda")
        full[:, :V] = torch.from_numpy(np.ascontiguousarray(x)).cuda()
        xd = full[:, :V]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = P.paged_gqa_topk_topp_mask(xd, k, p, out=xd if in_place else None, err_flag=err)
    torch.cuda.synchronize()
    return out.cpu().numpy(), int(err.item())


def _check(x, k, p, what="", **kw):
    got, flags = _run(x, k, p, **kw)
    want, margin = oracle.topk_topp_mask(x, k, p)
    assert flags == 0, f"{what}: flags {flags}"
    close = 0
    for r in range(x.shape[0]):
        if np.array_equal(got[r].view(np.uint32), want[r].view(np.uint32)):
            continue
        assert margin[r] < MARGIN, f"{what} row {r}: kept " \
            f"{np.flatnonzero(got[r] > -np.inf)[:8]} vs {np.flatnonzero(want[r] > -np.inf)[:8]}"
        close += 1
    if close:
        print(f"{what}: {close} rows decided within {MARGIN} of the top-p threshold")
    return got


def test_bench_workload():
    c = W.sampler_b16()
    got = _check(c.logits, c.k, c.p, c.name)
    kept = (got > -np.inf).sum(1)
    assert np.all(kept >= 1) and np.all(kept <= c.k)


@pytest.mark.parametrize("k", [1, 20, 64, 128])
@pytest.mark.parametrize("p", [1.0, 0.95, 0.5, 1e-6])
def test_k_and_p(k, p):
    c = W.logits_case("kp", B=8, V=50000, k=k, p=p, seed=500 + k)
    _check(c.logits, k, p, f"k={k} p={p}")


def test_ties_signed_zeros_and_neg_inf():
    rng = np.random.default_rng(501)
    x = np.round(rng.standard_normal((6, 20000)) * 2).astype(np.float32)   # 13 or so values
    x[1] = 0.0
    x[1, ::3] = -0.0
    x[2, :19000] = -np.inf
    x[3] = -np.inf
    x[4, 5000:] = 4.0                                                      # a wide tie at the top
    for k, p in ((20, 0.95), (128, 0.5), (1, 1.0), (77, 1.0)):
        _check(x, k, p, f"ties k={k} p={p}")


@pytest.mark.parametrize("V", [1, 5, 7, 8, 33, 1023, 262144, 327680])
def test_vocab_sizes(V):
    c = W.logits_case("vocab", B=3, V=V, seed=502, peaks=min(32, V))
    _check(c.logits, min(20, 128), 0.9, f"V={V}")


def test_many_rows():
    """300 rows: many waves of clusters."""
    c = W.logits_case("many", B=300, V=3000, seed=506, peaks=8)
    _check(c.logits, 20, 0.95, "B=300")


def test_strided_and_in_place():
    c = W.logits_case("strided", B=4, V=30001, seed=503)
    want, _ = oracle.topk_topp_mask(c.logits, 20, 0.95)
    a, _ = _run(c.logits, 20, 0.95, stride=30007)          # odd row stride: unaligned rows
    b, _ = _run(c.logits, 20, 0.95, in_place=True)
    assert np.array_equal(a.view(np.uint32), want.view(np.uint32))
    assert np.array_equal(b.view(np.uint32), want.view(np.uint32))


def test_unaligned_output_rows_and_in_place_unaligned_rows():
    """An output whose rows start off a 16-byte boundary (the -inf fill is
    then written by the threads during the sweep, not by bulk copies), and
    masking in place rows that start off a 16-byte boundary."""
    import torch
    import fp8_kv_cache_gb300 as P
    c = W.logits_case("unaligned_out", B=5, V=30001, seed=507)
    want, margin = oracle.topk_topp_mask(c.logits, 20, 0.95)
    x = torch.from_numpy(c.logits).cuda()
    big = torch.full((5, 30001 + 3), 5.0, dtype=torch.float32, device="cuda")
    out = big[:, 1:30002]                                  # rows at 4 bytes past an aligned start
    assert out.data_ptr() % 16 != 0
    P.paged_gqa_topk_topp_mask(x, 20, 0.95, out=out)
    buf = torch.full((5, 30007), 7.0, dtype=torch.float32, device="cuda")
    xs = buf[:, 1:30002]
    xs.copy_(x)
    P.paged_gqa_topk_topp_mask(xs, 20, 0.95, out=xs)      # in place, odd row stride
    torch.cuda.synchronize()
    for got in (out.cpu().numpy(), xs.cpu().numpy()):
        for r in range(5):
            if not np.array_equal(got[r].view(np.uint32), want[r].view(np.uint32)):
                assert margin[r] < MARGIN, f"row {r}"
    assert bool((big[:, 0] == 5.0).all()) and bool((big[:, 30002:] == 5.0).all())
    assert bool((buf[:, 0] == 7.0).all()) and bool((buf[:, 30002:] == 7.0).all())


def test_nan_or_inf_top_is_flagged():
    rng = np.random.default_rng(504)
    x = rng.standard_normal((3, 1000)).astype(np.float32)
    x[0, 17] = np.nan
    x[1, 400] = np.inf
    got, flags = _run(x, 5, 0.5)
    assert flags == 64
    assert np.array_equal(np.flatnonzero(~np.isneginf(got[2])),
                          np.flatnonzero(~np.isneginf(oracle.topk_topp_mask(x[2:], 5, 0.5)[0][0])))


def test_run_to_run_and_graph_replay_are_bitwise_equal():
    import torch
    import fp8_kv_cache_gb300 as P
    c = W.logits_case("graph", B=8, V=100000, seed=505)
    x = torch.from_numpy(c.logits).cuda()
    a = P.paged_gqa_topk_topp_mask(x, 20, 0.95)
    b = P.paged_gqa_topk_topp_mask(x, 20, 0.95)
    out = torch.empty_like(a)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        P.paged_gqa_topk_topp_mask(x, 20, 0.95, out=out)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            P.paged_gqa_topk_topp_mask(x, 20, 0.95, out=out)
    out.fill_(3.0)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    assert torch.equal(a.view(torch.int32), out.view(torch.int32))
