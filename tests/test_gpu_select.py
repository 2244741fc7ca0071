"""GPU parity of QSA block selection against the oracle, bit for bit.

The selection is integer work on the scores' bit patterns, so the library's
sel_idx rows must equal the oracle's exactly ("[Kernel][SM70] Accelerate
exact Qwen3.8 decode", Focused tests: QSA GPU exactness and CUDA-graph
replay).  Cases cover the benchmark workload, ties at the pivot, special
values, rows shorter than k, inert rows, strided score rows and rows longer
than the kernel's shared-memory stage."""
import numpy as np
import pytest

import oracle
from fp8_kv_cache_gb300 import workloads as W
from tests import gpu_util as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _run(scores, q_pos, kv_len, k, n_blocks=None):
    import torch
    import fp8_kv_cache_gb300 as P
    sc = torch.from_numpy(np.ascontiguousarray(scores)).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = P.paged_gqa_select_blocks(sc, U.dev(q_pos), kv_len, k, n_blocks=n_blocks, err_flag=err)
    torch.cuda.synchronize()
    return out.cpu().numpy(), int(err.item())


def _check(scores, q_pos, kv_len, k, n_blocks=None, what=""):
    got, flags = _run(scores, q_pos, kv_len, k, n_blocks)
    want, oflags = oracle.select_blocks(scores, q_pos, kv_len, k, n_blocks=n_blocks)
    bad = np.argwhere(np.any(got != want, axis=1)).ravel()
    assert bad.size == 0, f"{what}: {bad.size} rows differ, first {bad[:5]}: " \
                          f"{got[bad[0]][:12]} vs {want[bad[0]][:12]}"
    assert flags == oflags, f"{what}: flags {flags} != oracle {oflags}"
    return got


def test_bench_workload_bitwise():
    c = W.qsa_select_4096()
    got = _check(c.scores, c.q_pos, c.kv_len, c.k, what=c.name)
    assert np.all(got >= 0) and np.all(np.diff(got, axis=1) > 0)


@pytest.mark.parametrize("k", [1, 7, 64, 511, 512, 513, 3000])
def test_ties_and_k(k):
    rng = np.random.default_rng(300 + k)
    R, nb = 96, 2048
    sc = rng.integers(-6, 7, size=(R, nb)).astype(np.float32)   # 13 values: ties everywhere
    n = rng.integers(0, nb + 1, size=R)
    qp = (4 * n + rng.integers(0, 4, size=R)).astype(np.int32)
    _check(sc, qp, 4 * nb + 4, k, what=f"ties k={k}")


def test_constant_and_monotone_rows():
    nb = 4000
    rows = [np.full(nb, 1.5, np.float32), np.arange(nb, dtype=np.float32),
            np.arange(nb, 0, -1).astype(np.float32), np.zeros(nb, np.float32)]
    sc = np.stack(rows)
    qp = np.full(4, 4 * nb, dtype=np.int32)
    for k in (1, 100, 3999, 4000, 4001):
        _check(sc, qp, 4 * nb + 1, k, what=f"monotone k={k}")


def test_special_values():
    """+-0, +-inf, NaNs of both signs and payloads, subnormals, mixed in."""
    rng = np.random.default_rng(301)
    R, nb = 64, 1024
    bits = rng.standard_normal((R, nb)).astype(np.float32).view(np.uint32)
    specials = np.array([0x00000000, 0x80000000, 0x7F800000, 0xFF800000, 0x7FC00000,
                         0xFFC00000, 0x7F800001, 0xFFFFFFFF, 0x00000001, 0x80000001,
                         0x7F7FFFFF, 0xFF7FFFFF], dtype=np.uint32)
    mask = rng.random((R, nb)) < 0.3
    bits[mask] = rng.choice(specials, size=int(mask.sum()))
    sc = bits.view(np.float32)
    qp = (4 * rng.integers(0, nb + 1, size=R)).astype(np.int32)
    for k in (1, 16, 300):
        _check(sc, qp, 4 * nb + 4, k, what=f"specials k={k}")


@pytest.mark.parametrize("k", [100, 700, 1400])
def test_bucket_sizes(k):
    """Rows whose pivot falls in a first-digit bucket of 1500 keys (values in
    [1, 1.25) share their first 11 key bits): larger than the buckets ranked
    outright, so the later digits are histogrammed."""
    rng = np.random.default_rng(310 + k)
    R, nb = 8, 8000
    sc = -rng.random((R, nb)).astype(np.float32)                 # below the bucket
    idx = rng.random((R, nb)).argsort(axis=1)[:, :1500]
    vals = (1.0 + 0.25 * rng.random((R, 1500))).astype(np.float32)
    np.put_along_axis(sc, idx, vals, axis=1)
    sc[1] = np.round(sc[1] * 64) / 64                           # ties inside the bucket
    qp = np.full(R, 4 * nb + 1, dtype=np.int32)
    _check(sc, qp, 4 * nb + 4, k, what=f"bucket k={k}")


def test_inert_rows_and_flags():
    rng = np.random.default_rng(302)
    sc = rng.standard_normal((8, 100)).astype(np.float32)
    qp = np.array([-5, 0, 3, 7, 399, 1000, 401, 250], dtype=np.int32)
    _check(sc, qp, 420, 10, what="inert")                 # 1000 clamped; 401..419 past 100 scores
    _check(sc, qp, 0, 10, what="kv_len 0")
    _check(sc, qp, 420, 10, n_blocks=50, what="n_blocks 50")


def test_strided_score_rows():
    import torch
    import fp8_kv_cache_gb300 as P
    rng = np.random.default_rng(303)
    full = rng.standard_normal((40, 700)).astype(np.float32)
    qp = (4 * rng.integers(0, 600, size=40) + 2).astype(np.int32)
    sc = torch.from_numpy(full).cuda()[:, 50:650]          # row stride 700, 600 columns
    got = P.paged_gqa_select_blocks(sc, U.dev(qp), 4000, 37).cpu().numpy()
    want, _ = oracle.select_blocks(full[:, 50:650], qp, 4000, 37)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("k", [1, 1000, 39999])
def test_rows_longer_than_the_stage(k):
    """Rows of 40000 candidates read their keys from global memory."""
    rng = np.random.default_rng(304 + k)
    R, nb = 6, 40000
    sc = rng.standard_normal((R, nb)).astype(np.float32)
    sc[1] = np.round(sc[1] * 4)                            # heavy ties
    sc[2] = 0.25
    qp = np.full(R, 4 * nb + 3, dtype=np.int32)
    qp[5] = 4 * 17000                                     # just over the stage
    _check(sc, qp, 4 * nb + 4, k, what=f"long k={k}")


def test_run_to_run_and_graph_replay_are_bitwise_equal():
    import torch
    import fp8_kv_cache_gb300 as P
    c = W.select_case("graph", R=512, n_blocks=4096, k=256, seed=305, first_block=2048)
    sc, qp = torch.from_numpy(c.scores).cuda(), U.dev(c.q_pos)
    a = P.paged_gqa_select_blocks(sc, qp, c.kv_len, c.k)
    b = P.paged_gqa_select_blocks(sc, qp, c.kv_len, c.k)
    out = torch.empty_like(a)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        P.paged_gqa_select_blocks(sc, qp, c.kv_len, c.k, out=out)   # first call outside capture
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            P.paged_gqa_select_blocks(sc, qp, c.kv_len, c.k, out=out)
    out.fill_(-7)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(a, b) and torch.equal(a, out)


def test_selection_feeds_sparse_prefill():
    """select -> prefill on the GPU equals the oracle's prefill over the
    oracle's selection."""
    import torch
    import fp8_kv_cache_gb300 as P
    pc = W.prefill_case("qsa_step", R=48, n_sel=64, seed=306, first_block=96)
    sc = W.select_case("qsa_step_scores", R=48, n_blocks=pc.kv_len // 4, k=64, seed=307,
                       q_pos=pc.q_pos, kv_len=pc.kv_len)
    sel = P.paged_gqa_select_blocks(torch.from_numpy(sc.scores).cuda(), U.dev(pc.q_pos),
                                    pc.kv_len, 64)
    want_sel, _ = oracle.select_blocks(sc.scores, pc.q_pos, pc.kv_len, 64)
    assert np.array_equal(sel.cpu().numpy(), want_sel)
    _, k, v = U.dev_kv(pc)
    got = P.paged_gqa_sparse_prefill(U.dev(pc.q), k, v, U.dev(pc.block_table), pc.kv_len, sel,
                                     U.dev(pc.q_pos), pc.page_size, pc.softmax_scale, pc.kv_scale,
                                     num_pages=pc.num_pages)
    torch.cuda.synchronize()
    pc.sel_idx = want_sel
    want, _, _ = U.oracle_prefill(pc)
    U.assert_close(got.cpu().numpy(), want, "select -> prefill")
