"""GPU parity of batched paged decode against the FP64 oracle.

Every case compares the library's FP16 output element by element with the
oracle's FP16-rounded output (max abs <= 2e-3, rel L2 <= 5e-4).  Full-size
workloads run in the launch configuration the benchmark times (automatic
split) and are checked on every (sequence, head) row, with the strict 2e-3
bound (no FP16-ULP allowance used)."""
import numpy as np
import pytest

from fp8_kv_cache_gb300 import workloads as W
from tests import gpu_util as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _check_full(case, strict=False, **kw):
    got, flags = U.run_decode(case, **kw)
    want, _, oflags = U.oracle_decode(case)
    _, _, wide = U.assert_close(got, want, case.name)
    assert not (strict and wide), f"{case.name}: {wide} elements needed the ULP allowance"
    assert flags == oflags, f"{case.name}: flags {flags} != oracle {oflags}"
    return got


def _check_pairs(case, pairs, kv=None, **kw):
    got, flags = U.run_decode(case, kv=kv, **kw)
    want, _, oflags = U.oracle_decode(case, pairs=pairs)
    b, h = pairs[:, 0], pairs[:, 1]
    _, _, wide = U.assert_close(got[b, h], want[b, h], case.name)
    assert wide == 0, f"{case.name}: {wide} elements needed the ULP allowance"
    assert flags == oflags
    return got


# ---------------------------------------------------------------- the configs

def test_tiny_fp16_split_and_unsplit():
    c = W.tiny_fp16()
    a = _check_full(c, strict=True)
    b = _check_full(c, strict=True, workspace=False)
    U.assert_close(a, b, "split vs unsplit")


def test_e4m3_b8():
    _check_full(W.e4m3_b8(), strict=True)


@pytest.fixture(scope="module")
def long_case():
    c = W.long_e4m3()
    return c, U.dev_kv(c)


def test_long_e4m3_every_row(long_case):
    """The benchmark's long-context E4M3 workload: all 16 x 24 (sequence,
    head) rows against the oracle."""
    c, kv = long_case
    got, flags = U.run_decode(c, kv=kv)
    want, _, oflags = U.oracle_decode(c)
    _, _, wide = U.assert_close(got, want, c.name)
    assert wide == 0, f"{c.name}: {wide} elements needed the ULP allowance"
    assert flags == oflags == 0


def test_long_e4m3_sampled_pairs_match_full_oracle(long_case):
    """The oracle's (sequence, head) pair mode agrees with its full mode."""
    c, kv = long_case
    _check_pairs(c, U.sample_pairs(c.B, c.Hq, per_seq=3, seed=1), kv=kv)


@pytest.mark.parametrize("kvd", ["fp16", "e4m3"])
@pytest.mark.parametrize("L", [1024, 16384])
@pytest.mark.parametrize("B", [1, 2, 4, 8, 16])
def test_sweep(B, L, kvd):
    """The batch/context grid ([D] Performance contract), every row."""
    _check_full(W.sweep(B, L, kvd), strict=True)


# ---------------------------------------------------------------- shapes and edges

@pytest.mark.parametrize("kvd", ["fp16", "e4m3"])
@pytest.mark.parametrize("page_size", [16, 4, 48, 64, 128, 256, 784])
def test_ragged_lengths_and_page_sizes(page_size, kvd):
    lens = [1, 7, 8, 9, 15, 16, 17, 31, 33, 100, 257, 1500]
    c = W.decode_case(f"ragged_p{page_size}_{kvd}", B=len(lens), Hq=12, Hkv=2, seq_lens=lens,
                      kv_dtype=kvd, seed=60 + page_size)
    _check_full(c)
    _check_full(c, workspace=False)


@pytest.mark.parametrize("G", [1, 2, 3, 5, 6, 7, 8])
def test_group_sizes(G):
    c = W.decode_case(f"group{G}", B=3, Hq=2 * G, Hkv=2, seq_lens=[5, 200, 77], kv_dtype="e4m3",
                      seed=70 + G)
    _check_full(c)


@pytest.mark.parametrize("kvd", ["fp16", "e4m3"])
def test_interleaved_layout(kvd):
    c = W.decode_case(f"interleaved_{kvd}", B=4, Hq=24, Hkv=4, seq_lens=[300, 1, 64, 1000],
                      kv_dtype=kvd, seed=80, interleaved=True)
    _check_full(c)


@pytest.mark.parametrize("splits", [1, 2, 3, 5, 64, 1000])
def test_split_count_invariance(splits):
    c = W.decode_case("splits", B=3, Hq=24, Hkv=4, seq_lens=[700, 33, 2000], kv_dtype="e4m3",
                      seed=90)
    got = _check_full(c, force_splits=splits)
    ref, _ = U.run_decode(c)
    U.assert_close(got, ref, f"splits={splits} vs automatic")


@pytest.mark.parametrize("kvd", ["fp16", "e4m3"])
@pytest.mark.parametrize("B", [512, 513, 1500])
def test_large_batches(B, kvd):
    """Batches on both sides of 512, where the merge kernel switches from
    recomputing the cut from seq_lens to reading the prefix the split kernel
    leaves in the workspace; short ragged lengths with empty rows."""
    rng = np.random.default_rng(1000 + B)
    lens = rng.integers(-2, 200, size=B).astype(np.int32)
    c = W.decode_case(f"large_b{B}", B=B, Hq=12, Hkv=2, seq_lens=lens, kv_dtype=kvd,
                      seed=95 + B, max_seq_len=200)
    got = _check_full(c)
    for splits in (B // 3, 4 * B):
        alt, _ = U.run_decode(c, force_splits=splits)
        U.assert_close(alt, got, f"B={B} splits={splits} vs automatic")


def test_inert_inputs_match_oracle():
    c = W.decode_case("inert", B=6, Hq=12, Hkv=2, seq_lens=[40, 0, -3, 500, 64, 33],
                      kv_dtype="e4m3", seed=91, max_seq_len=256, num_pages=200)
    c.block_table[4, 1] = -1                  # a hole: tokens 16..31 skipped
    c.block_table[4, 2] = c.num_pages         # first out-of-range id
    c.block_table[5, 0] = 1 << 30
    for kw in ({}, {"workspace": False}, {"force_splits": 7}):
        got, flags = U.run_decode(c, **kw)
        want, _, oflags = U.oracle_decode(c)
        U.assert_close(got, want, f"inert {kw}")
        assert np.all(got[1] == 0) and np.all(got[2] == 0)
        assert flags == oflags == 1 | 2 | 4, (flags, oflags)


def test_all_pages_invalid_gives_zero_rows():
    c = W.decode_case("all_bad", B=2, Hq=6, Hkv=1, seq_lens=[20, 40], kv_dtype="fp16", seed=92)
    c.block_table[:] = -7
    for kw in ({}, {"workspace": False}, {"force_splits": 3}):
        got, flags = U.run_decode(c, **kw)
        assert np.all(got == 0) and flags == 1


def test_page_permutation_is_bitwise_invariant():
    c = W.decode_case("perm", B=4, Hq=24, Hkv=4, seq_lens=[900, 1, 64, 333], kv_dtype="e4m3",
                      seed=93)
    a, _ = U.run_decode(c)
    rng = np.random.default_rng(3)
    perm = rng.permutation(c.num_pages)
    c2 = W.decode_case("perm", B=4, Hq=24, Hkv=4, seq_lens=[900, 1, 64, 333], kv_dtype="e4m3",
                       seed=93)
    c2.kv = np.empty_like(c.kv)
    c2.kv[:, perm] = c.kv
    c2.k, c2.v = c2.kv[0], c2.kv[1]
    c2.block_table = perm[c.block_table].astype(np.int32)
    b, _ = U.run_decode(c2)
    assert np.array_equal(a.view(np.uint16), b.view(np.uint16))


def test_run_to_run_and_graph_replay_are_bitwise_equal():
    import torch
    import fp8_kv_cache_gb300 as P
    c = W.e4m3_b8()
    _, k, v = U.dev_kv(c)
    q, bt, sl = U.dev(c.q), U.dev(c.block_table), U.dev(c.seq_lens)
    ws = torch.empty(P.paged_gqa_decode_workspace_size(c.B, c.Hq, c.Hkv, c.D, c.max_seq_len),
                     dtype=torch.uint8, device="cuda")
    out = torch.empty_like(q)

    def call():
        P.paged_gqa_decode(q, k, v, bt, sl, c.page_size, c.kv_scale, c.softmax_scale, out,
                           max_seq_len=c.max_seq_len, workspace=ws)

    call()
    torch.cuda.synchronize()
    eager = out.clone()
    call()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call()                                # warm up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    for _ in range(2):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
