"""Bit-exact comparison of the kernels' gather and dequantisation with the
oracle: the dequantised rows the decode kernels read (E4M3 code value times
kv_scale, rounded once to float; FP16 exactly) and the token list of every
sparse-prefill row."""
import numpy as np
import pytest

import oracle
import fp8_kv_cache_gb300 as P
from fp8_kv_cache_gb300 import workloads as W
from tests import gpu_util as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _gather_equal(case, b_sel=None):
    _, k, v = U.dev_kv(case)
    bt = case.block_table if b_sel is None else case.block_table[b_sel]
    sl = case.seq_lens if b_sel is None else case.seq_lens[b_sel]
    for view, host in ((k, case.k), (v, case.v)):
        got = P.paged_gqa_gather_dequant(view, U.dev(bt), U.dev(sl), case.page_size,
                                         case.max_seq_len, case.kv_scale,
                                         num_pages=case.num_pages).cpu().numpy()
        want = oracle.gather_rows(host, bt, sl, case.page_size, case.num_pages, case.max_seq_len,
                                  case.kv_scale)
        nan = np.isnan(want)
        assert np.array_equal(np.isnan(got), nan)
        assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32)), case.name


def test_gather_e4m3_b8():
    _gather_equal(W.e4m3_b8())


def test_gather_tiny_fp16():
    _gather_equal(W.tiny_fp16())


def test_gather_long_e4m3_subset():
    _gather_equal(W.long_e4m3(), b_sel=np.array([0, 7, 15]))


def test_gather_interleaved_ragged_bad_pages():
    c = W.decode_case("g_il", B=3, Hq=12, Hkv=2, seq_lens=[50, 3, 200], kv_dtype="e4m3", seed=200,
                      interleaved=True, page_size=48, num_pages=40)
    c.block_table[2, 1] = -1
    c.block_table[0, 0] = c.num_pages
    _gather_equal(c)


def test_every_e4m3_code_including_nan():
    """A pool whose rows hold all 256 codes, NaN codes included."""
    c = W.decode_case("codes", B=1, Hq=6, Hkv=1, seq_lens=[16], kv_dtype="e4m3", seed=201,
                      num_pages=1)
    c.kv[0, 0, :, 0, :] = np.arange(256, dtype=np.uint8)[None, :]
    c.kv[1, 0, :, 0, :] = np.arange(256, dtype=np.uint8)[::-1][None, :]
    _gather_equal(c)


@pytest.mark.parametrize("case", ["small", "full"])
def test_prefill_token_lists(case):
    if case == "full":
        c = W.sparse_prefill_4096()
    else:
        c = W.prefill_case("tok_small", R=50, n_sel=30, seed=202, first_block=40,
                           tails=(1, 2, 3, 4))
        c.sel_idx[3, 2] = -1
        c.sel_idx[4, 0] = c.q_pos[4] // 4
        c.q_pos[5] = -1
        c.q_pos[6] = c.kv_len + 3
        c.block_table[1] = -1
    slots = P.paged_gqa_sparse_prefill_tokens(U.dev(c.block_table), c.num_pages, c.kv_len,
                                              U.dev(c.sel_idx), U.dev(c.q_pos),
                                              c.page_size).cpu().numpy()
    for r in range(c.R):
        got = slots[r][slots[r] >= 0].astype(np.int64)
        want = oracle.sparse_row_tokens(c.block_table, c.num_pages, c.kv_len, c.sel_idx[r],
                                        c.q_pos[r], c.page_size)
        assert np.array_equal(got, want), f"row {r}"


def _xor_words(rows):
    """XOR of every 32-bit word of the given rows (any shape, whole rows)."""
    a = np.ascontiguousarray(rows).reshape(-1).view(np.uint32)
    return int(np.bitwise_xor.reduce(a)) if a.size else 0


@pytest.mark.parametrize("kvd", ["fp16", "e4m3"])
@pytest.mark.parametrize("case", ["small", "full"])
def test_sparse_gather_probe_reads_exactly_the_attended_rows(case, kvd):
    """The gather-ceiling probe folds every word of the K and V rows each
    row attends (selected blocks, causal tail, inert entries skipped), so its
    per-row XOR equals the XOR of those rows read from the host copy."""
    if case == "full":
        c = W.sparse_prefill_4096(kv_dtype=kvd)
        rows = np.random.default_rng(4).choice(c.R, size=40, replace=False)
    else:
        c = W.prefill_case(f"gprobe_{kvd}", R=40, n_sel=30, seed=203, first_block=40,
                           tails=(1, 2, 3, 4), kv_dtype=kvd, Hq=12, Hkv=2)
        c.sel_idx[3, 2] = -1
        c.sel_idx[4, 0] = c.q_pos[4] // 4
        c.q_pos[5] = -1
        c.q_pos[6] = c.kv_len + 3
        c.block_table[1] = -1
        rows = np.arange(c.R)
    _, k, v = U.dev_kv(c)
    got = P.paged_gqa_sparse_gather_probe(k, v, U.dev(c.block_table), c.kv_len, U.dev(c.sel_idx),
                                          U.dev(c.q_pos), c.page_size,
                                          num_pages=c.num_pages).cpu().numpy().view(np.uint32)
    for r in rows:
        toks = oracle.sparse_row_tokens(c.block_table, c.num_pages, c.kv_len, c.sel_idx[r],
                                        c.q_pos[r], c.page_size)
        pages = c.block_table[toks // c.page_size]
        slots = toks % c.page_size
        for j in range(c.Hkv):
            want = _xor_words(c.k[pages, slots, j]) ^ _xor_words(c.v[pages, slots, j])
            assert int(got[r, j]) == want, f"row {r} head {j}"
