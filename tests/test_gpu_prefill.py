"""GPU parity of selected-sparse prefill against the FP64 oracle."""
import numpy as np
import pytest

from fp8_kv_cache_gb300 import workloads as W
from tests import gpu_util as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _check_full(case, **kw):
    got, flags = U.run_prefill(case, **kw)
    want, _, oflags = U.oracle_prefill(case, **kw)
    U.assert_close(got, want, case.name)
    assert flags == oflags, f"{case.name}: flags {flags} != oracle {oflags}"
    return got


def _small(seed, **kw):
    args = dict(R=37, n_sel=24, first_block=40, page_size=16, tails=(1, 2, 3, 4))
    args.update(kw)
    return W.prefill_case(f"prefill_s{seed}", seed=seed, **args)


@pytest.mark.parametrize("interleaved", [True, False])
@pytest.mark.parametrize("kvd", ["fp16", "e4m3"])
def test_small_layouts_and_dtypes(kvd, interleaved):
    _check_full(_small(100, kv_dtype=kvd, interleaved=interleaved))


@pytest.mark.parametrize("tail", [1, 2, 3, 4])
def test_each_tail_length(tail):
    _check_full(_small(110 + tail, tails=(tail,)))


@pytest.mark.parametrize("n_sel", [0, 1, 2, 3, 5, 511, 512])
def test_selection_counts(n_sel):
    _check_full(_small(120, n_sel=n_sel, first_block=max(n_sel, 8), R=9))


@pytest.mark.parametrize("page_size", [4, 8, 48, 784])
def test_page_sizes(page_size):
    _check_full(_small(130, page_size=page_size))


def test_grouped_heads_and_single_row():
    _check_full(_small(140, Hq=12, Hkv=2))
    _check_full(_small(141, Hq=16, Hkv=2, R=1))


def test_unsorted_selection_and_inert_entries():
    c = _small(150)
    rng = np.random.default_rng(5)
    for r in range(c.R):
        rng.shuffle(c.sel_idx[r])             # order is free
    c.sel_idx[3, :5] = -1                      # padding
    c.sel_idx[4, 0] = c.q_pos[4] // 4          # the row's own block: skipped, flagged
    c.sel_idx[5, 1] = c.q_pos[5] // 4 + 9      # a future block: skipped, flagged
    c.q_pos[6] = -2                            # zero row, flagged
    c.q_pos[7] = c.kv_len + 100                # clamped, flagged
    c.block_table[2] = -1                      # a hole in the page table
    got = _check_full(c)
    assert np.all(got[6] == 0)


def test_full_4096_rows_sampled():
    c = W.sparse_prefill_4096()
    got, flags = U.run_prefill(c)
    rows = np.random.default_rng(7).choice(c.R, size=24, replace=False).astype(np.int32)
    rows = np.concatenate([rows, [0, c.R - 1]]).astype(np.int32)
    want, _, oflags = U.oracle_prefill(c, rows=rows)
    U.assert_close(got[rows], want[rows], c.name)
    assert flags == 0 and oflags == 0
    again, _ = U.run_prefill(c)
    assert np.array_equal(got.view(np.uint16), again.view(np.uint16)), "run-to-run"


def test_full_4096_rows_interleaved_e4m3_sampled():
    """The E4M3 prefill exactly as the benchmark times it."""
    c = W.sparse_prefill_4096(kv_dtype="e4m3")
    got, flags = U.run_prefill(c)
    rows = np.random.default_rng(9).choice(c.R, size=24, replace=False).astype(np.int32)
    rows = np.concatenate([rows, [0, c.R - 1]]).astype(np.int32)
    want, _, oflags = U.oracle_prefill(c, rows=rows)
    U.assert_close(got[rows], want[rows], c.name)
    assert flags == 0 and oflags == 0


def test_full_4096_rows_contiguous_e4m3_sampled():
    c = W.prefill_case("prefill_4096_e4m3", R=4096, n_sel=512, seed=6, first_block=4096,
                       kv_len=32768, interleaved=False, kv_dtype="e4m3")
    got, _ = U.run_prefill(c)
    rows = np.random.default_rng(8).choice(c.R, size=16, replace=False).astype(np.int32)
    want, _, _ = U.oracle_prefill(c, rows=rows)
    U.assert_close(got[rows], want[rows], c.name)
