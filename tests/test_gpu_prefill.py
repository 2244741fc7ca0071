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


# Kernel routes: the per-row kernel, and the grouped tcgen05 kernel with the
# automatic group size and with forced sizes (the largest group of 128 slots,
# and a small one that leaves a ragged last group).
ROUTES = [dict(route=1), dict(route=2), dict(route=2, rows_per_group=3)]
ROUTE_IDS = ["rowwise", "grouped", "grouped3"]


def _check_full(case, route=None, **kw):
    got, flags = U.run_prefill(case, **(route or {}))
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


@pytest.mark.parametrize("interleaved", [True, False])
@pytest.mark.parametrize("route", ROUTES, ids=ROUTE_IDS)
@pytest.mark.parametrize("kvd", ["fp16", "e4m3"])
def test_small_layouts_routes(kvd, route, interleaved):
    _check_full(_small(101, kv_dtype=kvd, interleaved=interleaved), route)


@pytest.mark.parametrize("route", ROUTES, ids=ROUTE_IDS)
def test_e4m3_inert_entries_and_tails(route):
    c = _small(102, kv_dtype="e4m3", tails=(1, 2, 3, 4))
    c.sel_idx[3, :5] = -1
    c.sel_idx[4, 0] = c.q_pos[4] // 4
    c.q_pos[6] = -2
    c.block_table[1] = 10 ** 6
    _check_full(c, route)


@pytest.mark.parametrize("route", ROUTES, ids=ROUTE_IDS)
@pytest.mark.parametrize("tail", [1, 2, 3, 4])
def test_each_tail_length(tail, route):
    _check_full(_small(110 + tail, tails=(tail,)), route)


@pytest.mark.parametrize("route", ROUTES, ids=ROUTE_IDS)
@pytest.mark.parametrize("n_sel", [0, 1, 2, 3, 5, 511, 512])
def test_selection_counts(n_sel, route):
    _check_full(_small(120, n_sel=n_sel, first_block=max(n_sel, 8), R=9), route)


@pytest.mark.parametrize("route", ROUTES, ids=ROUTE_IDS)
@pytest.mark.parametrize("page_size", [4, 8, 48, 784])
def test_page_sizes(page_size, route):
    _check_full(_small(130, page_size=page_size), route)


@pytest.mark.parametrize("route", ROUTES, ids=ROUTE_IDS)
def test_grouped_heads_and_single_row(route):
    _check_full(_small(140, Hq=12, Hkv=2), route)
    _check_full(_small(141, Hq=16, Hkv=2, R=1), route)


@pytest.mark.parametrize("rows", [1, 2, 5, 16, 21])
def test_grouped_route_group_sizes(rows):
    """Groups of 1 .. 21 rows (126 of 128 slots at six heads per KV head),
    37 rows so most sizes leave a ragged last group."""
    _check_full(_small(160, R=37, n_sel=48, first_block=64), dict(route=2, rows_per_group=rows))


@pytest.mark.parametrize("route", ROUTES, ids=ROUTE_IDS)
def test_peaked_scores_rescale(route):
    """softmax_scale 1 makes scores spread over ~+-50 in the log2 domain, so
    the running maxima keep rising by more than the rescale slack of the
    grouped kernel and O is rescaled in tensor memory many times."""
    c = _small(170, R=21, n_sel=64, first_block=96)
    c.softmax_scale = 1.0
    _check_full(c, route)


@pytest.mark.parametrize("route", ROUTES, ids=ROUTE_IDS)
def test_duplicated_selections_count_per_listing(route):
    """A caller error that still has a meaning: a block listed twice counts
    twice (the oracle attends its tokens twice); the grouped kernel takes its
    slow recount path for such rows."""
    c = _small(180, R=21, n_sel=40, first_block=64)
    c.sel_idx[2, 1] = c.sel_idx[2, 0]
    c.sel_idx[5, 3] = c.sel_idx[5, 7] = c.sel_idx[5, 9]
    c.sel_idx[9, :] = c.sel_idx[9, 0]
    _check_full(c, route)


def test_grouped_route_union_in_two_mask_windows():
    """21 rows of 2048 selections each over ~8000 earlier blocks: the union
    (~8000 blocks, ~500 stages) exceeds the mask capacity of a 21-row group
    (390 stages), so the stage masks are rebuilt for a second window."""
    c = _small(190, R=21, n_sel=2048, first_block=8000, tails=(1, 2, 3))
    _check_full(c, dict(route=2, rows_per_group=21))
    _check_full(c, dict(route=1))


@pytest.mark.parametrize("route", ROUTES, ids=ROUTE_IDS)
def test_unsorted_selection_and_inert_entries(route):
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
    got = _check_full(c, route)
    assert np.all(got[6] == 0)


def test_routes_agree_at_4096_rows_and_grouped_is_deterministic():
    c = W.sparse_prefill_4096()
    grouped, f1 = U.run_prefill(c, route=2)
    rowwise, f2 = U.run_prefill(c, route=1)
    assert f1 == 0 and f2 == 0
    U.assert_close(grouped, rowwise.astype(np.float64), c.name + " grouped vs rowwise")
    again, _ = U.run_prefill(c, route=2)
    assert np.array_equal(grouped.view(np.uint16), again.view(np.uint16)), "run-to-run"


def _every_row(c, routes):
    """Every row of case c on each route against the oracle, strict bound."""
    want, _, oflags = U.oracle_prefill(c)
    outs = {}
    for name, route in routes.items():
        got, flags = U.run_prefill(c, **route)
        _, _, wide = U.assert_close(got, want, f"{c.name} {name}")
        assert wide == 0, f"{c.name} {name}: {wide} elements needed the ULP allowance"
        assert flags == oflags, f"{c.name} {name}: flags {flags} != oracle {oflags}"
        outs[name] = got
    return outs


ALL_ROUTES = {"auto": {}, "rowwise": dict(route=1), "grouped": dict(route=2)}


@pytest.mark.parametrize("kvd", ["fp16", "e4m3"])
def test_full_4096_rows_every_row_every_route(kvd):
    """The 4096-row workload exactly as the benchmark times it ([P] Test
    Result: the 4096-row interleaved-KV A/B), every row on the automatic,
    per-row and grouped routes, FP16 and E4M3 caches; run to run bitwise."""
    c = W.sparse_prefill_4096(kv_dtype=kvd)
    outs = _every_row(c, ALL_ROUTES)
    again, _ = U.run_prefill(c)
    assert np.array_equal(outs["auto"].view(np.uint16), again.view(np.uint16)), "run-to-run"


@pytest.mark.parametrize("R", [1, 4095, 4097])
def test_row_count_boundary(R):
    """[P] Test Result: 4095 rows around the 4096-row route.  The grouped
    route's rows per group depend on R (its groups fill whole waves), so
    1, 4095 and 4097 rows take different partitions and ragged last groups;
    4096 is the test above.  Every row on both routes."""
    c = W.sparse_prefill_4096(R=R)
    _every_row(c, {"rowwise": dict(route=1), "grouped": dict(route=2)})


def test_full_4096_rows_contiguous_e4m3_sampled():
    c = W.prefill_case("prefill_4096_e4m3", R=4096, n_sel=512, seed=6, first_block=4096,
                       kv_len=32768, interleaved=False, kv_dtype="e4m3")
    got, _ = U.run_prefill(c)
    rows = np.random.default_rng(8).choice(c.R, size=16, replace=False).astype(np.int32)
    want, _, _ = U.oracle_prefill(c, rows=rows)
    U.assert_close(got[rows], want[rows], c.name)


@pytest.mark.parametrize("route", [1, 2], ids=["rowwise", "grouped"])
def test_graph_replay_equals_eager(route):
    """[P] Test Result: graph replay equal to eager.  The prefill captured in a
    CUDA graph and replayed writes the same bits as the eager call, on the
    hybrid 784-token pages of the same page ([P] Test Result: 784/16)."""
    import torch
    import fp8_kv_cache_gb300 as P
    c = _small(200, R=40, n_sel=48, first_block=64, page_size=784)
    _, k, v = U.dev_kv(c)
    q, bt = U.dev(c.q), U.dev(c.block_table)
    sel, pos = U.dev(c.sel_idx), U.dev(c.q_pos)

    def call(out):
        return P.paged_gqa_sparse_prefill_route(q, k, v, bt, c.kv_len, sel, pos, c.page_size,
                                                c.softmax_scale, c.kv_scale, out,
                                                route=route, num_pages=c.num_pages)

    eager = call(torch.empty_like(q))
    out = torch.empty_like(q)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        call(out)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            call(out)
    out.fill_(7.0)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(eager.view(torch.int16), out.view(torch.int16))
    want, _, _ = U.oracle_prefill(c)
    U.assert_close(out.cpu().numpy(), want, c.name)


def test_grouped_route_long_sequence():
    """A ~99,800-token sequence (a 780-word union bitmap, close to the
    131,072-token limit of the grouped route): 48 rows near the end, each
    with 256 selections spread over ~25,000 earlier blocks."""
    c = _small(210, R=48, n_sel=256, first_block=24900, tails=(1, 2, 3))
    assert c.kv_len > 99000
    _check_full(c, dict(route=2))
    _check_full(c, dict(route=2, rows_per_group=21))


@pytest.mark.parametrize("route", ROUTES, ids=ROUTE_IDS)
def test_degenerate_inputs(route):
    """Every row empty (q_pos < 0), a zero-length sequence, every selection
    padding, and every page of the table invalid: outputs are zero or the
    tail alone, flags as the oracle's."""
    c = _small(220, R=9)
    c.q_pos[:] = -1                                            # all rows empty
    got = _check_full(c, route)
    assert np.all(got == 0)
    c = _small(221, R=9)
    c.kv_len = 0                                               # no tokens at all
    got = _check_full(c, route)
    assert np.all(got == 0)
    c = _small(222, R=9)
    c.sel_idx[:] = -1                                          # tails only
    _check_full(c, route)
    c = _small(223, R=9)
    c.block_table[:] = -5                                      # every page invalid
    got = _check_full(c, route)
    assert np.all(got == 0)


@pytest.mark.parametrize("Hq,Hkv,rows", [(2, 2, 128), (2, 2, 0), (6, 2, 42), (3, 1, 0)])
def test_grouped_route_head_groupings(Hq, Hkv, rows):
    """One query head per KV head (128 rows per group: 32 mask words per row,
    64 stages per mask window, so a union of ~130 stages is masked in three
    windows), three per KV head, two KV heads; forced and automatic group
    sizes."""
    c = _small(230 + Hq + Hkv + rows, R=150, n_sel=256, first_block=2000, Hq=Hq, Hkv=Hkv)
    _check_full(c, dict(route=2, rows_per_group=rows))


def test_grouped_wait_time_out_sets_the_flag_and_the_next_call_is_correct():
    """The grouped kernel's bounded waits ([P] Changes: invalid requests are
    inert, never fatal): through the test hook every wait gives up after
    2000 polls (a few milliseconds) and each CTA leaves its fourth ring stage
    unpublished, so the tensor-core thread's wait for it runs out.  The CTA
    must skip its remaining waits, let its issued MMAs finish, free its
    tensor memory and raise PAGED_GQA_FLAG_TIMEOUT; the context stays usable
    and the next call is correct.  With no stall the hook is the normal
    kernel."""
    import torch
    import fp8_kv_cache_gb300 as P
    c = _small(240, R=37, n_sel=48, first_block=64)
    _, k, v = U.dev_kv(c)
    q, bt, sel, pos = U.dev(c.q), U.dev(c.block_table), U.dev(c.sel_idx), U.dev(c.q_pos)
    want, _, _ = U.oracle_prefill(c)

    def hook(spin_limit, stall_stage):
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        out = P.paged_gqa_debug_grouped_prefill_stall(
            q, k, v, bt, c.kv_len, sel, pos, c.page_size, c.softmax_scale, c.kv_scale,
            spin_limit=spin_limit, stall_stage=stall_stage, num_pages=c.num_pages, err_flag=err)
        torch.cuda.synchronize()
        return out.cpu().numpy(), int(err.item())

    _, flags = hook(2000, 3)
    assert flags & P.FLAG_TIMEOUT, flags
    got, flags = hook(0, -1)                    # the hook without a stall
    assert flags == 0
    U.assert_close(got, want, "hook without a stall")
    got = _check_full(c, dict(route=2))         # a normal call after the time-out
    U.assert_close(got, want, "after the time-out")
    with pytest.raises(P.PagedGQAError):
        hook(-1, 0)
