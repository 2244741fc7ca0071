"""Pins of the oracle against facts that do not come from the oracle itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError
when it disagrees with:
  * library routines (numpy float16, torch float8_e4m3fn) on the number formats,
  * the closed form of OCP E4M3FN on landmark codes,
  * a textbook dense softmax(s q K^T) V over the unrolled block table,
  * invariants of softmax attention (convex hull, page-permutation invariance,
    one-token context, equal keys, zero query, split/merge identity),
  * the selected-sparse layout printed on the page (2051 tokens for 512 blocks
    plus a 3-token tail) and the dense causal special case,
  * for the block selection: numpy's stable argsort (ties to the lower index)
    on finite scores, closed forms (monotone and constant rows, k >= n), an
    IEEE totalOrder case written out by hand, the inert-row rules, and a
    brute-force dominance check over every subset of tiny rows,
  * for the top-k/top-p masking: numpy's stable argsort (top-k), the closed
    forms of uniform and two-valued rows, the shortest-prefix formulation of
    top-p through numpy's FP64 softmax and searchsorted, shift invariance at
    large logits, and -inf logits carrying no mass.
``ALL_PINS`` runs them all; test_oracle.py runs each one on the committed
oracle and test_oracle_mutants.py checks that broken copies fail some pin.
"""
from __future__ import annotations

import os

import numpy as np

from fp8_kv_cache_gb300 import workloads as W
from tests import refs

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

F64_TOL = 1e-12


def _close(a, b, tol=F64_TOL, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    err = np.max(np.abs(a - b) / (1.0 + np.abs(b))) if a.size else 0.0
    assert err <= tol, f"{what}: max rel err {err:.3e} > {tol:.1e}"


# ---------------------------------------------------------------- formats

def pin_f16_decode(o):
    """All 65536 binary16 patterns decode like numpy's float16."""
    bits = np.arange(65536, dtype=np.uint32)
    ref = bits.astype(np.uint16).view(np.float16).astype(np.float64)
    got = np.array([o.f16_to_f64(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan), "f16 NaN patterns"
    assert np.array_equal(got[~nan], ref[~nan]), "f16 values"
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan])), "f16 signs"


def _f16_encode_inputs(seed=11):
    rng = np.random.default_rng(seed)
    finite = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float64)
    mids = (finite[:-1] + finite[1:]) / 2.0               # exact ties
    near = mids * (1.0 + rng.choice([-1, 1], mids.size) * 2.0 ** -40)
    rand = rng.standard_normal(20000) * 10.0 ** rng.uniform(-9, 5, 20000)
    edge = np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e6, -1e6, 2.0 ** -24,
                     2.0 ** -25, 2.0 ** -25 * 1.0000001, 2.0 ** -14, 2.0 ** -14 * (1 - 2 ** -12),
                     np.inf, -np.inf])
    x = np.concatenate([mids, -mids, near, rand, edge])
    return x


def pin_f16_encode(o, sample=None):
    """double -> binary16 nearest-even matches numpy on ties, near-ties,
    random magnitudes and edge cases."""
    x = _f16_encode_inputs()
    if sample is not None:
        x = x[:: max(1, x.size // sample)]
    ref = x.astype(np.float16).view(np.uint16)
    got = np.array([o.f64_to_f16(float(v)) for v in x], dtype=np.uint16)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, f"f16 encode differs at {x[bad[:5]]}: {got[bad[:5]]} vs {ref[bad[:5]]}"


def pin_e4m3_library(o):
    """All 256 E4M3 codes decode like torch.float8_e4m3fn."""
    import torch
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([o.e4m3_to_f64(int(c)) for c in codes])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan), "E4M3 NaN codes"
    assert np.array_equal(got[~nan], ref[~nan]), "E4M3 values"
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan])), "E4M3 signs"


def pin_e4m3_landmarks(o):
    """Closed-form landmarks of OCP E4M3FN (bias 7, 3 mantissa bits)."""
    table = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6,
             0x38: 1.0, 0x39: 1.125, 0x40: 2.0, 0x7E: 448.0, 0xFE: -448.0, 0xB8: -1.0,
             0x77: 240.0, 0x30: 0.5}
    for c, v in table.items():
        assert o.e4m3_to_f64(c) == v, f"E4M3 code {c:#x}"
    assert np.signbit(o.e4m3_to_f64(0x80)) and o.e4m3_to_f64(0x80) == 0.0, "E4M3 -0"
    assert np.isnan(o.e4m3_to_f64(0x7F)) and np.isnan(o.e4m3_to_f64(0xFF)), "E4M3 NaN"


def pin_quantizer_nearest(o, n=4000, seed=12):
    """The generator's E4M3 encoding (torch cast after clamping) returns the
    nearest finite code by the oracle's decoder, ties to even mantissa."""
    finite = [c for c in range(256) if c not in (0x7F, 0xFF)]
    vals = np.array([o.e4m3_to_f64(c) for c in finite])
    rng = np.random.default_rng(seed)
    pos = np.unique(vals[vals >= 0])
    mids = (pos[:-1] + pos[1:]) / 2
    x = np.concatenate([rng.uniform(-448, 448, n), mids, -mids, [0.0, 448.0, -448.0]])
    x = x.astype(np.float32)
    codes = W.quantize_e4m3(x, np.float32(1.0))
    for xi, c in zip(x.astype(np.float64), codes):
        got = o.e4m3_to_f64(int(c))
        d = np.abs(vals - xi)
        best = d.min()
        assert abs(got - xi) == best, f"{xi}: code {c:#x} is not nearest"
        ties = [finite[i] for i in np.nonzero(d == best)[0] if vals[i] != 0 or xi == 0]
        if len({o.e4m3_to_f64(t) for t in ties}) > 1:
            assert (int(c) & 1) == 0, f"{xi}: tie not to even mantissa"


# ---------------------------------------------------------------- decode

def _small_cases():
    cases = [
        W.decode_case("g6_fp16", B=3, Hq=12, Hkv=2, seq_lens=[1, 37, 64], kv_dtype="fp16",
                      seed=21, D=32, page_size=8, num_pages=40),
        W.decode_case("g3_e4m3", B=2, Hq=6, Hkv=2, seq_lens=[50, 9], kv_dtype="e4m3",
                      seed=22, D=16, page_size=4, num_pages=40),
        W.decode_case("g6_e4m3_il", B=2, Hq=6, Hkv=1, seq_lens=[33, 16], kv_dtype="e4m3",
                      seed=23, D=256, page_size=16, interleaved=True, num_pages=9),
    ]
    return cases


def _run_decode(o, c, **kw):
    return o.decode(c.q, c.k, c.v, c.block_table, c.seq_lens, c.page_size, c.num_pages,
                    kw.pop("max_seq_len", c.max_seq_len), c.kv_scale, c.softmax_scale,
                    want_f64=True, **kw)


def pin_decode_dense(o):
    """Decode equals the dense numpy softmax(s q K^T) V over the unrolled table."""
    for c in _small_cases():
        _, got, flags = _run_decode(o, c)
        _close(got, refs.dense_decode(c), what=c.name)
        assert flags == 0, f"{c.name}: unexpected flags {flags}"


def pin_decode_fp16_rounding(o):
    """The FP16 output is numpy's nearest-even rounding of the FP64 output."""
    c = _small_cases()[0]
    f16, f64, _ = _run_decode(o, c)
    assert np.array_equal(f16.view(np.uint16), f64.astype(np.float16).view(np.uint16))


def pin_decode_convex(o):
    """Each output coordinate lies within the attended V values' range."""
    for c in _small_cases():
        _, got, _ = _run_decode(o, c)
        Vd = refs.lib_decode(c.v, c.kv_scale if c.kv_dtype == "e4m3" else 1.0)
        G = c.Hq // c.Hkv
        for b in range(c.B):
            Vb, _ = refs.unroll(Vd, c.block_table[b], np.arange(c.seq_lens[b]), c.page_size,
                                c.num_pages)
            for h in range(c.Hq):
                lo, hi = Vb[:, h // G].min(0), Vb[:, h // G].max(0)
                assert np.all(got[b, h] >= lo - 1e-12) and np.all(got[b, h] <= hi + 1e-12)


def pin_decode_page_permutation(o):
    """Moving pages around the pool and remapping the table changes nothing."""
    c = _small_cases()[0]
    rng = np.random.default_rng(31)
    perm = rng.permutation(c.num_pages)
    k2 = np.empty_like(c.k)
    v2 = np.empty_like(c.v)
    k2[perm] = c.k
    v2[perm] = c.v
    bt2 = perm[c.block_table].astype(np.int32)
    _, a, _ = _run_decode(o, c)
    _, b, _ = o.decode(c.q, k2, v2, bt2, c.seq_lens, c.page_size, c.num_pages, c.max_seq_len,
                       c.kv_scale, c.softmax_scale, want_f64=True)
    assert np.array_equal(a, b), "page permutation changed the output"


def pin_decode_one_token(o):
    """A one-token context returns that token's V row (then FP16-rounded)."""
    for kvd in ("fp16", "e4m3"):
        c = W.decode_case("one", B=2, Hq=6, Hkv=1, seq_lens=[1, 1], kv_dtype=kvd, seed=32,
                          D=64, page_size=16, num_pages=8)
        f16, _, _ = _run_decode(o, c)
        Vd = refs.lib_decode(c.v, c.kv_scale if kvd == "e4m3" else 1.0)
        for b in range(2):
            v0 = Vd[c.block_table[b, 0], 0, 0]
            want = v0.astype(np.float16)
            for h in range(6):
                assert np.array_equal(f16[b, h].view(np.uint16), want.view(np.uint16))


def pin_decode_equal_keys_and_zero_query(o):
    """Equal keys, or a zero query, give the plain mean of the V rows."""
    c = W.decode_case("eq", B=1, Hq=6, Hkv=1, seq_lens=[29], kv_dtype="fp16", seed=33, D=32,
                      page_size=8, num_pages=6)
    k_eq = np.broadcast_to(c.k[0, 0], c.k.shape).copy()
    _, got, _ = o.decode(c.q, k_eq, np.ascontiguousarray(c.v), c.block_table, c.seq_lens,
                         c.page_size, c.num_pages, c.max_seq_len, 1.0, c.softmax_scale,
                         want_f64=True)
    Vb, _ = refs.unroll(c.v.astype(np.float64), c.block_table[0], np.arange(29), 8, 6)
    mean = Vb[:, 0].mean(0)
    for h in range(6):
        _close(got[0, h], mean, what="equal keys")
    _, got0, _ = o.decode(np.zeros_like(c.q), c.k, c.v, c.block_table, c.seq_lens, c.page_size,
                          c.num_pages, c.max_seq_len, 1.0, c.softmax_scale, want_f64=True)
    for h in range(6):
        _close(got0[0, h], mean, what="zero query")


def pin_decode_scale_symmetry(o):
    """Doubling kv_scale and halving softmax_scale keeps the weights and
    exactly doubles the E4M3 output."""
    c = _small_cases()[1]
    _, a, _ = _run_decode(o, c)
    _, b, _ = o.decode(c.q, c.k, c.v, c.block_table, c.seq_lens, c.page_size, c.num_pages,
                       c.max_seq_len, 2 * c.kv_scale, c.softmax_scale / 2, want_f64=True)
    _close(b, 2 * a, tol=1e-13, what="scale symmetry")


def pin_decode_split_merge(o):
    """The LSE merge of the two halves of a context equals the whole."""
    c = _small_cases()[0]
    _, whole, _ = _run_decode(o, c)
    Kd = c.k.astype(np.float64)
    Vd = c.v.astype(np.float64)
    b = 2
    L = int(c.seq_lens[b])
    Kb, _ = refs.unroll(Kd, c.block_table[b], np.arange(L), c.page_size, c.num_pages)
    Vb, _ = refs.unroll(Vd, c.block_table[b], np.arange(L), c.page_size, c.num_pages)
    G = c.Hq // c.Hkv
    for h in range(c.Hq):
        qh = c.q[b, h].astype(np.float64)
        parts = [refs.lse_partial(qh, Kb[s, h // G], Vb[s, h // G], c.softmax_scale)
                 for s in (slice(0, 23), slice(23, 40), slice(40, L))]
        _close(refs.lse_merge(parts), whole[b, h], what="split/merge")


def pin_decode_inert(o):
    """Zero-length rows are zero; lengths past max_seq_len are clamped; tokens
    on out-of-range pages are skipped; each sets its flag."""
    c = _small_cases()[0]
    sl = c.seq_lens.copy()
    sl[0] = 0
    sl[1] = -5
    f16, _, fl = o.decode(c.q, c.k, c.v, c.block_table, sl, c.page_size, c.num_pages,
                          c.max_seq_len, 1.0, c.softmax_scale)
    assert np.all(f16[0] == 0) and np.all(f16[1] == 0) and fl & 4, "empty rows"
    sl = c.seq_lens.copy()
    sl[2] = 1000
    _, a, fl = o.decode(c.q, c.k, c.v, c.block_table, sl, c.page_size, c.num_pages, 64, 1.0,
                        c.softmax_scale, want_f64=True)
    sl[2] = 64
    _, b, _ = o.decode(c.q, c.k, c.v, c.block_table, sl, c.page_size, c.num_pages, 64, 1.0,
                       c.softmax_scale, want_f64=True)
    assert np.array_equal(a, b) and fl & 2, "seq_len clamp"
    # The pool holds c.num_pages pages but the call declares one fewer, so
    # entry n_valid is out of range for the method while its memory exists.
    n_valid = c.num_pages - 1
    bt = c.block_table.copy()
    bt[bt == n_valid] = 0
    bt[2, 1] = n_valid
    bt[2, 3] = -1
    bt[2, 5] = n_valid + 7
    _, got, fl = o.decode(c.q, c.k, c.v, bt, c.seq_lens, c.page_size, n_valid,
                          c.max_seq_len, 1.0, c.softmax_scale, want_f64=True)
    assert fl & 1, "bad page flag"
    Kd, Vd = c.k.astype(np.float64), c.v.astype(np.float64)
    Kb, _ = refs.unroll(Kd, bt[2], np.arange(64), c.page_size, n_valid)
    Vb, _ = refs.unroll(Vd, bt[2], np.arange(64), c.page_size, n_valid)
    assert Kb.shape[0] == 64 - 24
    G = c.Hq // c.Hkv
    for h in range(c.Hq):
        ref = refs.softmax_attention(c.q[2, h].astype(np.float64), Kb[:, h // G], Vb[:, h // G],
                                     c.softmax_scale)
        _close(got[2, h], ref, what="bad pages skipped")


def pin_gather_rows(o):
    """Gathered rows equal library-decoded rows picked by fancy indexing
    (bit-exact, float32, zero past each length)."""
    for c in _small_cases():
        for view in (c.k, c.v):
            got = o.gather_rows(view, c.block_table, c.seq_lens, c.page_size, c.num_pages,
                                c.max_seq_len, c.kv_scale)
            if c.kv_dtype == "fp16":
                vals = view.astype(np.float32)
            else:
                import torch
                vals = (torch.from_numpy(np.ascontiguousarray(view)).view(torch.float8_e4m3fn)
                        .to(torch.float32).numpy() * np.float32(c.kv_scale))
            want = np.zeros_like(got)
            for b in range(c.B):
                t = np.arange(int(min(c.seq_lens[b], c.max_seq_len)))
                want[b, t] = vals[c.block_table[b, t // c.page_size], t % c.page_size]
            assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), c.name


# ---------------------------------------------------------------- sparse prefill

def _small_prefill(seed=41, kv_dtype="fp16", interleaved=True, tails=(1, 2, 3, 4), **kw):
    args = dict(R=12, n_sel=6, first_block=10, Hq=6, Hkv=1, D=32, page_size=8)
    args.update(kw)
    return W.prefill_case("small_prefill", seed=seed, kv_dtype=kv_dtype,
                          interleaved=interleaved, tails=tails, **args)


def _run_prefill(o, c, **kw):
    return o.sparse_prefill(c.q, c.k, c.v, c.block_table, c.num_pages, c.kv_len, c.sel_idx,
                            kw.pop("q_pos", c.q_pos), c.page_size, c.softmax_scale, c.kv_scale,
                            want_f64=True, **kw)


def pin_prefill_dense(o):
    """Each row equals dense softmax attention over the row's token list as
    the page describes it (selected blocks, then the causal tail)."""
    for c in (_small_prefill(), _small_prefill(seed=42, kv_dtype="e4m3", interleaved=False),
              _small_prefill(seed=43, Hq=12, Hkv=2)):
        _, got, fl = _run_prefill(o, c)
        assert fl == 0, f"unexpected flags {fl}"
        for r in range(c.R):
            _close(got[r], refs.dense_prefill_row(c, r), what=f"prefill row {r}")


def pin_prefill_all_blocks_is_causal(o):
    """Selecting every block before the row's own block reduces to dense
    causal attention over positions 0..p."""
    c = _small_prefill(seed=44)
    own = c.q_pos // 4
    sel = np.full((c.R, int(own.max())), -1, dtype=np.int32)
    for r in range(c.R):
        sel[r, : own[r]] = np.arange(own[r])
    _, got, _ = o.sparse_prefill(c.q, c.k, c.v, c.block_table, c.num_pages, c.kv_len, sel,
                                 c.q_pos, c.page_size, c.softmax_scale, want_f64=True)
    Kd, Vd = c.k.astype(np.float64), c.v.astype(np.float64)
    for r in range(c.R):
        toks = np.arange(int(c.q_pos[r]) + 1)
        Kr, _ = refs.unroll(Kd, c.block_table, toks, c.page_size, c.num_pages)
        Vr, _ = refs.unroll(Vd, c.block_table, toks, c.page_size, c.num_pages)
        for h in range(c.Hq):
            ref = refs.softmax_attention(c.q[r, h].astype(np.float64), Kr[:, 0], Vr[:, 0],
                                         c.softmax_scale)
            _close(got[r, h], ref, what="causal special case")


def pin_prefill_equals_decode_on_gathered(o):
    """A row equals the decode oracle run on a contiguous copy of its tokens."""
    c = _small_prefill(seed=45)
    _, got, _ = _run_prefill(o, c)
    for r in (0, 5, 11):
        toks = o.sparse_row_tokens(c.block_table, c.num_pages, c.kv_len, c.sel_idx[r],
                                   c.q_pos[r], c.page_size)
        pages = c.block_table[toks // c.page_size]
        kr = np.ascontiguousarray(c.k[pages, toks % c.page_size])[:, None]   # [n,1,Hkv,D]
        vr = np.ascontiguousarray(c.v[pages, toks % c.page_size])[:, None]
        n = toks.size
        _, dec, _ = o.decode(c.q[r:r + 1], kr, vr, np.arange(n, dtype=np.int32)[None],
                             np.array([n], np.int32), 1, n, n, 1.0, c.softmax_scale,
                             want_f64=True)
        assert np.array_equal(dec[0], got[r]), "prefill row != decode over gathered copy"


def pin_prefill_token_lists(o):
    """Token lists follow the page's layout: n_sel four-token blocks then the
    causal tail; the golden file holds the counts printed on the page."""
    c = _small_prefill(seed=46)
    for r in range(c.R):
        toks = o.sparse_row_tokens(c.block_table, c.num_pages, c.kv_len, c.sel_idx[r],
                                   c.q_pos[r], c.page_size)
        want = refs.prefill_tokens(c.sel_idx[r], int(c.q_pos[r]), c.kv_len)
        assert np.array_equal(toks, want), f"row {r} token list"
    with open(os.path.join(GOLDEN, "sparse_layout.txt")) as f:
        rows = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    for n_sel, tail, count in ((int(a), int(b), int(cnt)) for a, b, cnt in rows):
        own = n_sel + 7
        sel = np.arange(n_sel, dtype=np.int32)
        p = 4 * own + tail - 1
        bt = np.arange(-(-(4 * own + 4) // 16), dtype=np.int32)
        toks = o.sparse_row_tokens(bt, bt.size, 4 * own + 4, sel, p, 16)
        assert toks.size == count, f"n_sel={n_sel} tail={tail}: {toks.size} != {count}"
        assert toks[-1] == p and np.all(np.diff(toks[-tail:]) == 1), "tail last, ending at p"


def pin_prefill_inert(o):
    """Negative positions give zero rows; positions past kv_len clamp; blocks
    at or after the row's own block are skipped; -1 entries are padding."""
    c = _small_prefill(seed=47)
    qp = c.q_pos.copy()
    qp[0] = -1
    f16, _, fl = o.sparse_prefill(c.q, c.k, c.v, c.block_table, c.num_pages, c.kv_len,
                                  c.sel_idx, qp, c.page_size, c.softmax_scale)
    assert np.all(f16[0] == 0) and fl & 4, "negative q_pos"
    qp = c.q_pos.copy()
    qp[3] = c.kv_len + 40
    _, a, fl = o.sparse_prefill(c.q, c.k, c.v, c.block_table, c.num_pages, c.kv_len, c.sel_idx,
                                qp, c.page_size, c.softmax_scale, want_f64=True)
    qp[3] = c.kv_len - 1
    _, b, _ = o.sparse_prefill(c.q, c.k, c.v, c.block_table, c.num_pages, c.kv_len, c.sel_idx,
                               qp, c.page_size, c.softmax_scale, want_f64=True)
    assert np.array_equal(a[3], b[3]) and fl & 8, "q_pos clamp"
    sel = c.sel_idx.copy()
    sel[2, 0] = c.q_pos[2] // 4          # the row's own block: skipped
    sel[2, 1] = -1                        # padding: skipped silently
    _, got, fl = o.sparse_prefill(c.q, c.k, c.v, c.block_table, c.num_pages, c.kv_len, sel,
                                  c.q_pos, c.page_size, c.softmax_scale, want_f64=True)
    assert fl == 16, f"flags {fl}"
    c2 = _small_prefill(seed=47)
    c2.sel_idx = sel
    _close(got[2], refs.dense_prefill_row(c2, 2), what="skipped blocks")


# ---------------------------------------------------------------- block selection

def _sel_positions(n_cands, rng=None):
    """q_pos values whose rows have exactly n_cands candidate blocks."""
    n_cands = np.asarray(n_cands, dtype=np.int64)
    tail = np.zeros_like(n_cands) if rng is None else rng.integers(0, 4, size=n_cands.shape)
    return (4 * n_cands + tail).astype(np.int32)


def pin_select_library(o):
    """Finite scores with many ties: the top k of the first floor(p/4) blocks
    are numpy's stable argsort of -score (equal scores keep increasing index
    order), sorted ascending."""
    rng = np.random.default_rng(61)
    R, nb = 64, 300
    sc = rng.integers(1, 40, size=(R, nb)).astype(np.float32) * 0.25   # no zeros, many ties
    sc[:, ::7] *= -1.0
    n = rng.integers(0, nb + 1, size=R)
    qp = _sel_positions(n, rng)
    for k in (1, 5, 64, 299, 400):
        got, flags = o.select_blocks(sc, qp, kv_len=4 * nb + 4, k=k)
        assert flags == 0
        for r in range(R):
            top = np.sort(np.argsort(-sc[r, :n[r]], kind="stable")[:k])
            want = np.full(k, -1, dtype=np.int32)
            want[:top.size] = top
            assert np.array_equal(got[r], want), (k, r)


def pin_select_closed_forms(o):
    """Increasing scores keep the last k candidates, decreasing the first k,
    constant rows the first k (ties go to the lower index); k >= n keeps all."""
    n, k = 50, 8
    inc = np.arange(1, n + 1, dtype=np.float32)
    sc = np.stack([inc, inc[::-1].copy(), np.full(n, 3.5, np.float32)])
    qp = _sel_positions([n, n, n])
    got, _ = o.select_blocks(sc, qp, kv_len=4 * n + 4, k=k)
    assert np.array_equal(got[0], np.arange(n - k, n)), got[0]
    assert np.array_equal(got[1], np.arange(k)), got[1]
    assert np.array_equal(got[2], np.arange(k)), got[2]
    got, _ = o.select_blocks(sc, _sel_positions([3, 0, 50]), kv_len=4 * n + 4, k=60)
    assert np.array_equal(got[0], np.r_[0, 1, 2, [-1] * 57])
    assert np.all(got[1] == -1)
    assert np.array_equal(got[2], np.r_[np.arange(50), [-1] * 10])


def pin_select_total_order(o):
    """A row holding +0, -0, +NaN, -inf, 1, -NaN, +inf, -1 (indices 0..7).
    IEEE totalOrder ranks them +NaN > +inf > 1 > +0 > -0 > -1 > -inf > -NaN,
    so the top k for k = 1..8 are, by hand:"""
    bits = np.array([0x00000000, 0x80000000, 0x7FC00000, 0xFF800000,
                     0x3F800000, 0xFFC00000, 0x7F800000, 0xBF800000], dtype=np.uint32)
    sc = bits.view(np.float32).reshape(1, 8)
    want = {1: [2], 2: [2, 6], 3: [2, 4, 6], 4: [0, 2, 4, 6], 5: [0, 1, 2, 4, 6],
            6: [0, 1, 2, 4, 6, 7], 7: [0, 1, 2, 3, 4, 6, 7], 8: list(range(8))}
    for k, w in want.items():
        got, _ = o.select_blocks(sc, _sel_positions([8]), kv_len=64, k=k)
        assert got[0].tolist() == w, (k, got[0].tolist())


def pin_select_inert(o):
    """q_pos < 0 or kv_len <= 0: a row of -1 and the empty-row bit; q_pos at or
    past kv_len is clamped to kv_len - 1 (bit 8); positions 0..3 have no
    candidate; more candidates than scores are cut to the scores (bit 32)."""
    rng = np.random.default_rng(62)
    sc = rng.standard_normal((6, 40)).astype(np.float32)
    qp = np.array([-1, 0, 3, 500, 77, 60], dtype=np.int32)
    got, flags = o.select_blocks(sc, qp, kv_len=100, k=6)
    assert flags == 4 | 8, flags
    assert np.all(got[:3] == -1)
    clamped, _ = o.select_blocks(sc[3:4], [99], kv_len=100, k=6)   # 24 candidates
    assert np.array_equal(got[3], clamped[0])
    sc[5, 39] = 100.0                                             # the best block is the last
    short, _ = o.select_blocks(sc[5:6], [159], kv_len=1000, k=6)   # 39 candidates < 50
    cut, f2 = o.select_blocks(sc[5:6], [200], kv_len=1000, k=6)    # 50 candidates > 40
    full, _ = o.select_blocks(sc[5:6], [160], kv_len=1000, k=6)    # exactly 40
    assert f2 == 32 and np.array_equal(cut, full) and not np.array_equal(short, full)
    none, f3 = o.select_blocks(sc[:2], [5, 9], kv_len=0, k=3)
    assert f3 == 4 and np.all(none == -1)


def pin_select_brute_force(o):
    """Rows of up to 7 blocks, every k: the chosen set is the only subset of
    size min(k, n) whose every member beats every non-member (higher score,
    or an equal score at a lower index), found by trying all subsets."""
    import itertools
    rng = np.random.default_rng(63)
    for trial in range(60):
        n = int(rng.integers(0, 8))
        row = rng.integers(-3, 4, size=max(n, 1)).astype(np.float32) + 0.5   # ties, no zeros
        for k in range(1, 9):
            got, _ = o.select_blocks(row.reshape(1, -1), _sel_positions([n]), kv_len=64, k=k)
            m = min(k, n)

            def beats(a, b):
                return row[a] > row[b] or (row[a] == row[b] and a < b)
            winners = [S for S in itertools.combinations(range(n), m)
                       if all(beats(a, b) for a in S for b in range(n) if b not in S)]
            assert len(winners) == 1, (n, k, winners)
            want = list(winners[0]) + [-1] * (k - m)
            assert got[0].tolist() == want, (trial, n, k, row.tolist(), got[0].tolist())


# ---------------------------------------------------------------- top-k / top-p masking

def _kept(masked):
    return [np.flatnonzero(r > -np.inf).tolist() for r in masked]


def pin_mask_topk_library(o):
    """p = 1: the kept logits are numpy's stable argsort of -x, first k
    (equal logits keep increasing index order), values unchanged."""
    rng = np.random.default_rng(71)
    x = np.round(rng.standard_normal((6, 500)) * 8).astype(np.float32) / 4   # many ties
    for k in (1, 7, 20, 499, 500, 800):
        out, _ = o.topk_topp_mask(x, k, 1.0)
        for r in range(x.shape[0]):
            want = sorted(np.argsort(-x[r], kind="stable")[:k].tolist())
            assert _kept(out[r:r + 1])[0] == want, (k, r)
            assert np.array_equal(out[r, want], x[r, want])


def pin_mask_uniform_rows(o):
    """V equal logits, no top-k cut: every logit has mass 1/V, so top-p keeps
    the first ceil(p V) indices.  Where p V is an integer and every mass is
    exact in binary (V = 4, 8), the run of exactly p V logits already reaches
    p and the next logit is not kept."""
    x = np.full((1, 25), 0.75, dtype=np.float32)
    for p, m in ((0.9, 23), (0.5, 13), (0.01, 1), (0.97, 25)):
        out, _ = o.topk_topp_mask(x, 25, p)
        assert _kept(out)[0] == list(range(m)), (p, _kept(out)[0])
    for V, p, m in ((4, 0.5, 2), (8, 0.25, 2), (8, 0.75, 6), (4, 1.0, 4)):
        out, _ = o.topk_topp_mask(np.full((1, V), -1.5, dtype=np.float32), V, p)
        assert _kept(out)[0] == list(range(m)), (V, p, _kept(out)[0])


def pin_mask_two_values(o):
    """Logits 0 and ln 3 carry mass 1/4 and 3/4: p = 0.7 keeps ln 3 alone,
    p = 0.8 keeps both; top-k 1 keeps ln 3 whatever p."""
    x = np.array([[0.0, np.log(3.0)]], dtype=np.float32)
    assert _kept(o.topk_topp_mask(x, 2, 0.7)[0])[0] == [1]
    assert _kept(o.topk_topp_mask(x, 2, 0.8)[0])[0] == [0, 1]
    assert _kept(o.topk_topp_mask(x, 1, 1.0)[0])[0] == [1]


def pin_mask_topp_prefix(o):
    """No top-k cut: the kept logits are the shortest run, in descending
    order, whose cumulative probability reaches p (numpy FP64 softmax and
    searchsorted), for rows whose decision is not within rounding of p."""
    rng = np.random.default_rng(72)
    x = (rng.standard_normal((12, 300)) * 2).astype(np.float32)
    for p in (0.3, 0.9, 0.95):
        out, margin = o.topk_topp_mask(x, 300, p)
        for r in range(x.shape[0]):
            if margin[r] < 1e-9:
                continue
            order = np.argsort(-x[r], kind="stable")
            pr = np.exp(x[r, order].astype(np.float64) - float(x[r, order[0]]))
            c = np.cumsum(pr / pr.sum())
            m = int(np.searchsorted(c, p, side="left")) + 1
            assert _kept(out[r:r + 1])[0] == sorted(order[:m].tolist()), (p, r)


def pin_mask_shift_invariance(o):
    """Adding 1024 to every logit (exact in binary32 for these values)
    changes no decision: the softmax is shift-invariant, and exp must not
    overflow."""
    rng = np.random.default_rng(73)
    x = (np.round(rng.standard_normal((8, 400)) * 64) / 64).astype(np.float32)
    a, _ = o.topk_topp_mask(x, 30, 0.9)
    b, _ = o.topk_topp_mask(x + np.float32(1024.0), 30, 0.9)
    assert _kept(a) == _kept(b)


def pin_mask_negative_infinity(o):
    """-inf logits carry no mass: in a row of 3 finite logits and -infs,
    k = 5 keeps at most the 3 finite ones; an all -inf row stays all -inf."""
    x = np.full((2, 10), -np.inf, dtype=np.float32)
    x[0, [2, 5, 7]] = [1.0, 3.0, 2.0]
    out, _ = o.topk_topp_mask(x, 5, 1.0)
    assert _kept(out)[0] == [2, 5, 7] and _kept(out)[1] == []
    out, _ = o.topk_topp_mask(x, 5, 0.5)
    assert _kept(out)[0] == [5]                 # 3.0 alone carries 0.665 >= 0.5


ALL_PINS = [
    pin_f16_decode, pin_f16_encode, pin_e4m3_library, pin_e4m3_landmarks, pin_quantizer_nearest,
    pin_decode_dense, pin_decode_fp16_rounding, pin_decode_convex, pin_decode_page_permutation,
    pin_decode_one_token, pin_decode_equal_keys_and_zero_query, pin_decode_scale_symmetry,
    pin_decode_split_merge, pin_decode_inert, pin_gather_rows,
    pin_prefill_dense, pin_prefill_all_blocks_is_causal, pin_prefill_equals_decode_on_gathered,
    pin_prefill_token_lists, pin_prefill_inert,
    pin_select_library, pin_select_closed_forms, pin_select_total_order, pin_select_inert,
    pin_select_brute_force,
    pin_mask_topk_library, pin_mask_uniform_rows, pin_mask_two_values, pin_mask_topp_prefix,
    pin_mask_shift_invariance, pin_mask_negative_infinity,
]
