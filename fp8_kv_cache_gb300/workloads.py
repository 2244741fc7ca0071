"""Seeded synthetic inputs for paged GQA decode and selected-sparse prefill.

This module only draws inputs: it holds none of the attention arithmetic and
imports neither the CUDA binding nor the CPU oracle, so both sides can take
their inputs from it.  Everything is drawn on the host with numpy's PCG64
``default_rng`` and returned as numpy arrays.

Shapes and value distributions follow the workloads the pages describe:

* decode: GQA-6 (Hq = 6 * Hkv), head dim 256, page size 16, shuffled block
  tables, FP16 KV or FP8-E4M3 KV with one per-tensor scale ("[Kernel][SM70]
  Scale NVFP4 E4M3 decode batches", Purpose and Performance contract: batch
  1..16, 1K and 16K contexts);
* sparse prefill: Hq6/Hkv1/D256 FP16, 4096 query rows, each attending to 512
  selected four-token blocks plus a causal tail of 1..3 tokens, contiguous or
  interleaved K/V ("[Kernel][SM70] Accelerate Qwen3.8 QSA paged prefill",
  Changes and Test Result);
* top-k/top-p masking: float32 logits of B8/B16 x 248,320 ("[Kernel][SM70]
  Scale NVFP4 E4M3 decode batches", Purpose; top-k 20, top-p 0.95 from its
  Performance contract).  No trained model is at hand: each row is
  N(0, 2.5^2) with 32 positions raised by U(5, 15), so a handful of logits
  carry most of the mass, as in a language model's next-token distribution;
* block selection: float32 block scores of the same 4096 rows, from which 512
  blocks per row are selected ("[Kernel][SM70] Accelerate exact Qwen3.8
  decode", Implementation).  The pages' scores come from a trained scorer,
  which is out of reach here; the stand-in draws N(0,1) values rounded to
  bfloat16 precision (through torch's bfloat16 cast), so equal scores at the
  selection pivot are common, as the page's tie rule anticipates.

E4M3 quantisation of the drawn values uses torch's float8_e4m3fn cast (a
library routine; round to nearest even) after dividing by the per-tensor scale
and clamping to the largest finite magnitude 448, so that no code is NaN.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

E4M3_MAX = 448.0


@dataclass
class DecodeCase:
    """One batched-decode input.  ``kv`` is the backing buffer; ``k`` and ``v``
    are 4-D views [num_pages, page_size, Hkv, D] into it (contiguous pools or
    one interleaved buffer)."""
    name: str
    q: np.ndarray                 # float16 [B, Hq, D]
    kv: np.ndarray                # uint8 (E4M3 codes) or float16 backing buffer
    k: np.ndarray
    v: np.ndarray
    kv_dtype: str                 # "fp16" | "e4m3"
    block_table: np.ndarray       # int32 [B, max_pages]
    seq_lens: np.ndarray          # int32 [B]
    page_size: int
    num_pages: int
    max_seq_len: int
    kv_scale: float               # float32-representable; 1.0 for FP16 KV
    softmax_scale: float
    interleaved: bool = False
    meta: dict = field(default_factory=dict)

    @property
    def B(self):
        return self.q.shape[0]

    @property
    def Hq(self):
        return self.q.shape[1]

    @property
    def Hkv(self):
        return self.k.shape[2]

    @property
    def D(self):
        return self.q.shape[2]


@dataclass
class PrefillCase:
    """One selected-sparse prefill input over a single sequence."""
    name: str
    q: np.ndarray                 # float16 [R, Hq, D]
    kv: np.ndarray
    k: np.ndarray                 # 4-D views [num_pages, page_size, Hkv, D]
    v: np.ndarray
    kv_dtype: str
    block_table: np.ndarray       # int32 [pages of this sequence]
    num_pages: int
    kv_len: int
    sel_idx: np.ndarray           # int32 [R, n_sel] four-token block ids
    q_pos: np.ndarray             # int32 [R]
    page_size: int
    kv_scale: float
    softmax_scale: float
    interleaved: bool = False
    meta: dict = field(default_factory=dict)

    @property
    def R(self):
        return self.q.shape[0]

    @property
    def Hq(self):
        return self.q.shape[1]

    @property
    def Hkv(self):
        return self.k.shape[2]

    @property
    def D(self):
        return self.q.shape[2]

    @property
    def n_sel(self):
        return self.sel_idx.shape[1]


# --------------------------------------------------------------------------
# value draws
# --------------------------------------------------------------------------

def _normal(rng, shape, scale=1.0):
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if scale != 1.0:
        x *= np.float32(scale)
    return x


def quantize_e4m3(x: np.ndarray, scale: np.float32) -> np.ndarray:
    """E4M3FN codes (uint8) of x / scale, clamped to +-448, nearest-even."""
    import torch  # CPU-only use: the library cast that encodes E4M3
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    t = (t / float(scale)).clamp_(-E4M3_MAX, E4M3_MAX)
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _kv_pools(rng, num_pages, page_size, Hkv, D, kv_dtype, value_scale, interleaved):
    """Draw K and V (N(0,1) * value_scale) and store them as FP16 or E4M3.
    Returns (backing buffer, k view, v view, kv_scale)."""
    shape = (num_pages, page_size, Hkv, D)
    kf = _normal(rng, shape, value_scale)
    vf = _normal(rng, shape, value_scale)
    if kv_dtype == "fp16":
        kq, vq, scale = kf.astype(np.float16), vf.astype(np.float16), 1.0
    elif kv_dtype == "e4m3":
        amax = max(float(np.abs(kf).max()), float(np.abs(vf).max()))
        scale = np.float32(amax / E4M3_MAX)
        kq, vq = quantize_e4m3(kf, scale), quantize_e4m3(vf, scale)
        scale = float(scale)
    else:
        raise ValueError(kv_dtype)
    del kf, vf
    if interleaved:
        buf = np.empty((num_pages, page_size, Hkv, 2, D), dtype=kq.dtype)
        buf[:, :, :, 0, :] = kq
        buf[:, :, :, 1, :] = vq
        return buf, buf[:, :, :, 0, :], buf[:, :, :, 1, :], scale
    buf = np.stack([kq, vq])            # [2, pages, P, Hkv, D]
    return buf, buf[0], buf[1], scale


def _block_tables(rng, B, max_pages, num_pages):
    """A seeded permutation of the pool cut into each sequence's pages."""
    if B * max_pages > num_pages:
        raise ValueError("pool too small for the block tables")
    perm = rng.permutation(num_pages).astype(np.int32)
    return np.ascontiguousarray(perm[: B * max_pages].reshape(B, max_pages))


# --------------------------------------------------------------------------
# decode cases
# --------------------------------------------------------------------------

def decode_case(name, *, B, Hq, Hkv, seq_lens, kv_dtype, seed, D=256, page_size=16,
                num_pages=None, max_seq_len=None, value_scale=None, interleaved=False,
                softmax_scale=None):
    rng = np.random.default_rng(seed)
    seq_lens = np.asarray(seq_lens, dtype=np.int32).reshape(B)
    if max_seq_len is None:
        max_seq_len = int(max(1, seq_lens.max()))
    max_pages = -(-max_seq_len // page_size)
    if num_pages is None:
        num_pages = B * max_pages
    if value_scale is None:
        value_scale = 2.0 if kv_dtype == "e4m3" else 1.0
    block_table = _block_tables(rng, B, max_pages, num_pages)
    q = _normal(rng, (B, Hq, D)).astype(np.float16)
    kv, k, v, scale = _kv_pools(rng, num_pages, page_size, Hkv, D, kv_dtype, value_scale,
                                interleaved)
    return DecodeCase(name=name, q=q, kv=kv, k=k, v=v, kv_dtype=kv_dtype,
                      block_table=block_table, seq_lens=seq_lens, page_size=page_size,
                      num_pages=num_pages, max_seq_len=max_seq_len, kv_scale=scale,
                      softmax_scale=float(softmax_scale if softmax_scale is not None
                                          else 1.0 / np.sqrt(D)),
                      interleaved=interleaved)


def tiny_fp16(seed=1):
    """B=1, Hkv=1, Hq=6, D=256, 64 tokens in 4 pages of 16 taken from a
    seeded permutation of a 16-page pool; FP16 N(0,1); softmax_scale 1/16."""
    return decode_case("tiny_fp16_b1_l64", B=1, Hq=6, Hkv=1, seq_lens=[64], kv_dtype="fp16",
                       seed=seed, num_pages=16)


def e4m3_b8(seed=2):
    """B=8, Hkv=4, Hq=24, 1024 tokens each, shuffled 512-page pool, E4M3 KV
    from N(0,1)*2 with a per-tensor scale."""
    return decode_case("e4m3_b8_l1024", B=8, Hq=24, Hkv=4, seq_lens=[1024] * 8, kv_dtype="e4m3",
                       seed=seed)


def long_e4m3(seed=3, B=16, page_size=16):
    """B=16, Hkv=4, Hq=24, seq_lens uniform in [12288, 16384], shuffled pool of
    16384 pages of 16 (or the same tokens in pages of page_size), E4M3 KV from
    N(0,1)*2."""
    rng = np.random.default_rng(seed + 1000)
    lens = rng.integers(12288, 16384, size=B, endpoint=True).astype(np.int32)
    pages = B * (-(-16384 // page_size))
    suffix = "" if page_size == 16 else f"_p{page_size}"
    return decode_case(f"long_e4m3_b{B}{suffix}", B=B, Hq=24, Hkv=4, seq_lens=lens,
                       kv_dtype="e4m3", seed=seed, max_seq_len=16384, num_pages=pages,
                       page_size=page_size)


def sweep(B, L, kv_dtype, seed=4):
    """Batch sweep point: Hkv=4, Hq=24, every sequence L tokens, pool of
    B*L/16 pages, N(0,1) values for both FP16 and E4M3 KV."""
    return decode_case(f"sweep_{kv_dtype}_b{B}_l{L}", B=B, Hq=24, Hkv=4, seq_lens=[L] * B,
                       kv_dtype=kv_dtype, seed=seed, value_scale=1.0)


# --------------------------------------------------------------------------
# sparse prefill cases
# --------------------------------------------------------------------------

def prefill_case(name, *, R, n_sel, seed, first_block, Hq=6, Hkv=1, D=256, page_size=16,
                 kv_len=None, kv_dtype="fp16", interleaved=True, tails=(1, 2, 3),
                 value_scale=1.0, softmax_scale=None):
    """Row r owns block c_r = first_block + r and sits at position
    p_r = 4*c_r + t_r - 1 with t_r drawn from ``tails``; it selects ``n_sel``
    distinct blocks drawn uniformly from [0, c_r), sorted ascending."""
    rng = np.random.default_rng(seed)
    if first_block < n_sel:
        raise ValueError("first_block must leave room for n_sel earlier blocks")
    c = first_block + np.arange(R, dtype=np.int64)
    t = rng.choice(np.asarray(tails, dtype=np.int64), size=R)
    q_pos = (4 * c + t - 1).astype(np.int32)
    need = int(4 * c[-1] + 4)
    if kv_len is None:
        kv_len = need
    kv_len = max(kv_len, need)
    num_pages = -(-kv_len // page_size)
    sel = np.empty((R, n_sel), dtype=np.int32)
    for r in range(R):
        sel[r] = np.sort(rng.choice(int(c[r]), size=n_sel, replace=False))
    block_table = rng.permutation(num_pages).astype(np.int32)
    q = _normal(rng, (R, Hq, D)).astype(np.float16)
    kv, k, v, scale = _kv_pools(rng, num_pages, page_size, Hkv, D, kv_dtype, value_scale,
                                interleaved)
    return PrefillCase(name=name, q=q, kv=kv, k=k, v=v, kv_dtype=kv_dtype,
                       block_table=block_table, num_pages=num_pages, kv_len=kv_len,
                       sel_idx=sel, q_pos=q_pos, page_size=page_size, kv_scale=scale,
                       softmax_scale=float(softmax_scale if softmax_scale is not None
                                           else 1.0 / np.sqrt(D)),
                       interleaved=interleaved)


def sparse_prefill_4096(seed=5, interleaved=True, R=4096, kv_dtype="fp16"):
    """4096 rows, Hq6/Hkv1/D256 FP16 (or E4M3 KV with a per-tensor scale), a
    32768-token cache in 2048 shuffled pages of 16; row r owns block 4096 + r
    (positions >= 16384 > 2051) and attends to 512 selected blocks plus a tail
    of 1..3 tokens."""
    suffix = "" if kv_dtype == "fp16" else f"_{kv_dtype}"
    return prefill_case(f"sparse_prefill_r{R}{suffix}", R=R, n_sel=512, seed=seed,
                        first_block=4096, kv_len=32768, interleaved=interleaved, kv_dtype=kv_dtype)


@dataclass
class SelectCase:
    """Inputs of one block-selection call: scores [R, score_stride] float32
    (the first n_blocks columns are used), q_pos int32 [R]."""
    name: str
    scores: np.ndarray
    q_pos: np.ndarray
    kv_len: int
    k: int
    n_blocks: int


def select_case(name, *, R, n_blocks, k, seed, kv_len=None, first_block=None, q_pos=None,
                score_stride=None, bf16_ties=True):
    """Scores N(0,1) (rounded to bfloat16 precision when ``bf16_ties``) for R
    rows; row r sits at q_pos[r] (default: owns block first_block + r with a
    tail of 1..3 tokens, as in the prefill workload)."""
    rng = np.random.default_rng(seed)
    stride = n_blocks if score_stride is None else score_stride
    x = rng.standard_normal((R, stride)).astype(np.float32)
    if bf16_ties:
        import torch
        x = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    if q_pos is None:
        fb = k if first_block is None else first_block
        own = fb + np.arange(R, dtype=np.int64)
        q_pos = 4 * own + rng.integers(0, 3, size=R)
    q_pos = np.asarray(q_pos, dtype=np.int32).reshape(R)
    if kv_len is None:
        kv_len = int(q_pos.max()) + 1 if R else 1
    return SelectCase(name=name, scores=np.ascontiguousarray(x), q_pos=q_pos, kv_len=int(kv_len),
                      k=int(k), n_blocks=int(n_blocks))


def qsa_select_4096(seed=6, R=4096):
    """The 4096 rows of the sparse-prefill workload (row r owns block
    4096 + r, 32768-token cache, so 8192 blocks): select 512 of the blocks
    before each row's own, from bfloat16-precision N(0,1) scores."""
    return select_case(f"qsa_select_r{R}", R=R, n_blocks=8192, k=512, seed=seed, kv_len=32768,
                       first_block=4096)


@dataclass
class MaskCase:
    """Inputs of one top-k/top-p masking call: logits float32 [B, V]."""
    name: str
    logits: np.ndarray
    k: int
    p: float


def logits_case(name, *, B, V=248320, k=20, p=0.95, seed=7, peaks=32):
    """B rows of V logits: N(0, 2.5^2) plus U(5, 15) at ``peaks`` random
    positions per row."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((B, V)).astype(np.float32) * np.float32(2.5)
    for b in range(B):
        idx = rng.choice(V, size=min(peaks, V), replace=False)
        x[b, idx] += rng.uniform(5.0, 15.0, size=idx.size).astype(np.float32)
    return MaskCase(name=name, logits=x, k=int(k), p=float(p))


def sampler_b16(seed=7):
    """B=16 rows of 248,320 logits, top-k 20, top-p 0.95."""
    return logits_case("topk_topp_b16", B=16, seed=seed)
