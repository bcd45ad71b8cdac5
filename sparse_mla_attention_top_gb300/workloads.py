"""Seeded synthetic inputs for sparse MLA decode and grouped prefill.

This module only draws inputs: block tables, top-k position lists, query and cache
contents. It holds none of the attention arithmetic, so both the CUDA library's tests and
the CPU oracle can consume the same bytes without sharing any of the method's code.

Shapes and distributions follow the workloads the pages measure on (real GLM-5.2 top-k
dumps and public text there, neither of which is available here; these generators stand in
for them):

* rows are 576 wide: 512 latent + 64 rope (vLLM PR #63104, bench script);
* q and the cache are N(0, 1) rounded to bf16;
* the fp8 cache stores 512 e4m3 codes, 4 fp32 scales (one per 128 channels, U[0.5, 2]) and
  64 bf16 rope values per row: 656 bytes;
* physical pages are a seeded permutation, so consecutive positions of a request land on
  scattered pages;
* decode top-k lists are distinct uniform positions in [0, ctx), in random order, padded
  with -1 when ctx < K;
* prefill lists: query i of the new tokens selects from its causal prefix; when the prefix
  holds at most K positions it takes them all, otherwise it keeps a uniform 70% of its
  predecessor's list and fills the rest with distinct new positions (neighbouring queries
  overlap, as the pages report for real top-k);
* indexer scores (the input of top-k selection): fp32 N(0, 1) values rounded to bf16
  precision, so equal scores occur as they do for a low-precision indexer, one row per
  query over its context (contexts as for the decode batch).
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

LATENT = 512
ROPE = 64
ROW = LATENT + ROPE
ROW_BYTES_BF16 = ROW * 2
ROW_BYTES_FP8 = LATENT + 16 + ROPE * 2  # 656
KV_BF16 = 0
KV_FP8_E4M3 = 1


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest even) and return the bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> 16) & 1) + np.uint32(0x7FFF)
    return ((u + bias) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


_CHUNK = 1 << 22


def _chunked(rng: np.random.Generator, n: int, fill) -> None:
    """Calls fill(sub_rng, start, end) for consecutive chunks of n items, in parallel threads.
    Chunk i draws from its own PCG64 stream seeded by (a number drawn from rng, i), so the
    bytes depend only on rng's state, not on the thread count."""
    from concurrent.futures import ThreadPoolExecutor
    import os

    base = int(rng.integers(0, 2 ** 63 - 1))
    chunks = (n + _CHUNK - 1) // _CHUNK

    def job(i):
        fill(np.random.default_rng([base, i]), i * _CHUNK, min(n, (i + 1) * _CHUNK))

    if chunks <= 1:
        for i in range(chunks):
            job(i)
        return
    with ThreadPoolExecutor(min(chunks, os.cpu_count() or 1, 32)) as ex:
        list(ex.map(job, range(chunks)))


def _normal_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, np.uint16)

    def fill(r, s, e):
        out[s:e] = f32_to_bf16_bits(r.standard_normal(e - s, dtype=np.float32))

    _chunked(rng, n, fill)
    return out.reshape(shape)


def _e4m3_codes(x: np.ndarray) -> np.ndarray:
    """Saturating round-to-nearest-even e4m3 codes of float32 values (via torch's cast)."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).clamp_(-448.0, 448.0)
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()


def make_cache(rng: np.random.Generator, num_rows: int, kv_dtype: int) -> np.ndarray:
    """Cache bytes [num_rows, row_bytes] (uint8)."""
    if kv_dtype == KV_BF16:
        return _normal_bf16(rng, (num_rows, ROW)).view(np.uint8).reshape(num_rows, ROW_BYTES_BF16)
    out = np.empty((num_rows, ROW_BYTES_FP8), np.uint8)
    rows_per_chunk = max(1, _CHUNK // LATENT)

    def fill(r, s, e):
        # rows s .. e-1 of this chunk: latent codes, block scales, rope
        out[s:e, :LATENT] = _e4m3_codes(r.standard_normal((e - s, LATENT), dtype=np.float32))
        scales = r.uniform(0.5, 2.0, size=(e - s, 4)).astype(np.float32)
        out[s:e, LATENT:LATENT + 16] = scales.view(np.uint8).reshape(e - s, 16)
        rope = f32_to_bf16_bits(r.standard_normal((e - s) * ROPE, dtype=np.float32))
        out[s:e, LATENT + 16:] = rope.view(np.uint8).reshape(e - s, ROPE * 2)

    base = int(rng.integers(0, 2 ** 63 - 1))
    from concurrent.futures import ThreadPoolExecutor
    import os

    chunks = (num_rows + rows_per_chunk - 1) // rows_per_chunk

    def job(i):
        fill(np.random.default_rng([base, i]), i * rows_per_chunk, min(num_rows, (i + 1) * rows_per_chunk))

    with ThreadPoolExecutor(max(1, min(chunks, os.cpu_count() or 1, 32))) as ex:
        list(ex.map(job, range(chunks)))
    return out


def _paged_requests(rng: np.random.Generator, ctxs, page_size: int, spare_pages: int = 0):
    """Block table [R, max_blocks] over a shuffled pool of physical pages (-1 past each request)."""
    pages = [math.ceil(c / page_size) for c in ctxs]
    total = int(sum(pages)) + spare_pages
    perm = rng.permutation(total).astype(np.int32)
    max_blocks = max(1, max(pages))
    bt = np.full((len(ctxs), max_blocks), -1, np.int32)
    off = 0
    for r, p in enumerate(pages):
        bt[r, :p] = perm[off:off + p]
        off += p
    return bt, total


@dataclass
class DecodeWorkload:
    """One decode batch: query t belongs to request req_of_token[t] (the identity here)."""
    name: str
    T: int
    H: int
    K: int
    page_size: int
    num_pages: int
    kv_dtype: int
    kv: np.ndarray              # [num_pages * page_size, row_bytes] uint8
    q_bits: np.ndarray          # [T, H, 576] uint16 (bf16 patterns)
    block_table: np.ndarray     # [R, max_blocks] int32
    seq_lens: np.ndarray        # [R] int32
    req_of_token: np.ndarray    # [T] int32
    topk: np.ndarray            # [T, K] int32 positions, -1 padded
    topk_len: Optional[np.ndarray]
    scale: float
    seed: int = 0
    info: dict = field(default_factory=dict)

    @property
    def row_bytes(self) -> int:
        return self.kv.shape[1]

    @property
    def num_slots(self) -> int:
        return self.num_pages * self.page_size


def make_decode(seed: int, T: int, H: int, K: int, ctx_lo: int, ctx_hi: int, page_size: int,
                kv_dtype: int = KV_BF16, scale: Optional[float] = None, name: str = "decode",
                identity_pages: bool = False) -> DecodeWorkload:
    """T requests with one decode query each; ctx uniform in [ctx_lo, ctx_hi]."""
    rng = np.random.default_rng(seed)
    ctxs = rng.integers(ctx_lo, ctx_hi + 1, size=T)
    bt, total_pages = _paged_requests(rng, ctxs, page_size)
    if identity_pages:
        # pages in order, request after request (used for the dense-layout checks)
        off = 0
        for r, c in enumerate(ctxs):
            p = math.ceil(c / page_size)
            bt[r, :p] = np.arange(off, off + p, dtype=np.int32)
            off += p
    kv = make_cache(rng, total_pages * page_size, kv_dtype)
    q_bits = _normal_bf16(rng, (T, H, ROW))
    topk = np.full((T, K), -1, np.int32)
    for t in range(T):
        n = min(K, int(ctxs[t]))
        topk[t, :n] = rng.choice(int(ctxs[t]), size=n, replace=False).astype(np.int32)
    return DecodeWorkload(name=name, T=T, H=H, K=K, page_size=page_size, num_pages=total_pages,
                          kv_dtype=kv_dtype, kv=kv, q_bits=q_bits, block_table=bt,
                          seq_lens=ctxs.astype(np.int32), req_of_token=np.arange(T, dtype=np.int32),
                          topk=topk, topk_len=None, scale=(ROW ** -0.5) if scale is None else scale,
                          seed=seed, info={"ctx": ctxs})


@dataclass
class PrefillWorkload:
    """One request of n_new new tokens on n_cached cached ones; query i sits at position
    n_cached + i and selects only from [0, n_cached + i]."""
    name: str
    T: int
    H: int
    G: int
    K: int
    page_size: int
    num_pages: int
    kv_dtype: int
    kv: np.ndarray
    q_bits: np.ndarray          # [T, H, 576]
    block_table: np.ndarray     # [1, max_blocks]
    seq_lens: np.ndarray        # [1]
    req_of_token: np.ndarray    # [T] zeros
    topk: np.ndarray            # [T, K] positions, -1 padded
    topk_len: Optional[np.ndarray]
    scale: float
    seed: int = 0

    @property
    def row_bytes(self) -> int:
        return self.kv.shape[1]

    @property
    def num_slots(self) -> int:
        return self.num_pages * self.page_size


def neighbour_topk(rng: np.random.Generator, n_new: int, n_cached: int, K: int, keep_frac: float = 0.7):
    """Top-k position lists [n_new, K] whose neighbours overlap by about keep_frac."""
    topk = np.full((n_new, K), -1, np.int32)
    prev = None
    keep_n = int(round(keep_frac * K))
    for i in range(n_new):
        cand = n_cached + i + 1  # positions 0 .. n_cached + i
        if cand <= K:
            sel = rng.permutation(cand).astype(np.int32)
            topk[i, :cand] = sel
            prev = sel
            continue
        if prev is None or len(prev) < K:
            if prev is None:
                sel = rng.choice(cand, size=K, replace=False).astype(np.int32)
            else:
                keep = rng.choice(prev, size=min(keep_n, len(prev)), replace=False)
                sel = _fill(rng, keep, cand, K)
        else:
            keep = rng.choice(prev, size=keep_n, replace=False)
            sel = _fill(rng, keep, cand, K)
        sel = rng.permutation(sel).astype(np.int32)
        topk[i] = sel
        prev = sel
    return topk


def _fill(rng, keep: np.ndarray, cand: int, K: int) -> np.ndarray:
    need = K - len(keep)
    if cand <= 4 * K:
        pool = np.setdiff1d(np.arange(cand, dtype=np.int64), keep, assume_unique=True)
        new = rng.choice(pool, size=need, replace=False)
    else:
        taken = set(int(x) for x in keep)
        new = []
        while len(new) < need:
            for x in rng.integers(0, cand, size=2 * (need - len(new))):
                x = int(x)
                if x not in taken:
                    taken.add(x)
                    new.append(x)
                    if len(new) == need:
                        break
        new = np.asarray(new, np.int64)
    return np.concatenate([keep.astype(np.int64), new])


def make_prefill(seed: int, n_new: int, n_cached: int, H: int, G: int, K: int, page_size: int,
                 kv_dtype: int = KV_BF16, scale: Optional[float] = None, name: str = "prefill",
                 keep_frac: float = 0.7) -> PrefillWorkload:
    rng = np.random.default_rng(seed)
    ctx = n_cached + n_new
    bt, total_pages = _paged_requests(rng, [ctx], page_size)
    kv = make_cache(rng, total_pages * page_size, kv_dtype)
    q_bits = _normal_bf16(rng, (n_new, H, ROW))
    topk = neighbour_topk(rng, n_new, n_cached, K, keep_frac)
    return PrefillWorkload(name=name, T=n_new, H=H, G=G, K=K, page_size=page_size, num_pages=total_pages,
                           kv_dtype=kv_dtype, kv=kv, q_bits=q_bits, block_table=bt,
                           seq_lens=np.array([ctx], np.int32), req_of_token=np.zeros(n_new, np.int32),
                           topk=topk, topk_len=None, scale=(ROW ** -0.5) if scale is None else scale, seed=seed)


# The five workloads of the benchmark, by name (sizes as stated in each description).

def tiny_decode() -> DecodeWorkload:
    """1 request, 8 heads, context 256, page_size 1 over a shuffled 256-page pool, 64 distinct
    positions, scale 1/sqrt(256), seed 0."""
    rng = np.random.default_rng(0)
    bt = rng.permutation(256).astype(np.int32)[None, :]
    kv = make_cache(rng, 256, KV_BF16)
    q_bits = _normal_bf16(rng, (1, 8, ROW))
    topk = rng.choice(256, size=64, replace=False).astype(np.int32)[None, :]
    return DecodeWorkload(name="tiny_decode_h8_k64_ctx256_p1", T=1, H=8, K=64, page_size=1, num_pages=256,
                          kv_dtype=KV_BF16, kv=kv, q_bits=q_bits, block_table=bt,
                          seq_lens=np.array([256], np.int32), req_of_token=np.zeros(1, np.int32), topk=topk,
                          topk_len=None, scale=1.0 / 16.0, seed=0)


def decode_bf16_batch(T: int = 64) -> DecodeWorkload:
    """64 requests x 64 heads, bf16 cache, page_size 64, contexts U{8192..32768}, top-k 2048."""
    return make_decode(1, T=T, H=64, K=2048, ctx_lo=8192, ctx_hi=32768, page_size=64, kv_dtype=KV_BF16,
                       name=f"decode_bf16_t{T}_h64_k2048_ctx8k-32k_p64")


def decode_fp8_batch(T: int = 128) -> DecodeWorkload:
    """128 requests x 64 heads, e4m3 latent + fp32 block scales + bf16 rope, contexts U{4096..47104}."""
    return make_decode(2, T=T, H=64, K=2048, ctx_lo=4096, ctx_hi=47104, page_size=64, kv_dtype=KV_FP8_E4M3,
                       name=f"decode_fp8_t{T}_h64_k2048_ctx4k-46k_p64")


def grouped_prefill(n_new: int = 8192) -> PrefillWorkload:
    """One request of 8192 new causal tokens, 64 heads, groups of 2, page_size 64, top-k 2048."""
    return make_prefill(3, n_new=n_new, n_cached=0, H=64, G=2, K=2048, page_size=64,
                        name=f"prefill_bf16_t{n_new}_h64_g2_k2048_p64")


def grouped_prefill_fp8(n_new: int = 8192) -> PrefillWorkload:
    """The 8192-token grouped prefill (64 heads, groups of 2) over an e4m3 cache."""
    return make_prefill(8, n_new=n_new, n_cached=0, H=64, G=2, K=2048, page_size=64, kv_dtype=KV_FP8_E4M3,
                        name=f"prefill_fp8_t{n_new}_h64_g2_k2048_p64")


def mixed_prefill(n_new: int = 8192) -> PrefillWorkload:
    """8192 new tokens on 24576 cached, 16 heads, groups of 8, page_size 64, top-k 2048."""
    return make_prefill(4, n_new=n_new, n_cached=24576, H=16, G=8, K=2048, page_size=64,
                        name=f"prefill_bf16_t{n_new}_c24576_h16_g8_k2048_p64")


def mixed_decode(T: int = 128) -> DecodeWorkload:
    """128 decodes of 16 heads, contexts U{16384..47104}, top-k 2048, bf16, page_size 64."""
    return make_decode(5, T=T, H=16, K=2048, ctx_lo=16384, ctx_hi=47104, page_size=64, kv_dtype=KV_BF16,
                       name=f"decode_bf16_t{T}_h16_k2048_ctx16k-46k_p64")


def dense_check() -> DecodeWorkload:
    """1 request at context 4096 with top-k = all 4096 positions (random order), 16 heads."""
    w = make_decode(6, T=1, H=16, K=4096, ctx_lo=4096, ctx_hi=4096, page_size=64, kv_dtype=KV_BF16,
                    name="dense_check_h16_ctx4096_p64")
    return w


@dataclass
class TopkWorkload:
    """Indexer scores for top-k selection: query t's candidates are positions 0..lens[t]-1."""
    name: str
    T: int
    N: int
    K: int
    scores: np.ndarray  # [T, N] float32
    lens: np.ndarray    # [T] int32
    seed: int


def make_topk(seed: int, T: int, K: int, ctx_lo: int, ctx_hi: int) -> TopkWorkload:
    rng = np.random.default_rng(seed)
    lens = rng.integers(ctx_lo, ctx_hi + 1, size=T).astype(np.int32)
    N = int(lens.max())
    scores = bf16_bits_to_f32(f32_to_bf16_bits(rng.standard_normal((T, N), dtype=np.float32)))
    return TopkWorkload(name=f"topk_t{T}_k{K}_ctx{ctx_lo}-{ctx_hi}", T=T, N=N, K=K, scores=scores, lens=lens,
                        seed=seed)


def topk_batch(T: int = 64) -> TopkWorkload:
    """The decode batch's selection: 64 queries, contexts 8K-32K, K = 2048."""
    return make_topk(7, T=T, K=2048, ctx_lo=8192, ctx_hi=32768)
