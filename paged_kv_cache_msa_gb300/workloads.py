"""Seeded synthetic inputs for the MSA fused producer.

This module only *makes inputs*: projection rows, positions, slot mappings, page
tables, norm weights, scales and cache layouts (with sentinel-filled pools and guard
bands).  It holds none of the producer's arithmetic, and both the CUDA path's tests
and the CPU oracle draw their inputs from it.

The shapes follow the pages' workloads: MiniMax-M3 MSA with 64 query heads, 8 K/V
heads, 8 index-Q heads and one index-K head of dim 128 (the "big" shapes), a small
variant with 8/2/2/1 heads of dim 64 (the "tiny" shapes), page size 64, fp8 E4M3
K/V caches in head-major (HND) pages, and decode, prefill and mixed batches.  The
pages measure on serving prompt sets that are not available here; these seeded
workloads stand in for them ("[None][perf] Fuse MiniMax-M3 MSA per-layer KV-cache
writes into one kernel", "Measured impact"; "[None][perf] Fuse MiniMax-M3 QKV and
index projection", "Performance").

Random streams: NumPy PCG64 seeded with 1000 * config + layer.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

DTYPE_BF16 = 0
DTYPE_E4M3 = 1
ELEM_SIZE = {DTYPE_BF16: 2, DTYPE_E4M3: 1}

ROPE_NEOX = 0
ROPE_GPTJ = 1

GUARD_BYTES = 4096          # sentinel bytes before and after every pool

TINY = dict(num_q_heads=8, num_kv_heads=2, num_idx_q_heads=2, num_idx_k_heads=1, head_dim=64)
BIG = dict(num_q_heads=64, num_kv_heads=8, num_idx_q_heads=8, num_idx_k_heads=1, head_dim=128)


@dataclass
class CacheSpec:
    """One paged cache: a strided view into a named pool allocation."""
    pool: str
    offset: int            # bytes from the pool's first byte to element 0
    dtype: int
    num_pages: int
    num_heads: int
    stride_page: int       # elements
    stride_head: int       # elements
    stride_token: int      # elements (the dim stride is 1)

    def elem_size(self) -> int:
        return ELEM_SIZE[self.dtype]


@dataclass
class Workload:
    name: str
    shape: dict
    qkv: np.ndarray                 # uint16 (bf16 bits) [T, row_stride]
    row_stride: int
    positions: np.ndarray           # int32 [T]
    slot_mapping: np.ndarray        # int64 [T]
    page_table: np.ndarray | None   # int32 [S, max_blocks]
    weights: dict                   # q/k/idx_q/idx_k -> uint16 [D]
    scales: np.ndarray              # float32
    caches: dict                    # k/v/idx_k -> CacheSpec | None
    pools: dict                     # pool name -> size in bytes (guards included)
    seed: int = 0
    meta: dict = field(default_factory=dict)

    @property
    def num_tokens(self) -> int:
        return int(self.positions.shape[0])

    @property
    def width(self) -> int:
        s = self.shape
        return (s["num_q_heads"] + 2 * s["num_kv_heads"] + s["num_idx_q_heads"]
                + s["num_idx_k_heads"]) * s["head_dim"]

    def algorithmic_bytes(self) -> int:
        """Bytes a producer must move: the rows' W bf16 values, position, slot and one
        page-table entry read per token; compact Q/idx-Q and the cache rows written
        for each token whose slot is valid."""
        s, T = self.shape, self.num_tokens
        D = s["head_dim"]
        read = T * (2 * self.width + 4 + 8 + (4 if self.page_table is not None else 0))
        write = T * 2 * D * (s["num_q_heads"] + s["num_idx_q_heads"])
        nvalid = int(self.meta.get("num_valid", T))
        for key, heads in (("k", s["num_kv_heads"]), ("v", s["num_kv_heads"]),
                           ("idx_k", s["num_idx_k_heads"])):
            c = self.caches.get(key)
            if c is not None:
                write += nvalid * heads * D * c.elem_size()
        return read + write


# ----------------------------------------------------------------------------
# value generators
# ----------------------------------------------------------------------------

def _to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns via torch's rounding cast (input preparation)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def _normal_bf16(rng: np.random.Generator, shape, outlier_frac=0.0, outlier_mult=20.0,
                 chunk_rows=4096) -> np.ndarray:
    """N(0,1) values rounded to bf16; a seeded fraction of elements times outlier_mult."""
    shape = tuple(int(v) for v in shape)
    out = np.empty(shape, dtype=np.uint16)
    rows = shape[0]
    flat_cols = int(np.prod(shape[1:])) if len(shape) > 1 else 1
    out2 = out.reshape(rows, flat_cols)
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        x = rng.standard_normal((r1 - r0, flat_cols), dtype=np.float32)
        if outlier_frac > 0:
            n = x.size
            k = int(round(n * outlier_frac))
            idx = rng.integers(0, n, size=k)
            x.reshape(-1)[idx] *= np.float32(outlier_mult)
        out2[r0:r1] = _to_bf16_bits(x)
    return out


def _weights(rng: np.random.Generator, D: int) -> dict:
    return {k: _to_bf16_bits(rng.uniform(0.5, 1.5, size=D).astype(np.float32))
            for k in ("q", "k", "idx_q", "idx_k")}


def _shape(base: dict, rotary_dim=None, rope_style=ROPE_NEOX, page_size=64,
           rope_theta=1e4, rms_eps=1e-6, scale_mode=0) -> dict:
    s = dict(base)
    s["rotary_dim"] = s["head_dim"] if rotary_dim is None else int(rotary_dim)
    s["rope_style"] = int(rope_style)
    s["page_size"] = int(page_size)
    s["rope_theta"] = float(rope_theta)
    s["rms_eps"] = float(rms_eps)
    s["scale_mode"] = int(scale_mode)
    return s


def _hnd_cache(pool: str, dtype: int, num_pages: int, heads: int, P: int, D: int,
               page_pad_bytes: int = 0, offset: int = GUARD_BYTES) -> CacheSpec:
    """Head-major page [heads, P, D]; optional padding after every page."""
    es = ELEM_SIZE[dtype]
    assert page_pad_bytes % es == 0
    sT = D
    sH = P * D
    sP = heads * P * D + page_pad_bytes // es
    return CacheSpec(pool, offset, dtype, num_pages, heads, sP, sH, sT)


def cache_extent_bytes(c: CacheSpec, page_size: int, head_dim: int) -> int:
    """One past the last byte a write can reach, from element 0."""
    last = ((c.num_pages - 1) * c.stride_page + (c.num_heads - 1) * c.stride_head
            + (page_size - 1) * c.stride_token + head_dim)
    return last * c.elem_size()


def _pool_sizes(caches: dict, page_size: int, head_dim: int) -> dict:
    pools: dict = {}
    for c in caches.values():
        if c is None:
            continue
        end = c.offset + cache_extent_bytes(c, page_size, head_dim) + GUARD_BYTES
        pools[c.pool] = max(pools.get(c.pool, 0), end)
    # round up to 16 bytes so every pool can be viewed as 16-byte words
    return {k: (v + 15) // 16 * 16 for k, v in pools.items()}


def _finish(name, shape, qkv, row_stride, pos, slots, pt, weights, scales, caches, seed,
            valid_mask):
    """``valid_mask`` records, by construction, which tokens were given a slot that
    lands in a page (the others were made padding or out of range on purpose)."""
    pools = _pool_sizes(caches, shape["page_size"], shape["head_dim"])
    meta = {"valid_mask": np.asarray(valid_mask, dtype=bool),
            "num_valid": int(np.count_nonzero(valid_mask))}
    return Workload(name, shape, qkv, row_stride, pos.astype(np.int32), slots.astype(np.int64),
                    None if pt is None else np.ascontiguousarray(pt, dtype=np.int32),
                    weights, np.asarray(scales, dtype=np.float32), caches, pools, seed, meta)


# ----------------------------------------------------------------------------
# generic decode / prefill builder
# ----------------------------------------------------------------------------

def make_batch(name: str, seed: int, heads: dict, seq_positions: list, max_blocks: int,
               num_pages: int, *, rotary_dim=None, rope_style=ROPE_NEOX, page_size=64,
               row_pad=0, kv_dtype=DTYPE_E4M3, idx_k_dtype=DTYPE_E4M3, with_idx_k=True,
               page_pad_bytes=0, pad_frac=0.0, outlier_frac=0.0, use_page_table=True,
               scale=0.05, scale_mode=0, shuffle_pages=True, make_rows=True) -> Workload:
    """A batch of sequences; ``seq_positions[s]`` lists the new tokens' positions of
    sequence s.  Logical slot = s * max_blocks * P + pos through a page table that
    is a seeded permutation of the pages, or, with ``use_page_table=False``, the
    physical slot page * P + pos % P the table would give."""
    rng = np.random.default_rng(seed)
    shape = _shape(heads, rotary_dim, rope_style, page_size, scale_mode=scale_mode)
    D, P = shape["head_dim"], page_size
    S = len(seq_positions)
    perm = rng.permutation(num_pages) if shuffle_pages else np.arange(num_pages)
    need = S * max_blocks
    if need <= num_pages:
        pt = perm[:need].reshape(S, max_blocks).astype(np.int32)
    else:
        pt = np.full((S, max_blocks), -1, dtype=np.int32)
        flat = pt.reshape(-1)
        flat[:num_pages] = perm
    seq_ids = np.concatenate([np.full(len(p), s, dtype=np.int64) for s, p in enumerate(seq_positions)])
    pos = np.concatenate([np.asarray(p, dtype=np.int64) for p in seq_positions])
    assert pos.max(initial=0) < max_blocks * P
    if use_page_table:
        slots = seq_ids * (max_blocks * P) + pos
    else:
        slots = pt[seq_ids, pos // P].astype(np.int64) * P + pos % P
    T = pos.shape[0]
    valid = pt[seq_ids, pos // P] >= 0
    if pad_frac > 0 and T > 0:
        k = int(round(T * pad_frac))
        padded = rng.choice(T, size=k, replace=False)
        slots[padded] = -1
        valid[padded] = False
    W = (heads["num_q_heads"] + 2 * heads["num_kv_heads"] + heads["num_idx_q_heads"]
         + heads["num_idx_k_heads"]) * D
    row_stride = W + row_pad
    if make_rows:
        qkv = _normal_bf16(rng, (T, row_stride), outlier_frac=outlier_frac)
    else:   # the rows are made by a projection from hidden states instead
        qkv = np.zeros((T, 0), dtype=np.uint16)
    weights = _weights(rng, D)
    nscales = 3 if scale_mode == 0 else 2 * heads["num_kv_heads"] + heads["num_idx_k_heads"]
    scales = np.full(nscales, scale, dtype=np.float32)
    caches = {
        "k": _hnd_cache("k", kv_dtype, num_pages, heads["num_kv_heads"], P, D, page_pad_bytes),
        "v": _hnd_cache("v", kv_dtype, num_pages, heads["num_kv_heads"], P, D, page_pad_bytes),
        "idx_k": (_hnd_cache("idx_k", idx_k_dtype, num_pages, heads["num_idx_k_heads"], P, D,
                             page_pad_bytes) if with_idx_k else None),
    }
    return _finish(name, shape, qkv, row_stride, pos, slots, pt if use_page_table else None,
                   weights, scales, caches, seed, valid)


# ----------------------------------------------------------------------------
# the five named workloads
# ----------------------------------------------------------------------------

def config1_tiny_decode(seed: int = 1000) -> Workload:
    """4 sequences x 1 token, tiny shapes, positions U[0, 512), 64 pages in a
    seeded permuted page table [8, 8] (rows 0..3 used), fp8 K/V (scale 0.05),
    bf16 index-K."""
    rng = np.random.default_rng(seed)
    pos = [[int(p)] for p in rng.integers(0, 512, size=4)]
    w = make_batch("tiny_decode_4", seed + 1, TINY, pos, max_blocks=8, num_pages=64,
                   idx_k_dtype=DTYPE_BF16)
    # the page table is the full permutation reshaped [8, 8]
    rng2 = np.random.default_rng(seed + 2)
    full = rng2.permutation(64).astype(np.int32).reshape(8, 8)
    w.page_table = full
    return w


def config2_decode64(seed: int = 2000) -> Workload:
    """64 sequences x 1 token, context lengths U{1..9216} (position = length - 1),
    big shapes, 9216 shuffled pages, HND pages padded by 256 bytes, fp8 K/V/idx-K,
    10% of slots padding (-1)."""
    rng = np.random.default_rng(seed)
    L = rng.integers(1, 9216 + 1, size=64)
    pos = [[int(l) - 1] for l in L]
    return make_batch("decode_64", seed + 1, BIG, pos, max_blocks=144, num_pages=9216,
                      page_pad_bytes=256, pad_frac=0.10)


def config3_decode_step(layer: int, big: bool = False, seed_base: int = 3000) -> Workload:
    """One layer of the 60-layer decode step at batch 256: tiny shapes, positions
    U[0, 512), 2048 pages per layer (or big shapes, positions U[0, 128), 512 pages)."""
    seed = seed_base + layer
    rng = np.random.default_rng(seed)
    if big:
        pos = [[int(p)] for p in rng.integers(0, 128, size=256)]
        return make_batch(f"decode_step_big_l{layer}", seed + 100000, BIG, pos, max_blocks=2,
                          num_pages=512)
    pos = [[int(p)] for p in rng.integers(0, 512, size=256)]
    return make_batch(f"decode_step_tiny_l{layer}", seed + 100000, TINY, pos, max_blocks=8,
                      num_pages=2048, idx_k_dtype=DTYPE_BF16)


def config4_prefill(seed: int = 4000, num_seqs: int = 8, seq_len: int = 8192) -> Workload:
    """8 sequences x 8192 tokens (positions 0..8191), big shapes, N(0,1) inputs with
    1% of elements x20, 1024 pages in a shuffled table, contiguous HND fp8 caches."""
    P = 64
    max_blocks = seq_len // P
    pos = [list(range(seq_len)) for _ in range(num_seqs)]
    return make_batch(f"prefill_{num_seqs}x{seq_len}", seed, BIG, pos, max_blocks=max_blocks,
                      num_pages=num_seqs * max_blocks, outlier_frac=0.01)


def config5_mixed(seed: int = 5000, num_pages: int = 24576, chunk_len: int = 2048,
                  num_chunks: int = 4, num_decode: int = 192) -> Workload:
    """4 prefill chunks of 2048 tokens (starts drawn from {0, 2048, 4096, 6144}) plus
    192 decode tokens (context U{1..9216}); rotary dim 64 of 128; rows strided by
    width + 64; one fp8 K/V pool [pages, 2, 8, 64, 128] over 2^31 elements, K and V
    being its non-contiguous halves; page-table entries not referenced are -1; 5% of
    slots are -1 and 1% fall outside the pool (a logical block past the table, or a
    table entry >= the page count)."""
    rng = np.random.default_rng(seed)
    P, D, max_blocks = 64, 128, 144
    heads = BIG
    starts = rng.choice([0, 2048, 4096, 6144], size=num_chunks)
    seq_positions = [list(range(int(s), int(s) + chunk_len)) for s in starts]
    L = rng.integers(1, 9216 + 1, size=num_decode)
    seq_positions += [[int(l) - 1] for l in L]
    S = len(seq_positions)
    # referenced blocks get distinct pages drawn from the whole pool; one extra
    # table row holds entries at or beyond the page count
    pt = np.full((S + 1, max_blocks), -1, dtype=np.int32)
    referenced = []
    for s, p in enumerate(seq_positions):
        for b in sorted({q // P for q in p}):
            referenced.append((s, b))
    assert len(referenced) <= num_pages
    pages = rng.permutation(num_pages)[:len(referenced)]
    for (s, b), pg in zip(referenced, pages):
        pt[s, b] = pg
    pt[S, :] = num_pages + rng.integers(0, 1000, size=max_blocks)
    seq_ids = np.concatenate([np.full(len(p), s, dtype=np.int64) for s, p in enumerate(seq_positions)])
    pos = np.concatenate([np.asarray(p, dtype=np.int64) for p in seq_positions])
    slots = seq_ids * (max_blocks * P) + pos
    T = pos.shape[0]
    pick = rng.permutation(T)
    n_pad = int(round(0.05 * T))
    n_out = int(round(0.01 * T))
    slots[pick[:n_pad]] = -1
    out_idx = pick[n_pad:n_pad + n_out]
    half = len(out_idx) // 2
    # logical block past the table
    slots[out_idx[:half]] = (pt.size + rng.integers(0, 64, size=half)) * P + rng.integers(0, P, size=half)
    # table entry >= num_pages (the extra row)
    slots[out_idx[half:]] = S * max_blocks * P + rng.integers(0, max_blocks * P, size=len(out_idx) - half)
    W = (heads["num_q_heads"] + 2 * heads["num_kv_heads"] + heads["num_idx_q_heads"]
         + heads["num_idx_k_heads"]) * D
    row_stride = W + 64
    qkv = _normal_bf16(rng, (T, row_stride))
    weights = _weights(rng, D)
    shape = _shape(heads, rotary_dim=64)
    Hkv = heads["num_kv_heads"]
    # pool [pages, 2, Hkv, P, D] fp8: K = [:, 0], V = [:, 1]
    sP = 2 * Hkv * P * D
    k = CacheSpec("kv", GUARD_BYTES, DTYPE_E4M3, num_pages, Hkv, sP, P * D, D)
    v = CacheSpec("kv", GUARD_BYTES + Hkv * P * D, DTYPE_E4M3, num_pages, Hkv, sP, P * D, D)
    ik = _hnd_cache("idx_k", DTYPE_E4M3, num_pages, heads["num_idx_k_heads"], P, D)
    caches = {"k": k, "v": v, "idx_k": ik}
    valid = np.ones(T, dtype=bool)
    valid[pick[:n_pad + n_out]] = False
    return _finish("mixed_4x2048_192", shape, qkv, row_stride, pos, slots, pt, weights,
                   np.full(3, 0.05, dtype=np.float32), caches, seed, valid)


CONFIGS = {
    1: config1_tiny_decode,
    2: config2_decode64,
    4: config4_prefill,
    5: config5_mixed,
}


# ----------------------------------------------------------------------------
# sentinel-filled host pools
# ----------------------------------------------------------------------------

def sentinel_pool(nbytes: int, seed: int) -> np.ndarray:
    """A pool filled with a seeded pseudo-random byte pattern (a 1 MiB block tiled),
    so that any stray write shows up as a changed byte."""
    rng = np.random.default_rng(0x5E11 + seed)
    block = rng.integers(0, 256, size=1 << 20, dtype=np.uint8)
    reps = -(-nbytes // block.size)
    if reps == 1:
        return block[:nbytes].copy()
    return np.tile(block, reps)[:nbytes]


def host_pools(w: Workload) -> dict:
    return {name: sentinel_pool(n, i + w.seed) for i, (name, n) in enumerate(sorted(w.pools.items()))}


def oracle_cache_args(w: Workload, pools: dict) -> dict:
    """Cache descriptors for the oracle's forward(): key -> dict or None."""
    out = {}
    for key in ("k", "v", "idx_k"):
        c = w.caches.get(key)
        if c is None:
            out[key] = None
            continue
        out[key] = dict(data=pools[c.pool], offset=c.offset, dtype=c.dtype, num_pages=c.num_pages,
                        num_heads=c.num_heads, stride_page=c.stride_page,
                        stride_head=c.stride_head, stride_token=c.stride_token)
    return out


def empty_outputs(w: Workload):
    s, T = w.shape, w.num_tokens
    D = s["head_dim"]
    q = np.zeros((T, s["num_q_heads"], D), dtype=np.uint16)
    iq = np.zeros((T, s["num_idx_q_heads"], D), dtype=np.uint16)
    return q, iq


def subset(w: Workload, idx) -> Workload:
    """The same workload restricted to the tokens ``idx`` (order kept); pools and
    page table unchanged."""
    idx = np.asarray(idx, dtype=np.int64)
    mask = w.meta["valid_mask"][idx]
    meta = dict(w.meta, valid_mask=mask, num_valid=int(np.count_nonzero(mask)))
    return Workload(w.name + f"[{len(idx)}]", w.shape, np.ascontiguousarray(w.qkv[idx]),
                    w.row_stride, w.positions[idx].copy(), w.slot_mapping[idx].copy(),
                    w.page_table, w.weights, w.scales, w.caches, w.pools, w.seed, meta)


# ----------------------------------------------------------------------------
# indexer inputs: queries over an index-K cache holding each sequence's history
# ----------------------------------------------------------------------------

@dataclass
class IndexerWorkload:
    name: str
    idx_q: np.ndarray          # uint16 (bf16 bits) [T, H, D]
    kv_len: np.ndarray         # int32 [T]: visible tokens of each query
    table_offset: np.ndarray   # int64 [T]: start of the query's row in the flattened table
    page_table: np.ndarray     # int32 [S, max_pages]
    cache: CacheSpec           # one head
    pool_bytes: int
    pool_fill: np.ndarray      # uint8 pool contents (the history)
    k_scale: float
    page_size: int
    block_tokens: int
    topk: int
    max_blocks: int
    seed: int = 0

    def algorithmic_bytes(self) -> int:
        """Bytes an indexer must move: each query's heads and visible index-K rows read,
        one page-table entry per page, the block scores and top-k ids written."""
        T, H, D = self.idx_q.shape
        es = self.cache.elem_size()
        read = T * H * D * 2 + int(self.kv_len.sum()) * D * es
        read += int(np.ceil(self.kv_len / self.page_size).sum()) * 4 + T * (4 + 8)
        write = T * (self.max_blocks * 4 + self.topk * 4)
        return read + write


def _random_cache_codes(rng, n, dtype):
    if dtype == DTYPE_E4M3:
        # every finite E4M3 code, the two NaN codes (0x7F, 0xFF) excluded
        codes = rng.integers(0, 254, size=n, dtype=np.uint16).astype(np.uint8)
        return np.where(codes >= 0x7F, codes + 1, codes).astype(np.uint8)
    vals = _to_bf16_bits(rng.standard_normal(n // 2, dtype=np.float32))
    return vals.view(np.uint8)


def make_indexer_batch(name: str, seed: int, kv_lens, heads: int = 8, head_dim: int = 128,
                       page_size: int = 64, block_tokens: int = 128, topk: int = 16,
                       dtype: int = DTYPE_E4M3, k_scale: float = 0.05, page_pad_bytes: int = 0,
                       extra_pages: int = 16, max_blocks=None) -> IndexerWorkload:
    """One decode query per sequence; sequence s sees kv_lens[s] tokens of history
    in pages given by a seeded permutation; the pool holds random finite codes."""
    rng = np.random.default_rng(seed)
    kv_lens = np.asarray(kv_lens, dtype=np.int64)
    S = len(kv_lens)
    pages_per_seq = np.maximum(1, -(-kv_lens // page_size))
    max_pages = int(pages_per_seq.max())
    num_pages = int(pages_per_seq.sum()) + extra_pages
    perm = rng.permutation(num_pages).astype(np.int32)
    pt = np.full((S, max_pages), -1, dtype=np.int32)
    k = 0
    for s in range(S):
        n = int(pages_per_seq[s])
        pt[s, :n] = perm[k:k + n]
        k += n
    cache = _hnd_cache("idx_k", dtype, num_pages, 1, page_size, head_dim, page_pad_bytes)
    pool_bytes = _pool_sizes({"idx_k": cache}, page_size, head_dim)["idx_k"]
    pool = _random_cache_codes(rng, pool_bytes, dtype)
    idx_q = _normal_bf16(rng, (S, heads, head_dim))
    if max_blocks is None:
        max_blocks = int(max(1, -(-int(kv_lens.max()) // block_tokens)))
    return IndexerWorkload(name, idx_q, kv_lens.astype(np.int32),
                           (np.arange(S, dtype=np.int64) * max_pages), pt, cache, pool_bytes,
                           pool, float(k_scale), page_size, block_tokens, topk, max_blocks, seed)


def indexer_decode64(seed: int = 6000) -> IndexerWorkload:
    """The decode-batch-64 layer's indexer: 64 queries, contexts U{1..9216}, 8 index
    heads of dim 128, fp8 index-K cache, top-16 of 128-token blocks."""
    rng = np.random.default_rng(seed)
    return make_indexer_batch("indexer_decode_64", seed + 1, rng.integers(1, 9216 + 1, size=64))


def make_indexer_prefill(name: str, seed: int, seq_lens, heads: int = 8, head_dim: int = 128,
                         page_size: int = 64, block_tokens: int = 128, topk: int = 16,
                         dtype: int = DTYPE_E4M3, k_scale: float = 0.05, page_pad_bytes: int = 0,
                         interleave: bool = False, max_blocks=None) -> IndexerWorkload:
    """Prefill queries: sequence s contributes seq_lens[s] queries, the one at
    position p seeing the p + 1 tokens up to and including itself (causal), all
    through the sequence's row of the page table.  Queries come sequence by
    sequence in position order, or (``interleave``) in a seeded shuffled order so
    that runs of one sequence are broken up."""
    base = make_indexer_batch(name, seed, seq_lens, heads, head_dim, page_size, block_tokens, topk,
                              dtype, k_scale, page_pad_bytes, max_blocks=max_blocks)
    rng = np.random.default_rng(seed + 17)
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    kv = np.concatenate([np.arange(1, int(L) + 1, dtype=np.int64) for L in seq_lens])
    seq = np.concatenate([np.full(int(L), s, dtype=np.int64) for s, L in enumerate(seq_lens)])
    if interleave:
        order = rng.permutation(kv.shape[0])
        kv, seq = kv[order], seq[order]
    max_pages = base.page_table.shape[1]
    idx_q = _normal_bf16(rng, (kv.shape[0], heads, head_dim))
    return IndexerWorkload(name, idx_q, kv.astype(np.int32), seq * max_pages, base.page_table,
                           base.cache, base.pool_bytes, base.pool_fill, base.k_scale, page_size,
                           block_tokens, topk, base.max_blocks, seed)


def indexer_prefill(seed: int = 6100, num_seqs: int = 8, seq_len: int = 8192) -> IndexerWorkload:
    """The prefill batch's indexer: 8 sequences x 8192 queries, causal, 8 index heads
    of dim 128, fp8 index-K cache, top-16 of 128-token blocks (64 per query row)."""
    return make_indexer_prefill(f"indexer_prefill_{num_seqs}x{seq_len}", seed,
                                [seq_len] * num_seqs)


def indexer_cache_arg(w: IndexerWorkload, pool: np.ndarray) -> dict:
    c = w.cache
    return dict(data=pool, offset=c.offset, dtype=c.dtype, num_pages=c.num_pages, num_heads=1,
                stride_page=c.stride_page, stride_head=c.stride_head, stride_token=c.stride_token)


# ----------------------------------------------------------------------------
# projection inputs: hidden states and the packed [Q | K | V | idx-Q | idx-K]
# weight, for the projection with the producer in its epilogue
# ----------------------------------------------------------------------------

@dataclass
class ProjectionWorkload:
    """Hidden states and an output-major weight whose product is the producer's
    rows; ``producer`` holds everything else (heads, positions, slots, page table,
    norm weights, scales, caches) and has no rows of its own (qkv is [T, 0]).
    Operands are bf16 bits (uint16) or E4M3 codes (uint8) with per-token and
    per-output dequantisation scales."""
    name: str
    producer: Workload
    hidden: np.ndarray         # [T, hidden_stride]: uint16 bf16 bits or uint8 E4M3 codes
    hidden_size: int
    weight: np.ndarray         # [W, weight_stride], same element type
    hidden_scales: np.ndarray | None = None   # float32 [T]
    weight_scales: np.ndarray | None = None   # float32 [W]

    @property
    def operand_dtype(self) -> int:
        return DTYPE_BF16 if self.hidden.dtype == np.uint16 else DTYPE_E4M3

    @property
    def num_tokens(self) -> int:
        return self.producer.num_tokens

    @property
    def width(self) -> int:
        return self.producer.width

    def flops(self) -> int:
        """Multiply-adds x 2 of the projection."""
        return 2 * self.num_tokens * self.width * self.hidden_size

    def with_rows(self, rows: np.ndarray) -> Workload:
        """The producer workload with the given projection rows [T, W]."""
        w = self.producer
        return Workload(w.name, w.shape, np.ascontiguousarray(rows), rows.shape[1], w.positions,
                        w.slot_mapping, w.page_table, w.weights, w.scales, w.caches, w.pools,
                        w.seed, w.meta)


def _e4m3_rows(x: np.ndarray):
    """Per-row E4M3 quantisation of float32 rows (input preparation): the scale is
    the row's largest magnitude / 448 (1 for an all-zero row) and the codes are
    torch's rounding cast of x / scale."""
    import torch
    amax = np.abs(x).max(axis=1)
    scale = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    t = torch.from_numpy(np.ascontiguousarray(x / scale[:, None], dtype=np.float32))
    codes = t.to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()
    return codes, scale


def make_projection_batch(name: str, seed: int, heads: dict, seq_positions: list,
                          hidden_size: int, *, hidden_pad: int = 0, weight_pad: int = 0,
                          operand_dtype: int = DTYPE_BF16, **batch_kw) -> ProjectionWorkload:
    """Hidden states N(0, 1) and weights N(0, 1/hidden_size), so that the projection
    rows are about N(0, 1) like the producer's own inputs, as bf16 or as E4M3 with
    one scale per token and per output row; the rest from ``make_batch`` (same
    keyword arguments) without rows.  Row strides are widened by ``hidden_pad`` /
    ``weight_pad`` elements filled with NaN, which no correct kernel reads."""
    w = make_batch(name, seed, heads, seq_positions, make_rows=False, **batch_kw)
    rng = np.random.default_rng(seed + 7919)
    T, W, K = w.num_tokens, w.width, int(hidden_size)
    fp8 = operand_dtype == DTYPE_E4M3
    etype, nan = (np.uint8, 0x7F) if fp8 else (np.uint16, 0x7FC0)
    hidden = np.full((T, K + hidden_pad), nan, dtype=etype)
    weight = np.full((W, K + weight_pad), nan, dtype=etype)
    sx = np.empty(T, dtype=np.float32) if fp8 else None
    sw = np.empty(W, dtype=np.float32) if fp8 else None
    for r0 in range(0, T, 4096):
        r1 = min(T, r0 + 4096)
        x = rng.standard_normal((r1 - r0, K), dtype=np.float32)
        if fp8:
            hidden[r0:r1, :K], sx[r0:r1] = _e4m3_rows(x)
        else:
            hidden[r0:r1, :K] = _to_bf16_bits(x)
    for r0 in range(0, W, 2048):
        r1 = min(W, r0 + 2048)
        x = rng.standard_normal((r1 - r0, K), dtype=np.float32) * np.float32(1.0 / np.sqrt(K))
        if fp8:
            weight[r0:r1, :K], sw[r0:r1] = _e4m3_rows(x)
        else:
            weight[r0:r1, :K] = _to_bf16_bits(x)
    return ProjectionWorkload(name, w, hidden, K, weight, sx, sw)


PROJECTION_HIDDEN = 6144


def projection_prefill(seed: int = 7000, num_seqs: int = 8, seq_len: int = 8192,
                       hidden_size: int = PROJECTION_HIDDEN,
                       operand_dtype: int = DTYPE_BF16) -> ProjectionWorkload:
    """The prefill batch of the producer (8 sequences x 8192 tokens, big shapes,
    1,024 shuffled pages, contiguous HND fp8 caches) made from hidden states of
    size 6,144 through the packed 11,392-output projection (bf16 or E4M3 operands)."""
    P = 64
    max_blocks = seq_len // P
    pos = [list(range(seq_len)) for _ in range(num_seqs)]
    tag = "e4m3" if operand_dtype == DTYPE_E4M3 else "bf16"
    return make_projection_batch(f"projection_prefill_{num_seqs}x{seq_len}_h{hidden_size}_{tag}",
                                 seed, BIG, pos, hidden_size, max_blocks=max_blocks,
                                 num_pages=num_seqs * max_blocks, operand_dtype=operand_dtype)


def projection_decode(seed: int = 7100, batch: int = 64, hidden_size: int = PROJECTION_HIDDEN,
                      operand_dtype: int = DTYPE_BF16) -> ProjectionWorkload:
    """Decode: ``batch`` sequences x 1 token with contexts U{1..9216}, big shapes,
    9,216 shuffled pages padded by 256 bytes, 10% padded slots."""
    rng = np.random.default_rng(seed)
    L = rng.integers(1, 9216 + 1, size=batch)
    pos = [[int(l) - 1] for l in L]
    tag = "e4m3" if operand_dtype == DTYPE_E4M3 else "bf16"
    return make_projection_batch(f"projection_decode_{batch}_h{hidden_size}_{tag}", seed + 1, BIG,
                                 pos, hidden_size, max_blocks=144, num_pages=9216,
                                 page_pad_bytes=256, pad_frac=0.10, operand_dtype=operand_dtype)
