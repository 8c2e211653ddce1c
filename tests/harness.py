"""Shared test helpers: running the oracle on a workload and comparing results.

Nothing here computes the producer; the expected values come from the oracle
(``oracle/``) and the textbook/library pins in ``oracle_pins.py``.
"""
from __future__ import annotations

import numpy as np

from paged_kv_cache_msa_gb300 import workloads as wl

# Tolerances stated by the producer's specification: bf16 outputs within
# 2e-2 absolute + 1e-2 relative of the oracle; fp8 cache entries within one E4M3
# step on the ordered code line; placement and the set of written bytes exact.
BF16_ATOL = 2e-2
BF16_RTOL = 1e-2
E4M3_MAX_ULP = 1


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def e4m3_ordinal(c: np.ndarray) -> np.ndarray:
    """Position of an E4M3 code on the monotone integer line of sign-magnitude codes
    (+0 and -0 both map to 0)."""
    c = np.asarray(c, dtype=np.int32)
    mag = c & 0x7F
    return np.where(c & 0x80, -mag, mag)


def e4m3_ulp_distance(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    return np.abs(e4m3_ordinal(a) - e4m3_ordinal(b))


def run_oracle(w: wl.Workload, pools: dict | None = None, token_range=None):
    """Runs the oracle on ``w`` into fresh sentinel pools (or the given ones).
    Returns (q_out, idx_q_out, pools)."""
    import oracle
    if pools is None:
        pools = wl.host_pools(w)
    q, iq = wl.empty_outputs(w)
    ca = wl.oracle_cache_args(w, pools)
    kw = {}
    if token_range is not None:
        kw = dict(token_offset=token_range[0], num_tokens=token_range[1] - token_range[0])
    oracle.forward(w.shape, w.qkv, w.row_stride, w.positions, w.slot_mapping, w.page_table,
                   w.weights, q, iq, ca["k"], ca["v"], ca["idx_k"], w.scales, **kw)
    return q, iq, pools


def cache_cells(w: wl.Workload, key: str, placements) -> np.ndarray:
    """Byte offsets (into the pool) of every element a cache write covers, for the
    given per-token placements [(page, off) or None]; shape [n_valid, heads, D*es]."""
    c = w.caches[key]
    es = c.elem_size()
    D = w.shape["head_dim"]
    rows = []
    for pl in placements:
        if pl is None:
            continue
        page, off = pl
        heads = []
        for h in range(c.num_heads):
            e0 = page * c.stride_page + h * c.stride_head + off * c.stride_token
            heads.append(c.offset + es * e0 + np.arange(D * es))
        rows.append(heads)
    if not rows:
        return np.zeros((0, c.num_heads, D * es), dtype=np.int64)
    return np.asarray(rows, dtype=np.int64)


def compare_bf16(actual_bits, expected_bits, what: str):
    a = bf16_bits_to_f32(actual_bits).astype(np.float64)
    e = bf16_bits_to_f32(expected_bits).astype(np.float64)
    bad = ~(np.abs(a - e) <= BF16_ATOL + BF16_RTOL * np.abs(e))
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} outside "
                           f"{BF16_ATOL} + {BF16_RTOL}*|ref|; first at {np.argwhere(bad)[:5].tolist()}")
