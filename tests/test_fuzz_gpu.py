"""Seeded random configurations of the producer and the indexer against the oracle (GPU).

Every case draws its shapes and options from a seeded generator -- head counts,
head_dim, rotary dim and style, page size, cache dtypes, padded pages, strided
rows, page-table or physical slots, padded and out-of-range slots, token counts,
launch mode, scale mode -- and is checked exactly as the named workloads are.
"""
import numpy as np
import pytest

from paged_kv_cache_msa_gb300 import binding as B
from paged_kv_cache_msa_gb300 import workloads as wl

from gpu_harness import check_against_oracle

pytestmark = pytest.mark.gpu


def _random_case(seed):
    rng = np.random.default_rng(10_000 + seed)
    D = int(rng.choice([64, 128]))
    heads = dict(num_q_heads=int(rng.integers(0, 40)), num_kv_heads=int(rng.integers(1, 9)),
                 num_idx_q_heads=int(rng.integers(0, 9)), num_idx_k_heads=int(rng.integers(0, 3)),
                 head_dim=D)
    if sum(heads[k] for k in heads if k != "head_dim") == 0:
        heads["num_q_heads"] = 1
    style = int(rng.integers(0, 2))
    step = 16 if style == wl.ROPE_NEOX else 8
    rd = int(rng.integers(0, D // step + 1)) * step
    P = int(rng.choice([16, 32, 48, 64, 128]))
    S = int(rng.integers(1, 12))
    max_blocks = int(rng.integers(1, 8))
    seq_positions = []
    for _ in range(S):
        n = int(rng.choice([1, 1, 2, 5, 40]))
        start = int(rng.integers(0, max(1, max_blocks * P - n)))
        seq_positions.append(list(range(start, min(start + n, max_blocks * P))))
    kv_dtype = int(rng.choice([wl.DTYPE_E4M3, wl.DTYPE_BF16]))
    ik_dtype = int(rng.choice([wl.DTYPE_E4M3, wl.DTYPE_BF16]))
    w = wl.make_batch(f"fuzz{seed}", 20_000 + seed, heads, seq_positions, max_blocks=max_blocks,
                      num_pages=S * max_blocks + int(rng.integers(0, 5)), rotary_dim=rd,
                      rope_style=style, page_size=P, row_pad=8 * int(rng.integers(0, 5)),
                      kv_dtype=kv_dtype, idx_k_dtype=ik_dtype,
                      with_idx_k=bool(rng.integers(0, 4)),
                      page_pad_bytes=16 * int(rng.integers(0, 3)),
                      pad_frac=float(rng.choice([0.0, 0.1, 0.5])),
                      use_page_table=bool(rng.integers(0, 4)),
                      scale=float(rng.uniform(0.01, 0.5)),
                      scale_mode=int(rng.integers(0, 2)), outlier_frac=0.01)
    if w.page_table is not None and rng.integers(0, 2):
        pt = np.array(w.page_table, copy=True)
        pt.reshape(-1)[rng.integers(0, pt.size)] = -1
        w.page_table = pt
    flags = int(rng.choice([0, B.MSA_LAUNCH_PERSISTENT, B.MSA_LAUNCH_PERSISTENT | B.MSA_LAUNCH_PDL]))
    return w, flags


@pytest.mark.parametrize("seed", range(40))
def test_random_producer_configuration(seed):
    w, flags = _random_case(seed)
    check_against_oracle(w, flags)


@pytest.mark.parametrize("seed", range(12))
def test_random_indexer_configuration(seed):
    from test_indexer_gpu import _check
    rng = np.random.default_rng(30_000 + seed)
    D = int(rng.choice([64, 128]))
    lens = rng.integers(0, 3000, size=int(rng.integers(1, 20)))
    w = wl.make_indexer_batch(f"ifuzz{seed}", 40_000 + seed, lens, heads=int(rng.integers(1, 17)),
                              head_dim=D, page_size=int(rng.choice([16, 64, 96])),
                              block_tokens=int(rng.choice([32, 64, 128, 256])),
                              topk=int(rng.integers(1, 40)),
                              dtype=int(rng.choice([wl.DTYPE_E4M3, wl.DTYPE_BF16])),
                              page_pad_bytes=16 * int(rng.integers(0, 3)))
    _check(w)


@pytest.mark.parametrize("seed", range(16))
def test_random_projection_configuration(seed):
    """The projection with the producer in its epilogue over random head counts,
    head_dim, RoPE style and rotary dim, token counts, hidden sizes, row padding,
    operand type (with per-token / per-output scales for E4M3), cache dtypes,
    scale mode and padded slots."""
    from test_projection_gpu import check_projection
    rng = np.random.default_rng(50_000 + seed)
    D = int(rng.choice([64, 128]))
    heads = dict(num_q_heads=int(rng.integers(0, 12)), num_kv_heads=int(rng.integers(1, 5)),
                 num_idx_q_heads=int(rng.integers(0, 5)), num_idx_k_heads=int(rng.integers(0, 2)),
                 head_dim=D)
    style = int(rng.integers(0, 2))
    step = 16 if style == wl.ROPE_NEOX else 8
    rd = int(rng.choice([D, D // 2, 0, int(rng.integers(0, D // step + 1)) * step]))
    T = int(rng.choice([1, 17, 128, 129, 255, 256, 300]))
    K = int(rng.integers(1, 40)) * 8
    dt = int(rng.choice([wl.DTYPE_BF16, wl.DTYPE_E4M3]))
    mult = 16 if dt == wl.DTYPE_E4M3 else 8
    P = int(rng.choice([16, 64]))
    start = int(rng.integers(0, 64))
    max_blocks = -(-(start + T) // P)
    pw = wl.make_projection_batch(
        f"pfuzz{seed}", 60_000 + seed, heads, [list(range(start, start + T))], K,
        hidden_pad=(-K) % mult + mult * int(rng.integers(0, 3)),
        weight_pad=(-K) % mult + mult * int(rng.integers(0, 3)), operand_dtype=dt,
        max_blocks=max_blocks, num_pages=max_blocks + int(rng.integers(0, 4)), page_size=P,
        rotary_dim=rd, rope_style=style,
        kv_dtype=int(rng.choice([wl.DTYPE_E4M3, wl.DTYPE_BF16])),
        idx_k_dtype=int(rng.choice([wl.DTYPE_E4M3, wl.DTYPE_BF16])),
        with_idx_k=bool(rng.integers(0, 4)), pad_frac=float(rng.choice([0.0, 0.2])),
        use_page_table=bool(rng.integers(0, 3)), scale_mode=int(rng.integers(0, 2)),
        scale=float(rng.uniform(0.02, 0.3)))
    check_projection(pw)
