"""Parity of the CUDA indexer with the oracle, through the C ABI (GPU).

Block scores: within fp32 accumulation error of the oracle (both fp32, different
summation order), exact -inf pattern.  Top-k ids: equal to the oracle's wherever
the oracle's ranking separates neighbours by more than that error; otherwise the
two ids must be within it of each other (either order is a correct answer)."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_msa_gb300 import build as build_mod
from paged_kv_cache_msa_gb300 import workloads as wl
from paged_kv_cache_msa_gb300.device import DeviceIndexer

from oracle_pins import check_indexer_against_reference

pytestmark = pytest.mark.gpu


def _check(w, pool=None, flags=0):
    build_mod.build()
    pool = w.pool_fill if pool is None else pool
    ref_s, ref_top = oracle.indexer(w.idx_q, w.kv_len, w.table_offset, w.page_table,
                                    wl.indexer_cache_arg(w, pool), w.k_scale, w.page_size,
                                    w.block_tokens, w.topk, w.max_blocks)
    dv = DeviceIndexer(w, pool=pool)
    dv.run(launch_flags=flags)
    torch.cuda.synchronize()
    s = dv.block_scores.cpu().numpy()
    top = dv.topk_ids.cpu().numpy()
    check_indexer_against_reference(w, s, top, ref_s.astype(np.float64), ref_top)
    # the ids are a valid ranking of the kernel's own scores
    for t in range(s.shape[0]):
        ids = [i for i in top[t] if i >= 0]
        assert len(set(ids)) == len(ids)
        vals = [s[t, i] for i in ids]
        assert all(vals[i] >= vals[i + 1] for i in range(len(vals) - 1))
        nfin = int(np.isfinite(s[t]).sum())
        assert len(ids) == min(w.topk, nfin)
    return dv


def test_indexer_decode64():
    _check(wl.indexer_decode64())


@pytest.mark.parametrize("dtype,D,heads", [(wl.DTYPE_E4M3, 64, 4), (wl.DTYPE_BF16, 128, 8),
                                           (wl.DTYPE_BF16, 64, 16), (wl.DTYPE_E4M3, 128, 1)])
def test_indexer_shapes_and_dtypes(dtype, D, heads):
    lens = [0, 1, 31, 32, 127, 128, 129, 1000, 4096, 9216]
    _check(wl.make_indexer_batch("shapes", 70 + D + heads, lens, heads=heads, head_dim=D,
                                 dtype=dtype, topk=16))


@pytest.mark.parametrize("bt,topk,P", [(32, 1, 16), (256, 64, 64), (1024, 5, 48)])
def test_indexer_block_sizes_topk_and_pages(bt, topk, P):
    _check(wl.make_indexer_batch("blocks", 90 + bt, [5, 300, 2000, 5000], block_tokens=bt,
                                 topk=topk, page_size=P))


def test_indexer_rows_longer_than_the_shared_ranking():
    """More than 1,024 blocks per query (40,000 tokens in blocks of 32): the top-k is
    taken from block_scores in global memory instead of the shared-memory ranking."""
    _check(wl.make_indexer_batch("long_rows", 95, [40000, 100, 33000], block_tokens=32, topk=16))


def test_indexer_table_holes_and_padded_pages():
    w = wl.make_indexer_batch("holes", 97, [700, 1500, 64], page_pad_bytes=256)
    pt = np.array(w.page_table, copy=True)
    pt[0, 2] = -1
    pt[1, 5] = 10**6
    w.page_table = pt
    _check(w)


def test_indexer_exact_ties_rank_lower_id_first():
    w = wl.make_indexer_batch("ties", 98, [512], heads=2, head_dim=64, dtype=wl.DTYPE_BF16, topk=4)
    pool = np.array(w.pool_fill, copy=True)
    c, pt = w.cache, w.page_table
    for j in range(128):       # block 3 := block 1, so their scores are identical
        src = c.offset + 2 * (int(pt[0, (128 + j) // 64]) * c.stride_page + (j % 64) * c.stride_token)
        dst = c.offset + 2 * (int(pt[0, (384 + j) // 64]) * c.stride_page + (j % 64) * c.stride_token)
        pool[dst:dst + 128] = pool[src:src + 128]
    dv = _check(w, pool)
    s = dv.block_scores.cpu().numpy()[0]
    top = dv.topk_ids.cpu().numpy()[0].tolist()
    assert s[1] == s[3] and top.index(1) < top.index(3)


def test_indexer_pdl_back_to_back_in_a_graph():
    """Programmatic dependent launch: back-to-back calls in one CUDA graph reuse the
    same output buffers (the score kernel of call i+1 may start while the top-k of
    call i runs), after a kernel that rewrites the queries; results equal a plain
    call's."""
    from paged_kv_cache_msa_gb300 import binding as B
    w = wl.indexer_decode64()
    ref = _check(w)
    dv = DeviceIndexer(w)
    real_q = dv.idx_q.clone()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        dv.idx_q.zero_()
        dv.run(stream=s, launch_flags=B.MSA_LAUNCH_PDL)
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            dv.idx_q.copy_(real_q)            # the previous kernel writes the queries
            for _ in range(4):
                dv.run(stream=s, launch_flags=B.MSA_LAUNCH_PDL)
        for _ in range(3):
            g.replay()
        s.synchronize()
    assert torch.equal(ref.block_scores, dv.block_scores)
    assert torch.equal(ref.topk_ids, dv.topk_ids)



# ---------------------------------------------------------------------------
# decode batches on the tensor-core kernel over a flat (query, block) list
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("case", ["many_short", "limit_1024", "over_limit_1025", "heads_16",
                                  "empty_between", "all_empty", "one_item"])
def test_decode_flat_list_batches(case):
    """E4M3 keys of 128 dims in whole-page boxes: batch shapes that stress the flat item
    list (a CTA's share spanning many queries, the 1,024-query limit and one past it,
    which takes the per-query kernel, 16 heads, histories without a token between
    others, a batch with no item at all and one with a single item, where every CTA or
    all CTAs but one have nothing to score), against the oracle."""
    rng = np.random.default_rng(700 + len(case))
    heads = 8
    if case == "many_short":
        lens = rng.integers(1, 300, size=600)
    elif case == "limit_1024":
        lens = rng.integers(1, 1200, size=1024)
    elif case == "over_limit_1025":
        lens = rng.integers(1, 1200, size=1025)
    elif case == "heads_16":
        lens = rng.integers(1, 9216, size=48)
        heads = 16
    elif case == "all_empty":
        lens = np.zeros(40, dtype=np.int64)
    elif case == "one_item":
        lens = np.array([1])
    else:
        lens = rng.integers(1, 4000, size=64)
        lens[::5] = 0
    _check(wl.make_indexer_batch(f"flat_{case}", 710 + len(case), lens, heads=heads, topk=16))


@pytest.mark.parametrize("P", [8, 32, 128, 256])
def test_decode_flat_list_page_sizes(P):
    """The flat decode kernel with one TMA box per page for page sizes 8 to 128 and
    128-row boxes inside 256-row pages, against the oracle."""
    _check(wl.make_indexer_batch(f"flat_p{P}", 730 + P, [1, 127, 128, 129, 700, 3000, 9216, 0], page_size=P))


# ---------------------------------------------------------------------------
# query runs (prefill): tiles of consecutive queries on the tcgen05 tensor cores
# ---------------------------------------------------------------------------

def _runs():
    from paged_kv_cache_msa_gb300 import binding as B
    return B.MSA_LAUNCH_QUERY_RUNS


@pytest.mark.parametrize("dtype", [wl.DTYPE_E4M3, wl.DTYPE_BF16], ids=["fp8", "bf16"])
@pytest.mark.parametrize("D,heads", [(128, 8), (64, 8), (128, 12), (64, 3)])
def test_query_runs_prefill_shapes(dtype, D, heads):
    """Causal prefill queries of ragged sequences (tiles with partial and empty
    rows, blocks with partial visibility), 8 and 16 rows per query."""
    w = wl.make_indexer_prefill(f"runs{D}_{heads}", 300 + D + heads, [300, 129, 16, 1, 257],
                                heads=heads, head_dim=D, dtype=dtype)
    _check(w, flags=_runs())


@pytest.mark.parametrize("P", [16, 64, 96])
def test_query_runs_interleaved_sequences_and_pages(P):
    """Queries of three sequences in shuffled order: most tiles hold several
    sequences and are scored one sequence at a time; page sizes that split blocks."""
    w = wl.make_indexer_prefill(f"inter{P}", 400 + P, [200, 333, 90], page_size=P,
                                interleave=True, page_pad_bytes=32)
    _check(w, flags=_runs())


@pytest.mark.parametrize("P,pad", [(64, 128), (96, 0), (16, 384), (256, 0), (8, 0), (32, 0), (128, 0),
                                   (64, 16)],
                         ids=["unused_rows_between_pages", "page_96", "page_16_padded", "page_256",
                              "page_8", "page_32", "page_128", "off_the_row_grid"])
def test_query_runs_key_row_layouts(P, pad):
    """E4M3 keys of 128 dims: pages that span a whole number of token rows take the
    TMA key copies (whole pages as boxes for page sizes 8 to 128, 128-row boxes inside
    256-row pages, with unused rows between pages; row gathers for page size 96);
    padding off the row grid takes the register gather.  All against the oracle."""
    w = wl.make_indexer_prefill(f"rows{P}_{pad}", 560 + P + pad, [700, 333, 129], page_size=P,
                                page_pad_bytes=pad)
    _check(w, flags=_runs())


def test_query_runs_in_a_graph_with_two_caches():
    """Query-run calls on two batches with different caches (one on the row grid, one
    off it) captured in one CUDA graph with programmatic dependent launch, replayed
    twice: each call keeps its own key-row tensor map (a by-value kernel argument) and
    equals a plain call bit for bit."""
    from paged_kv_cache_msa_gb300 import binding as B
    ws = [wl.make_indexer_prefill("graph_grid", 571, [300, 129], page_size=64),
          wl.make_indexer_prefill("graph_offgrid", 572, [200, 90], page_size=64, page_pad_bytes=16)]
    flags = _runs()
    ref = []
    for w in ws:
        dv = DeviceIndexer(w)
        dv.run(launch_flags=flags)
        torch.cuda.synchronize()
        ref.append((dv.block_scores.clone(), dv.topk_ids.clone()))
    dvs = [DeviceIndexer(w) for w in ws]
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for dv in dvs:
            dv.run(stream=s, launch_flags=flags)
        s.synchronize()
        for dv in dvs:
            dv.block_scores.fill_(float("nan"))
            dv.topk_ids.fill_(-7)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for dv in dvs:
                dv.run(stream=s, launch_flags=flags | B.MSA_LAUNCH_PDL)
        for _ in range(2):
            g.replay()
        s.synchronize()
    for dv, (rs, rt) in zip(dvs, ref):
        assert torch.equal(dv.block_scores, rs)
        assert torch.equal(dv.topk_ids, rt)


def test_query_runs_table_holes_and_topk_sizes():
    w = wl.make_indexer_prefill("holes_runs", 501, [700, 260], topk=3)
    pt = np.array(w.page_table, copy=True)
    pt[0, 2] = -1
    pt[1, 1] = 10**6
    w.page_table = pt
    _check(w, flags=_runs())


@pytest.mark.parametrize("lens,heads", [
    ([9000, 5, 300, 0, 4000, 128], 8),
    ([70000, 300, 0], 8),                  # 547 blocks a row: past the shared ranking's short rows
    ([70000, 66000, 10, 0], 12),           # 8 queries a tile
], ids=["mixed", "long_rows", "long_rows_12_heads"])
def test_query_runs_long_and_empty_histories(lens, heads):
    """The query-run kernel on one query per sequence, with long and empty histories,
    against the oracle."""
    w = wl.make_indexer_batch(f"runs_rank_{heads}_{len(lens)}", 520 + len(lens) + heads, lens,
                              heads=heads, topk=16)
    _check(w, flags=_runs())


@pytest.mark.parametrize("flags", [0, 4], ids=["per_query", "query_runs"])
@pytest.mark.parametrize("seqs,topk", [([2100], 16), ([1100, 1000, 300], 64)])
def test_top_k_of_several_rows_per_cta(flags, seqs, topk):
    """Batches of 2,048 queries and more with short rows take the top-k kernel that
    ranks up to 16 rows per CTA: against the oracle, through both score kernels
    (including rows past a query's history, written -inf by the top-k kernel)."""
    _check(wl.make_indexer_prefill(f"rows_{len(seqs)}_{topk}", 540 + len(seqs), seqs, topk=topk),
           flags=flags)


def test_query_runs_match_the_per_query_kernel():
    """The same prefill batch through both score kernels: the block scores agree to
    fp32 accumulation error and the -inf pattern is identical."""
    w = wl.make_indexer_prefill("both", 502, [400, 130])
    a = DeviceIndexer(w)
    a.run()
    b = DeviceIndexer(w)
    b.run(launch_flags=_runs())
    torch.cuda.synchronize()
    sa, sb = a.block_scores.cpu().numpy(), b.block_scores.cpu().numpy()
    assert np.array_equal(np.isfinite(sa), np.isfinite(sb))
    fin = np.isfinite(sa)
    assert np.allclose(sa[fin], sb[fin], rtol=1e-5, atol=1e-3)


def test_query_runs_prefill_65536_sampled():
    """The prefill batch (8 x 8192 causal queries, 8 heads x 128, fp8 index-K):
    block scores and top-k of sampled queries -- a random one from every 16-query
    tile, sequence starts and ends, tile edges -- against the oracle (run over a
    process pool); every row's ids a valid ranking of its scores."""
    from dataclasses import replace
    from oracle_pool import indexer_rows
    w = wl.indexer_prefill()
    dv = DeviceIndexer(w)
    dv.run(launch_flags=_runs())
    torch.cuda.synchronize()
    s_all = dv.block_scores.cpu().numpy()
    top_all = dv.topk_ids.cpu().numpy()
    T = w.kv_len.shape[0]
    rng = np.random.default_rng(5)
    tiles = np.arange(0, T, 16)
    per_tile = np.minimum(tiles + rng.integers(0, 16, size=tiles.size), T - 1)
    idx = np.unique(np.concatenate([[0, 1, 15, 16, 17, 8191, 8192, 8193, T - 17, T - 16, T - 1],
                                    rng.integers(0, T, size=37), per_tile]))
    sub = replace(w, idx_q=np.ascontiguousarray(w.idx_q[idx]), kv_len=w.kv_len[idx].copy(),
                  table_offset=w.table_offset[idx].copy())
    ref_s, ref_top = indexer_rows(w, idx, wl.indexer_cache_arg(w, w.pool_fill))
    check_indexer_against_reference(sub, s_all[idx], top_all[idx], ref_s.astype(np.float64), ref_top)
    fin = np.isfinite(s_all)
    nfin = fin.sum(axis=1)
    assert np.array_equal(nfin, np.minimum(-(-w.kv_len // 128), w.max_blocks))
    for t in rng.integers(0, T, size=200):
        ids = [i for i in top_all[t] if i >= 0]
        vals = [s_all[t, i] for i in ids]
        assert len(ids) == min(w.topk, int(nfin[t]))
        assert all(vals[i] >= vals[i + 1] for i in range(len(vals) - 1))


def test_decode_layer_producer_then_indexer_in_a_graph():
    """The producer and the indexer chained as a decode layer (the indexer reads
    the compact index-Q and the index-K cache the producer just wrote), launched
    with programmatic dependent launch, 3 layers captured in one CUDA graph: the
    same bytes as the two kernels launched plainly one after the other."""
    from paged_kv_cache_msa_gb300 import binding as B
    from paged_kv_cache_msa_gb300.device import DecodeLayer, DeviceWorkload
    w = wl.config2_decode64()
    plain, chained = [], []
    for _ in range(3):
        plain.append(DecodeLayer(DeviceWorkload(w), max_blocks_per_seq=144))
        chained.append(DecodeLayer(DeviceWorkload(w), max_blocks_per_seq=144))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for layer in plain:
            layer.run(s, 0)
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for layer in chained:
                layer.run(s, B.MSA_LAUNCH_PDL)
        g.replay()
        s.synchronize()
    for a, b in zip(plain, chained):
        assert torch.equal(a.dw.q_out, b.dw.q_out) and torch.equal(a.dw.idx_q_out, b.dw.idx_q_out)
        for k in a.dw.pools:
            assert torch.equal(a.dw.pools[k], b.dw.pools[k])
        assert torch.equal(a.block_scores, b.block_scores)
        assert torch.equal(a.topk_ids, b.topk_ids)
        fin = torch.isfinite(a.block_scores).sum(dim=1)
        assert int(fin.min()) >= 1      # every token sees at least one scored block
