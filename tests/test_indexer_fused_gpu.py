"""The single-launch indexer (msa_indexer_forward_fused) against the two-kernel one
and the oracle, through the C ABI (GPU).

The fused entry runs the per-query score kernel with the top-k taken by the last CTA
of each query.  The two-kernel path runs the same kernel, except for decode batches
of E4M3 keys in whole-page boxes, which take the tensor-core kernel over a flat item
list (E4M3 query halves, so its scores differ within the oracle tolerance).  So the
two entries must agree bit for bit, or within that tolerance with the same ids
wherever the scores separate them; both must pass the oracle check, and the
per-query counters must be zero again after every launch."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_msa_gb300 import binding as B
from paged_kv_cache_msa_gb300 import build as build_mod
from paged_kv_cache_msa_gb300 import workloads as wl
from paged_kv_cache_msa_gb300.device import DeviceIndexer

from oracle_pins import check_indexer_against_reference, same_indexer_results as same_results

pytestmark = pytest.mark.gpu


def _both(w, pool=None, flags=0):
    """(two-kernel indexer, fused indexer) after one call each on the same inputs."""
    build_mod.build()
    two = DeviceIndexer(w, pool=pool)
    two.run(launch_flags=flags)
    fused = DeviceIndexer(w, pool=pool)
    fused.block_scores.fill_(float("nan"))     # every entry must be written
    fused.topk_ids.fill_(-7)
    fused.run(launch_flags=flags, fused=True)
    torch.cuda.synchronize()
    return two, fused


def _check(w, pool=None, flags=0):
    two, fused = _both(w, pool, flags)
    same_results(w, fused.block_scores, fused.topk_ids, two.block_scores, two.topk_ids)
    assert int(fused.counters.abs().sum().item()) == 0
    pool = w.pool_fill if pool is None else pool
    ref_s, ref_top = oracle.indexer(w.idx_q, w.kv_len, w.table_offset, w.page_table,
                                    wl.indexer_cache_arg(w, pool), w.k_scale, w.page_size,
                                    w.block_tokens, w.topk, w.max_blocks)
    check_indexer_against_reference(w, fused.block_scores.cpu().numpy(), fused.topk_ids.cpu().numpy(),
                                    ref_s.astype(np.float64), ref_top)
    return fused


def test_fused_decode64():
    _check(wl.indexer_decode64())


@pytest.mark.parametrize("dtype,D,heads", [(wl.DTYPE_E4M3, 64, 4), (wl.DTYPE_BF16, 128, 8),
                                           (wl.DTYPE_BF16, 64, 16), (wl.DTYPE_E4M3, 128, 1)])
def test_fused_shapes_and_dtypes_with_empty_histories(dtype, D, heads):
    # lengths 0 (no CTA scores: the query's first CTA ranks alone), 1, block and CTA
    # boundaries (a CTA spans 4 blocks), and the longest history
    lens = [0, 1, 127, 128, 129, 511, 512, 513, 1000, 4096, 9216, 0]
    _check(wl.make_indexer_batch("fused_shapes", 170 + D + heads, lens, heads=heads, head_dim=D,
                                 dtype=dtype, topk=16))


@pytest.mark.parametrize("bt,topk,P", [(32, 1, 16), (256, 64, 64), (1024, 5, 48)])
def test_fused_block_sizes_topk_and_pages(bt, topk, P):
    _check(wl.make_indexer_batch("fused_blocks", 190 + bt, [5, 300, 2000, 5000], block_tokens=bt,
                                 topk=topk, page_size=P))


def test_fused_rows_longer_than_the_shared_ranking():
    """More than 1,024 blocks per query: the last CTA ranks from global memory, which
    other CTAs of the same launch wrote."""
    _check(wl.make_indexer_batch("fused_long", 195, [40000, 100, 33000, 0], block_tokens=32, topk=16))


def test_fused_table_holes_and_padded_pages():
    w = wl.make_indexer_batch("fused_holes", 197, [700, 1500, 64], page_pad_bytes=256)
    pt = np.array(w.page_table, copy=True)
    pt[0, 2] = -1
    pt[1, 5] = 10**6
    w.page_table = pt
    _check(w)


def test_fused_back_to_back_in_a_graph_with_pdl():
    """Four back-to-back single-launch calls per graph, replayed three times, with
    programmatic dependent launch, after a kernel that rewrites the queries: the
    counters return to zero after every call and the results equal a plain call's."""
    w = wl.indexer_decode64()
    ref = _check(w)
    dv = DeviceIndexer(w)
    real_q = dv.idx_q.clone()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        dv.idx_q.zero_()
        dv.run(stream=s, launch_flags=B.MSA_LAUNCH_PDL, fused=True)
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            dv.idx_q.copy_(real_q)            # the previous kernel writes the queries
            for _ in range(4):
                dv.run(stream=s, launch_flags=B.MSA_LAUNCH_PDL, fused=True)
        for _ in range(3):
            g.replay()
        s.synchronize()
    assert torch.equal(ref.block_scores, dv.block_scores)
    assert torch.equal(ref.topk_ids, dv.topk_ids)
    assert int(dv.counters.abs().sum().item()) == 0


def test_fused_entry_with_query_runs_leaves_the_counters_alone():
    """With MSA_LAUNCH_QUERY_RUNS the fused entry runs the query-run kernel and the
    top-k kernel; the counters are not read or written."""
    w = wl.make_indexer_prefill("fused_runs", 199, [300, 129, 16], topk=8)
    build_mod.build()
    two = DeviceIndexer(w)
    two.run(launch_flags=B.MSA_LAUNCH_QUERY_RUNS)
    dv = DeviceIndexer(w)
    dv.counters.fill_(7)
    dv.run(launch_flags=B.MSA_LAUNCH_QUERY_RUNS, fused=True)
    torch.cuda.synchronize()
    assert torch.equal(two.block_scores, dv.block_scores)
    assert torch.equal(two.topk_ids, dv.topk_ids)
    assert bool((dv.counters == 7).all())


def test_fused_decode_layer_in_a_graph():
    """Producer then the single-launch indexer, 4 layers in one graph with PDL: every
    layer's ids and scores agree with the two-kernel path's (see same_results)."""
    from paged_kv_cache_msa_gb300.device import DecodeLayer, DeviceWorkload
    build_mod.build()
    w = wl.config2_decode64()
    layers = [DecodeLayer(DeviceWorkload(w), max_blocks_per_seq=144) for _ in range(4)]
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for layer in layers:
            layer.run(s, B.MSA_LAUNCH_PDL)
        s.synchronize()
        ref = [(l.block_scores.clone(), l.topk_ids.clone()) for l in layers]
        for l in layers:
            l.block_scores.fill_(float("nan"))
            l.topk_ids.fill_(-7)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for layer in layers:
                layer.run(s, B.MSA_LAUNCH_PDL, fused=True)
        for _ in range(2):
            g.replay()
        s.synchronize()
    from types import SimpleNamespace
    for l, (rs, rt) in zip(layers, ref):
        same_results(SimpleNamespace(topk=int(rt.shape[1])), l.block_scores, l.topk_ids, rs, rt)
        assert int(l.counters.abs().sum().item()) == 0
