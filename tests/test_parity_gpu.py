"""Parity of the CUDA producer with the oracle, through the C ABI (GPU).

Tolerances (stated by the producer's specification): placement and the set of
written bytes exact; compact bf16 Q / index-Q within 2e-2 + 1e-2*|ref|; fp8
cache entries within one E4M3 step; bf16 cache entries like Q.
"""
import numpy as np
import pytest
import torch

from paged_kv_cache_msa_gb300 import binding as B
from paged_kv_cache_msa_gb300 import build as build_mod
from paged_kv_cache_msa_gb300 import workloads as wl
from paged_kv_cache_msa_gb300.device import DeviceWorkload

from gpu_harness import check_against_oracle
from harness import compare_bf16, run_oracle

pytestmark = pytest.mark.gpu

ONE_SHOT = 0
PERSISTENT = B.MSA_LAUNCH_PERSISTENT
FLAGS = [ONE_SHOT, PERSISTENT, PERSISTENT | B.MSA_LAUNCH_PDL]
FLAG_IDS = ["one_shot", "persistent", "persistent_pdl"]


@pytest.fixture(scope="module", autouse=True)
def library():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build_mod.build()
    return B.load()


# ---------------------------------------------------------------------------
# the five workloads
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("flags", FLAGS, ids=FLAG_IDS)
def test_config1_tiny_decode(flags):
    check_against_oracle(wl.config1_tiny_decode(), flags)


@pytest.mark.parametrize("flags", [ONE_SHOT, PERSISTENT], ids=FLAG_IDS[:2])
def test_config2_decode64_padded_hnd_pages(flags):
    check_against_oracle(wl.config2_decode64(), flags)


def test_config3_decode_step_layers_tiny_and_big():
    for layer in (0, 1, 59):
        check_against_oracle(wl.config3_decode_step(layer), PERSISTENT)
    check_against_oracle(wl.config3_decode_step(7, big=True), PERSISTENT)


def test_config4_prefill_full_size():
    """65,536 tokens, every output and cache cell against the oracle."""
    w = wl.config4_prefill()
    check_against_oracle(w, PERSISTENT)


def test_config5_mixed_over_2_31_elements():
    w = wl.config5_mixed()
    kv = w.caches["v"]
    # the pool really needs 64-bit offsets: written pages beyond 2^31 elements
    assert kv.num_pages * kv.stride_page > 2**31
    check_against_oracle(w, PERSISTENT)


# ---------------------------------------------------------------------------
# edge cases
# ---------------------------------------------------------------------------

def _small(seed, heads=wl.TINY, T_seqs=5, positions_hi=300, **kw):
    rng = np.random.default_rng(seed)
    seq_positions = [[int(p)] for p in rng.integers(0, positions_hi, size=T_seqs)]
    max_blocks = -(-positions_hi // kw.get("page_size", 64))
    npages = kw.pop("num_pages", T_seqs * max_blocks)
    return wl.make_batch(f"edge{seed}", seed, heads, seq_positions, max_blocks=max_blocks,
                         num_pages=npages, **kw)


@pytest.mark.parametrize("flags", FLAGS, ids=FLAG_IDS)
def test_zero_tokens_launches_nothing(flags):
    w = _small(1)
    dw = DeviceWorkload(w)
    before = {k: v.clone() for k, v in dw.pools.items()}
    assert dw.run(flags, num_tokens=0) == B.MSA_OK
    torch.cuda.synchronize()
    for k in before:
        assert torch.equal(before[k], dw.pools[k])


def test_all_tokens_padded_write_only_q():
    w = _small(2, T_seqs=9)
    w.slot_mapping[:] = -1
    w.meta["valid_mask"][:] = False
    check_against_oracle(w, PERSISTENT)


@pytest.mark.parametrize("T", [1, 3, 31, 257, 1000])
def test_ragged_token_counts(T):
    rng = np.random.default_rng(T)
    seq_positions = [list(range(int(s), int(s) + T))
                     for s in rng.integers(0, 64, size=1)]
    w = wl.make_batch(f"ragged{T}", 100 + T, wl.BIG, seq_positions, max_blocks=-(-(T + 64) // 64),
                      num_pages=64, rotary_dim=64, pad_frac=0.1)
    for flags in (ONE_SHOT, PERSISTENT):
        check_against_oracle(w, flags)


@pytest.mark.parametrize("style,rd,D", [
    (wl.ROPE_NEOX, 0, 64), (wl.ROPE_NEOX, 16, 64), (wl.ROPE_NEOX, 32, 128),
    (wl.ROPE_NEOX, 96, 128), (wl.ROPE_GPTJ, 64, 64), (wl.ROPE_GPTJ, 8, 64),
    (wl.ROPE_GPTJ, 128, 128), (wl.ROPE_GPTJ, 40, 128),
])
def test_rope_variants(style, rd, D):
    heads = wl.TINY if D == 64 else wl.BIG
    w = _small(300 + rd + D, heads=heads, rotary_dim=rd, rope_style=style)
    check_against_oracle(w, PERSISTENT)


@pytest.mark.parametrize("draft_len", [1, 3, 7])
def test_multi_token_decode_rows(draft_len):
    """Speculative verify: every sequence brings 1 + draft_len new tokens at consecutive
    positions (some crossing a page boundary), each with its own slot."""
    rng = np.random.default_rng(50 + draft_len)
    S = 48
    starts = rng.integers(0, 1024 - draft_len - 1, size=S)
    starts[:4] = [63 - draft_len // 2, 127 - draft_len, 0, 64]   # page-boundary crossings
    seq_positions = [list(range(int(s0), int(s0) + 1 + draft_len)) for s0 in starts]
    w = wl.make_batch(f"verify{draft_len}", 60 + draft_len, wl.BIG, seq_positions, max_blocks=16,
                      num_pages=S * 16, pad_frac=0.05)
    for flags in (PERSISTENT, PERSISTENT | B.MSA_LAUNCH_PDL):
        check_against_oracle(w, flags)


def test_physical_slots_without_page_table():
    w = _small(4, T_seqs=40, use_page_table=False, pad_frac=0.2)
    assert w.page_table is None
    check_against_oracle(w, ONE_SHOT)


def test_no_index_k_cache():
    w = _small(5, T_seqs=16, with_idx_k=False)
    check_against_oracle(w, PERSISTENT)


def test_dense_layer_without_index_heads():
    heads = dict(num_q_heads=16, num_kv_heads=4, num_idx_q_heads=0, num_idx_k_heads=0, head_dim=128)
    w = _small(6, heads=heads, T_seqs=12, with_idx_k=False)
    check_against_oracle(w, PERSISTENT)


def test_bf16_kv_caches_and_fp8_index_k():
    w = _small(7, heads=wl.BIG, T_seqs=20, kv_dtype=wl.DTYPE_BF16, idx_k_dtype=wl.DTYPE_E4M3)
    check_against_oracle(w, PERSISTENT)


def test_per_head_scales():
    w = _small(8, heads=wl.BIG, T_seqs=20, scale_mode=1)
    rng = np.random.default_rng(8)
    w.scales = rng.uniform(0.01, 0.2, size=w.scales.shape).astype(np.float32)
    check_against_oracle(w, PERSISTENT)


def test_per_head_scales_many_tokens_per_cta():
    """Per-head scales when each CTA of the persistent grid has many tokens (about 40):
    the kernel then takes the caches' reciprocal scales from a per-CTA table instead of
    computing them per head row; 40 prefill sequences of 456 tokens."""
    rng = np.random.default_rng(18)
    seq_positions = [list(range(int(s0), int(s0) + 456)) for s0 in rng.integers(0, 4000, size=40)]
    w = wl.make_batch("per_head_many", 18, wl.BIG, seq_positions, max_blocks=72, num_pages=40 * 72,
                      scale_mode=1, pad_frac=0.05)
    w.scales = rng.uniform(0.01, 0.2, size=w.scales.shape).astype(np.float32)
    check_against_oracle(w, PERSISTENT)


def test_saturation_with_small_scale_and_outliers():
    w = _small(9, heads=wl.BIG, T_seqs=20, outlier_frac=0.05, scale=0.002)
    check_against_oracle(w, PERSISTENT)


def test_large_positions():
    w = _small(10, heads=wl.TINY, T_seqs=16, positions_hi=1 << 19, num_pages=16 * 8192)
    check_against_oracle(w, PERSISTENT)


def test_page_size_not_a_power_of_two():
    w = _small(11, heads=wl.TINY, T_seqs=24, page_size=48, positions_hi=480)
    check_against_oracle(w, PERSISTENT)


def test_many_heads_take_several_register_batches():
    heads = dict(num_q_heads=160, num_kv_heads=16, num_idx_q_heads=8, num_idx_k_heads=2, head_dim=128)
    w = _small(12, heads=heads, T_seqs=10)
    check_against_oracle(w, PERSISTENT)


def test_nhd_cache_layout():
    w = _small(13, heads=wl.BIG, T_seqs=24)
    # NHD pages [P, H, D] over the same pools
    for key in ("k", "v"):
        c = w.caches[key]
        c.stride_head, c.stride_token = 128, c.num_heads * 128
    check_against_oracle(w, PERSISTENT)


def test_table_entries_out_of_range_and_past_the_table():
    w = _small(14, heads=wl.TINY, T_seqs=30)
    pt = np.array(w.page_table, copy=True)
    pt.reshape(-1)[::3] = -1
    pt.reshape(-1)[1::5] = 10**6
    w.page_table = pt
    w.slot_mapping[::7] = pt.size * 64 + 5        # logical block past the table
    check_against_oracle(w, PERSISTENT)


def test_cache_with_fewer_pages_than_the_others():
    w = _small(15, heads=wl.TINY, T_seqs=30)
    w.caches["idx_k"].num_pages = w.caches["idx_k"].num_pages // 2
    check_against_oracle(w, PERSISTENT)


# ---------------------------------------------------------------------------
# CUDA graphs
# ---------------------------------------------------------------------------

def test_graph_replay_sees_new_inputs():
    """One capture, two replays with different row contents and slots."""
    w1 = _small(20, heads=wl.BIG, T_seqs=32)
    w2 = _small(21, heads=wl.BIG, T_seqs=32)
    # the captured call keeps its pointers: only the contents of the rows,
    # positions and slots change between replays
    w2.page_table, w2.weights, w2.scales = w1.page_table, w1.weights, w1.scales
    dw = DeviceWorkload(w1)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        dw.run(PERSISTENT, stream=s)
    for w in (w1, w2):
        dw.qkv.copy_(torch.from_numpy(w.qkv.view(np.int16)))
        dw.positions.copy_(torch.from_numpy(w.positions))
        dw.slots.copy_(torch.from_numpy(w.slot_mapping))
        g.replay()
        torch.cuda.synchronize()
        q_o, iq_o, _ = run_oracle(w)
        q_d, iq_d = dw.outputs_to_host()
        compare_bf16(q_d, q_o, "q_out")
        compare_bf16(iq_d, iq_o, "idx_q_out")


def test_sixty_layer_decode_step_in_one_graph():
    """60 tiny-shape layers at batch 256, each with its own pools, captured as 60
    launches in one graph; every layer checked against the oracle after replay."""
    from harness import e4m3_ulp_distance
    layers = [wl.config3_decode_step(l) for l in range(60)]
    dws = [DeviceWorkload(w) for w in layers]
    sentinels = [wl.host_pools(w) for w in layers]
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for dw in dws:
            dw.run(PERSISTENT | B.MSA_LAUNCH_PDL, stream=s)
    g.replay()
    torch.cuda.synchronize()
    from gpu_harness import oracle_written_mask
    for w, dw, sent in zip(layers, dws, sentinels):
        q_o, iq_o, pools_o = run_oracle(w)
        q_d, iq_d = dw.outputs_to_host()
        compare_bf16(q_d, q_o, f"{w.name} q_out")
        compare_bf16(iq_d, iq_o, f"{w.name} idx_q_out")
        masks = oracle_written_mask(w)
        pools_d = dw.pools_to_host()
        for name in w.pools:
            m = masks[name]
            assert np.array_equal(pools_d[name][~m], sent[name][~m]), f"{w.name}: stray write"
            if w.caches[name].dtype == wl.DTYPE_E4M3:
                assert e4m3_ulp_distance(pools_d[name][m], pools_o[name][m]).max(initial=0) <= 1
            else:
                compare_bf16(pools_d[name][m].view(np.uint16), pools_o[name][m].view(np.uint16), name)


def test_pdl_chain_reads_metadata_staged_launches_back():
    """Under programmatic dependent launch the producer reads its positions and slots
    before waiting on the kernels ahead of it, and lets the next kernel start at once,
    so a run of such launches may be in flight together; the metadata must be staged
    by kernels launched without programmatic dependent launch before the run.  Per
    layer, in one CUDA graph: copy kernels stage the layer's positions and slots, the
    indexer runs (its kernels launched with PDL), another layer's producer runs
    (PDL), then this layer's producer (PDL): the metadata it reads first was written
    two and more launches back.  The buffers start stale (slots -1, positions 0x7fff);
    every layer must match the oracle."""
    from harness import e4m3_ulp_distance
    from gpu_harness import oracle_written_mask
    from paged_kv_cache_msa_gb300.device import DeviceIndexer
    n_layers = 12
    layers = [wl.config3_decode_step(l) for l in range(n_layers)]
    others = [wl.config3_decode_step(200 + l) for l in range(n_layers)]
    dws = [DeviceWorkload(w) for w in layers]
    dos = [DeviceWorkload(w) for w in others]
    iw = wl.indexer_decode64()
    ix = DeviceIndexer(iw)
    slot_src = [dw.slots.clone() for dw in dws]
    pos_src = [dw.positions.clone() for dw in dws]
    s = torch.cuda.Stream()
    flags = PERSISTENT | B.MSA_LAUNCH_PDL
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for dw, do, ss, ps in zip(dws, dos, slot_src, pos_src):
            dw.slots.copy_(ss)
            dw.positions.copy_(ps)
            ix.run(stream=s, launch_flags=B.MSA_LAUNCH_PDL)
            do.run(flags, stream=s)
            dw.run(flags, stream=s)
    for dw in dws:
        dw.slots.fill_(-1)
        dw.positions.fill_(0x7FFF)
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    for w, dw in zip(layers, dws):
        sent = wl.host_pools(w)
        q_o, iq_o, pools_o = run_oracle(w)
        q_d, iq_d = dw.outputs_to_host()
        compare_bf16(q_d, q_o, f"{w.name} q_out")
        compare_bf16(iq_d, iq_o, f"{w.name} idx_q_out")
        masks = oracle_written_mask(w)
        pools_d = dw.pools_to_host()
        for name in w.pools:
            m = masks[name]
            assert m.any(), f"{w.name}: the slots should place tokens in {name}"
            assert np.array_equal(pools_d[name][~m], sent[name][~m]), f"{w.name}: stray write"
            if w.caches[name].dtype == wl.DTYPE_E4M3:
                assert e4m3_ulp_distance(pools_d[name][m], pools_o[name][m]).max(initial=0) <= 1
            else:
                compare_bf16(pools_d[name][m].view(np.uint16), pools_o[name][m].view(np.uint16), name)
