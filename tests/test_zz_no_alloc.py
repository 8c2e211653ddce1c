"""msa_indexer_forward_fused_noalloc: the single-launch indexer on the library's own
counters.  Two calls in a row must each equal the allocating single-launch entry's
results bit for bit (the first call on the device clears the counters, every call
leaves them zero for the next), and agree with the two-kernel entry (bit for bit,
or within the oracle tolerance where that entry takes the tensor-core decode
kernel).  The file is collected last so that it also runs after every other test
in the same process."""
import pytest
import torch

from paged_kv_cache_msa_gb300 import binding as B
from paged_kv_cache_msa_gb300 import build as build_mod
from paged_kv_cache_msa_gb300 import workloads as wl
from paged_kv_cache_msa_gb300.device import DeviceIndexer

from oracle_pins import same_indexer_results as same_results

BASE = 0x7F0000000000


def _noalloc(dv, flags=0):
    p = lambda t: int(t.data_ptr())
    B.msa_indexer_forward_fused_noalloc(dv.cfg, dv.w.idx_q.shape[0], p(dv.idx_q), p(dv.kv_len),
                                        p(dv.table_offset), p(dv.page_table), dv.page_table.numel(),
                                        dv.cache, p(dv.k_scale), p(dv.block_scores), p(dv.topk_ids),
                                        flags, stream=torch.cuda.current_stream().cuda_stream)


@pytest.mark.gpu
@pytest.mark.parametrize("make", [
    wl.indexer_decode64,
    lambda: wl.make_indexer_batch("noalloc", 211, [0, 1, 129, 513, 4096, 9216, 0, 640], topk=16),
], ids=["decode64", "ragged_with_empty"])
def test_two_calls_match_the_allocating_entry_points(make):
    build_mod.build()
    w = make()
    ref = DeviceIndexer(w)
    ref.run(fused=True)                 # caller-owned counters
    two = DeviceIndexer(w)
    two.run()                           # score kernel + top-k kernel
    torch.cuda.synchronize()
    same_results(w, ref.block_scores, ref.topk_ids, two.block_scores, two.topk_ids)
    for call in range(2):
        dv = DeviceIndexer(w)
        dv.block_scores.fill_(float("nan"))
        dv.topk_ids.fill_(-7)
        _noalloc(dv, B.MSA_LAUNCH_PDL if call else 0)
        torch.cuda.synchronize()
        assert torch.equal(ref.block_scores, dv.block_scores), call
        assert torch.equal(ref.topk_ids, dv.topk_ids), call


def test_batches_above_the_library_counters_are_rejected_on_the_host():
    build_mod.build()
    cfg = B.make_indexer_cfg(8, 128, 64, 128, 16, 72)
    cache = B.make_cache(BASE + 20 * 2**34, B.MSA_DTYPE_FP8_E4M3, 9216, 1, 64 * 128, 64 * 128, 128)
    args = (cfg, 65537, BASE, BASE + 2**32, BASE + 2 * 2**32, BASE + 3 * 2**32, 10**6, cache,
            BASE + 4 * 2**32, BASE + 5 * 2**32, BASE + 6 * 2**32)
    got = B.msa_indexer_forward_fused_noalloc(*args, 0, stream=0, check=False)
    assert got == B.MSA_ERR_UNSUPPORTED, B.last_error_detail()
    got = B.msa_indexer_forward_fused_noalloc(cfg, 0, None, *args[3:], 0, stream=0, check=False)
    assert got == B.MSA_OK, B.last_error_detail()
