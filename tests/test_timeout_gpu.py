"""The bounded-wait timeout path, on the GPU, in the starved test build (GPU).

Every wait of the kernels on an mbarrier (operand tiles landed, accumulator
complete or drained in the projection; keys staged, MMA done, query tile loaded in
the query-run indexer) gives up after a time limit instead of spinning forever.
The starved build (``build.build_starved()``: -DMSA_STARVE, limit 50 ms) makes
those waits run out on purpose, safely: the projection's TMA warps and the
indexer's MMA thread issue nothing, so no copy and no MMA is ever in flight when a
wait gives up.  Each kernel must then stop without writing any output (the
projection) or score every block it could not finish NaN (the indexer), report
the timeout (the projection's status word) and release its tensor memory: a
normal call right after, on the normal library, must match the oracle.  (The
producer kernel has no such wait: its rows are staged with cp.async, whose
wait_group cannot spin.)"""
import numpy as np
import pytest
import torch

from paged_kv_cache_msa_gb300 import binding as B
from paged_kv_cache_msa_gb300 import build as build_mod
from paged_kv_cache_msa_gb300 import workloads as wl
from paged_kv_cache_msa_gb300.device import DeviceIndexer, DeviceProjection

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def libs():
    normal = B.load(build_mod.build())
    starved = B.load(build_mod.build_starved())
    saved = B._lib
    yield normal, starved
    B._lib = saved


def _use(lib):
    B._lib = lib


def _snapshot(tensors):
    return [t.clone() for t in tensors]


def _unchanged(before, tensors):
    return all(torch.equal(a, b) for a, b in zip(before, tensors))


@pytest.mark.parametrize("T,hidden,heads", [(300, 200, "tiny"), (64, 512, "big")],
                         ids=["two_sm_kernel", "split_over_k"])
def test_projection_stops_and_reports(libs, T, hidden, heads):
    from test_projection_gpu import _batch, check_projection
    normal, starved = libs
    shape = wl.TINY if heads == "tiny" else dict(wl.BIG, num_q_heads=6)
    pw = _batch(700 + T, shape, T, hidden, pad_frac=0.1)
    _use(starved)
    dp = DeviceProjection(pw, rows_out=True)
    outs = [dp.dw.q_out, dp.dw.idx_q_out, dp.rows_out] + [dp.pools[k] for k in sorted(dp.pools)]
    before = _snapshot(outs)
    torch.cuda.synchronize()
    dp.run()
    torch.cuda.synchronize()
    assert int(dp.status.item()) & B.MSA_STATUS_WAIT_TIMEOUT
    assert _unchanged(before, outs), "a timed-out projection wrote an output"
    _use(normal)
    check_projection(pw)


@pytest.mark.parametrize("pad", [0, 16], ids=["tma_key_rows", "register_gather"])
def test_query_run_indexer_scores_nan_and_selects_nothing(libs, pad):
    """Both query-run kernels: E4M3 keys on one row grid (TMA key copies) and off it
    (the register gather)."""
    from test_indexer_gpu import _check
    normal, starved = libs
    w = wl.make_indexer_prefill(f"starved_runs_{pad}", 901, [40, 200, 7], page_pad_bytes=pad)
    _use(starved)
    dv = DeviceIndexer(w)
    dv.run(launch_flags=B.MSA_LAUNCH_QUERY_RUNS)
    torch.cuda.synchronize()
    s = dv.block_scores.cpu().numpy()
    top = dv.topk_ids.cpu().numpy()
    nb = -(-w.kv_len.astype(np.int64) // w.block_tokens)
    for t in range(s.shape[0]):
        assert np.isnan(s[t, :nb[t]]).all(), t          # every block the query sees
        assert (np.isnan(s[t]) | (s[t] == -np.inf)).all(), t
    assert (top == -1).all(), "a block whose wait ran out must never be selected"
    _use(normal)
    _check(w, flags=B.MSA_LAUNCH_QUERY_RUNS)
