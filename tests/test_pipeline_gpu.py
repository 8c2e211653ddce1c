"""The host pipeline (chunked copies in, producer, copies out) against a direct
device run: per-token results do not depend on chunking, so outputs and cache
bytes must be identical (GPU)."""
import numpy as np
import pytest
import torch

from paged_kv_cache_msa_gb300 import binding as B
from paged_kv_cache_msa_gb300 import build as build_mod
from paged_kv_cache_msa_gb300 import workloads as wl
from paged_kv_cache_msa_gb300.device import DeviceWorkload
from paged_kv_cache_msa_gb300.pipeline import HostPipeline

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("chunk", [1000, 4096, 20000])
def test_host_pipeline_matches_device_run(chunk):
    build_mod.build()
    w = wl.config4_prefill(num_seqs=2, seq_len=4096)      # 8,192 tokens, ragged last chunk
    ref = DeviceWorkload(w)
    ref.run(B.MSA_LAUNCH_PERSISTENT)
    dw = DeviceWorkload(w)
    pipe = HostPipeline(dw.cfg, w.row_stride, min(chunk, w.num_tokens), dw.qkv.device,
                        (dw.weights["q"], dw.weights["k"], dw.weights["idx_q"], dw.weights["idx_k"]),
                        (dw.caches["k"], dw.caches["v"], dw.caches["idx_k"]), dw.scales,
                        dw.page_table, B.MSA_LAUNCH_PERSISTENT)
    h_qkv = torch.from_numpy(w.qkv.view(np.int16)).pin_memory()
    h_pos = torch.from_numpy(w.positions).pin_memory()
    h_slot = torch.from_numpy(w.slot_mapping).pin_memory()
    h_q = torch.zeros(dw.q_out.shape, dtype=torch.int16).pin_memory()
    h_iq = torch.zeros(dw.idx_q_out.shape, dtype=torch.int16).pin_memory()
    for _ in range(2):                                     # slots are reused across calls
        pipe.run(h_qkv, h_pos, h_slot, h_q, h_iq)
    torch.cuda.synchronize()
    assert torch.equal(h_q, ref.q_out.cpu()) and torch.equal(h_iq, ref.idx_q_out.cpu())
    h_q.zero_()
    h_iq.zero_()
    pipe.run_zero_copy(h_qkv, h_pos, h_slot, h_q, h_iq)
    torch.cuda.synchronize()
    assert torch.equal(h_q, ref.q_out.cpu()) and torch.equal(h_iq, ref.idx_q_out.cpu())
    for name in w.pools:
        assert torch.equal(dw.pools[name], ref.pools[name]), name


def test_pageable_host_memory_is_refused():
    build_mod.build()
    a = np.zeros(1024, dtype=np.int16)
    assert B.msa_host_buffer_device_address(a.ctypes.data) is None
    t = torch.zeros(1024, dtype=torch.int16).pin_memory()
    assert B.msa_host_buffer_device_address(t.data_ptr()) is not None
