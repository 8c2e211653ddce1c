"""Device-resident buffers for a workload, and the C-ABI call on them.

``DeviceWorkload`` copies a ``workloads.Workload`` (rows, positions, slots, page
table, weights, scales and sentinel-filled cache pools) into CUDA memory with
torch, builds the cache descriptors, and calls ``msa_producer_forward`` through
the binding.  torch is used for memory and streams only.
"""
from __future__ import annotations

import numpy as np

from . import binding as B
from . import workloads as wl


def _t(a: np.ndarray, device):
    import torch
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


class DeviceWorkload:
    def __init__(self, w: wl.Workload, device="cuda", host_pools: dict | None = None,
                 pools_on_device: dict | None = None):
        import torch
        self.w = w
        self.device = torch.device(device)
        s = w.shape
        self.cfg = B.make_cfg(s["num_q_heads"], s["num_kv_heads"], s["num_idx_q_heads"],
                              s["num_idx_k_heads"], s["head_dim"], s["rotary_dim"], s["rope_style"],
                              s["page_size"], s["rope_theta"], s["rms_eps"], s.get("scale_mode", 0))
        self.qkv = _t(w.qkv, self.device)
        self.positions = _t(w.positions, self.device)
        self.slots = _t(w.slot_mapping, self.device)
        self.page_table = None if w.page_table is None else _t(w.page_table.reshape(-1), self.device)
        self.weights = {k: (None if v is None else _t(v, self.device)) for k, v in w.weights.items()}
        self.scales = _t(w.scales, self.device)
        T, D = w.num_tokens, s["head_dim"]
        self.q_out = torch.zeros((T, s["num_q_heads"], D), dtype=torch.int16, device=self.device)
        self.idx_q_out = torch.zeros((T, s["num_idx_q_heads"], D), dtype=torch.int16,
                                     device=self.device)
        if pools_on_device is not None:
            self.pools = pools_on_device
        else:
            if host_pools is None:
                host_pools = wl.host_pools(w)
            self.pools = {k: _t(v, self.device) for k, v in host_pools.items()}
        self.caches = {}
        for key in ("k", "v", "idx_k"):
            c = w.caches.get(key)
            self.caches[key] = None if c is None else B.make_cache(
                self.pools[c.pool].data_ptr() + c.offset, c.dtype, c.num_pages, c.num_heads,
                c.stride_page, c.stride_head, c.stride_token)

    def args(self, launch_flags=0, num_tokens=None, qkv_ptr=None):
        """Positional arguments of msa_producer_forward minus the stream."""
        w = self.w
        p = lambda t: None if t is None else int(t.data_ptr())
        T = w.num_tokens if num_tokens is None else int(num_tokens)
        return (self.cfg, T, p(self.qkv) if qkv_ptr is None else qkv_ptr, w.row_stride,
                p(self.positions), p(self.slots), p(self.page_table),
                0 if self.page_table is None else self.page_table.numel(),
                p(self.weights.get("q")), p(self.weights.get("k")), p(self.weights.get("idx_q")),
                p(self.weights.get("idx_k")), p(self.q_out), p(self.idx_q_out),
                self.caches["k"], self.caches["v"], self.caches["idx_k"], p(self.scales),
                launch_flags)

    def run(self, launch_flags=0, stream=None, num_tokens=None):
        import torch
        if stream is None:
            stream = torch.cuda.current_stream(self.device)
        return B.msa_producer_forward(*self.args(launch_flags, num_tokens), stream=stream.cuda_stream)

    def outputs_to_host(self):
        q = self.q_out.cpu().numpy().view(np.uint16)
        iq = self.idx_q_out.cpu().numpy().view(np.uint16)
        return q, iq

    def pools_to_host(self):
        return {k: v.cpu().numpy() for k, v in self.pools.items()}


class DeviceIndexer:
    """Device copies of an indexer workload (queries, lengths, table, the index-K
    history pool) and the C-ABI call on them."""

    def __init__(self, w: wl.IndexerWorkload, device="cuda", pool=None):
        import torch
        self.w = w
        self.device = torch.device(device)
        T, H, D = w.idx_q.shape
        self.cfg = B.make_indexer_cfg(H, D, w.page_size, w.block_tokens, w.topk, w.max_blocks)
        self.idx_q = _t(w.idx_q, self.device)
        self.kv_len = _t(w.kv_len, self.device)
        self.table_offset = _t(w.table_offset, self.device)
        self.page_table = _t(w.page_table.reshape(-1), self.device)
        self.pool = _t(w.pool_fill if pool is None else pool, self.device)
        self.k_scale = torch.tensor([w.k_scale], dtype=torch.float32, device=self.device)
        self.block_scores = torch.empty((T, w.max_blocks), dtype=torch.float32, device=self.device)
        self.topk_ids = torch.empty((T, w.topk), dtype=torch.int32, device=self.device)
        self.counters = torch.zeros((T,), dtype=torch.int32, device=self.device)
        c = w.cache
        self.cache = B.make_cache(self.pool.data_ptr() + c.offset, c.dtype, c.num_pages, 1,
                                  c.stride_page, c.stride_head, c.stride_token)

    def run(self, stream=None, launch_flags=0, fused=False):
        """msa_indexer_forward, or with ``fused`` msa_indexer_forward_fused on this
        indexer's zeroed per-query counters."""
        import torch
        if stream is None:
            stream = torch.cuda.current_stream(self.device)
        p = lambda t: int(t.data_ptr())
        args = (self.cfg, self.w.idx_q.shape[0], p(self.idx_q), p(self.kv_len),
                p(self.table_offset), p(self.page_table), self.page_table.numel(), self.cache,
                p(self.k_scale), p(self.block_scores), p(self.topk_ids))
        if fused:
            return B.msa_indexer_forward_fused(*args, p(self.counters), launch_flags,
                                               stream=stream.cuda_stream)
        return B.msa_indexer_forward(*args, launch_flags, stream=stream.cuda_stream)


class DeviceProjection:
    """Device copies of a projection workload: hidden states, the packed weight and,
    through a ``DeviceWorkload`` of the producer part, everything the epilogue
    writes; ``run`` calls msa_projection_forward on them."""

    def __init__(self, pw: wl.ProjectionWorkload, device="cuda", pools_on_device: dict | None = None,
                 rows_out: bool = False):
        import torch
        self.pw = pw
        self.dw = DeviceWorkload(pw.producer, device, pools_on_device=pools_on_device)
        self.device = self.dw.device
        self.hidden = _t(pw.hidden, self.device)
        self.weight = _t(pw.weight, self.device)
        self.hidden_scales = None if pw.hidden_scales is None else _t(pw.hidden_scales, self.device)
        self.weight_scales = None if pw.weight_scales is None else _t(pw.weight_scales, self.device)
        self.rows_out = (torch.zeros((pw.num_tokens, pw.width), dtype=torch.int16, device=self.device)
                         if rows_out else None)
        self.status = torch.zeros(1, dtype=torch.int32, device=self.device)

    @property
    def pools(self):
        return self.dw.pools

    def args(self):
        """Positional arguments of msa_projection_forward minus the stream."""
        dw, pw = self.dw, self.pw
        p = lambda t: None if t is None else int(t.data_ptr())
        return (dw.cfg, pw.num_tokens, p(self.hidden), pw.hidden_size, pw.hidden.shape[1],
                p(self.weight), pw.weight.shape[1], pw.operand_dtype, p(self.hidden_scales),
                p(self.weight_scales), p(dw.positions), p(dw.slots), p(dw.page_table),
                0 if dw.page_table is None else dw.page_table.numel(),
                p(dw.weights.get("q")), p(dw.weights.get("k")), p(dw.weights.get("idx_q")),
                p(dw.weights.get("idx_k")), p(dw.q_out), p(dw.idx_q_out), dw.caches["k"],
                dw.caches["v"], dw.caches["idx_k"], p(dw.scales), p(self.rows_out),
                0 if self.rows_out is None else pw.width, p(self.status))

    def run(self, stream=None):
        import torch
        if stream is None:
            stream = torch.cuda.current_stream(self.device)
        return B.msa_projection_forward(*self.args(), stream=stream.cuda_stream)

    def outputs_to_host(self):
        return self.dw.outputs_to_host()

    def rows_to_host(self):
        return self.rows_out.cpu().numpy().view(np.uint16)


class DecodeLayer:
    """One MSA decode layer's hot path on the device: the producer (rows -> compact
    Q / index-Q, K/V/index-K into the caches) followed by the indexer on what the
    producer wrote (its compact index-Q and index-K cache), each token's visible
    history being its position + 1 tokens in its sequence's page-table row."""

    def __init__(self, dw: DeviceWorkload, max_blocks_per_seq: int, block_tokens: int = 128,
                 topk: int = 16):
        import torch
        self.dw = dw
        w = dw.w
        s = w.shape
        assert w.page_table is not None and dw.caches.get("idx_k") is not None
        P = s["page_size"]
        self.cfg = B.make_indexer_cfg(s["num_idx_q_heads"], s["head_dim"], P, block_tokens, topk,
                                      -(-max_blocks_per_seq * P // block_tokens))
        T = w.num_tokens
        pt = w.page_table.reshape(w.page_table.shape[0], -1)
        # the sequence of each token is its slot's table row (logical slots); a padded
        # token keeps the row of its position in the batch
        seq = np.where(w.slot_mapping >= 0, w.slot_mapping // (pt.shape[1] * P),
                       np.arange(T) % pt.shape[0])
        self.kv_len = _t((w.positions.astype(np.int64) + 1).astype(np.int32), dw.device)
        self.table_offset = _t((seq * pt.shape[1]).astype(np.int64), dw.device)
        self.k_scale = dw.scales[2:3] if s.get("scale_mode", 0) == 0 else dw.scales[-1:]
        self.block_scores = torch.empty((T, self.cfg.max_blocks), dtype=torch.float32,
                                        device=dw.device)
        self.topk_ids = torch.empty((T, topk), dtype=torch.int32, device=dw.device)
        self.counters = torch.zeros((T,), dtype=torch.int32, device=dw.device)

    def run(self, stream, flags=0, fused=False):
        """The producer, then the indexer on what it wrote (with ``fused``, the
        single-launch indexer on this layer's zeroed counters)."""
        dw = self.dw
        p = lambda t: int(t.data_ptr())
        dw.run(B.MSA_LAUNCH_PERSISTENT | (flags & B.MSA_LAUNCH_PDL), stream=stream)
        args = (self.cfg, dw.w.num_tokens, p(dw.idx_q_out), p(self.kv_len), p(self.table_offset),
                p(dw.page_table), dw.page_table.numel(), dw.caches["idx_k"], p(self.k_scale),
                p(self.block_scores), p(self.topk_ids))
        if fused:
            B.msa_indexer_forward_fused(*args, p(self.counters), flags & B.MSA_LAUNCH_PDL,
                                        stream=stream.cuda_stream)
        else:
            B.msa_indexer_forward(*args, flags & B.MSA_LAUNCH_PDL, stream=stream.cuda_stream)
