"""The producer over token rows that live in host memory.

Two ways are offered.  ``run`` overlaps copies with the kernel; ``run_zero_copy``
passes the pinned host buffers straight to the kernel, which then reads the rows
and writes the compact outputs across the CPU-GPU link itself (on Grace-Blackwell,
NVLink-C2C), with no staging copies at all.

Copy pipeline: tokens are independent, so a batch whose rows, positions and slots sit in pinned
host memory can be cut into chunks: while chunk k is produced on the compute
stream, chunk k+1's inputs are copied in on a copy-in stream and chunk k-1's
compact Q / index-Q are copied out on a copy-out stream.  Two device staging
slots alternate; events order the three streams.  The page table, norm weights,
scales and caches stay resident on the device.  torch supplies the device
buffers, streams and events; every producer step runs in the CUDA library.
"""
from __future__ import annotations

from . import binding as B


class HostPipeline:
    def __init__(self, cfg: B.MsaProducerCfg, row_stride: int, chunk_tokens: int, device,
                 norm_weights, caches, scales, page_table=None, launch_flags=0):
        """``norm_weights``: (q, k, idx_q, idx_k) device bf16 tensors (or None);
        ``caches``: (k, v, idx_k) MsaCacheDesc (or None); ``scales``: device fp32
        tensor or None; ``page_table``: device int32 tensor or None."""
        import torch
        self.torch = torch
        self.cfg = cfg
        self.device = torch.device(device)
        self.row_stride = int(row_stride)
        self.chunk = int(chunk_tokens)
        self.weights = norm_weights
        self.caches = caches
        self.scales = scales
        self.page_table = page_table
        self.flags = int(launch_flags)
        D = cfg.head_dim
        bf16 = torch.int16  # bf16 payloads are moved as raw 16-bit words
        self.slots = []
        for _ in range(2):
            self.slots.append(dict(
                qkv=torch.empty((self.chunk, self.row_stride), dtype=bf16, device=self.device),
                pos=torch.empty(self.chunk, dtype=torch.int32, device=self.device),
                slot=torch.empty(self.chunk, dtype=torch.int64, device=self.device),
                q=torch.empty((self.chunk, cfg.num_q_heads, D), dtype=bf16, device=self.device),
                iq=torch.empty((self.chunk, cfg.num_idx_q_heads, D), dtype=bf16, device=self.device),
                h2d=torch.cuda.Event(), comp=torch.cuda.Event(), d2h=torch.cuda.Event(),
                used=False))
        self.s_in = torch.cuda.Stream(device=self.device)
        self.s_comp = torch.cuda.Stream(device=self.device)
        self.s_out = torch.cuda.Stream(device=self.device)

    def run(self, h_qkv, h_pos, h_slots, h_q, h_iq) -> None:
        """Produces every token of the host batch.  ``h_qkv`` [T, row_stride] (16-bit
        words), ``h_pos`` int32 [T], ``h_slots`` int64 [T] are pinned host inputs;
        ``h_q`` [T, Hq, D] and ``h_iq`` [T, Hiq, D] pinned host outputs.  Returns once
        the outputs are on the host."""
        torch = self.torch
        T = h_pos.shape[0]
        p = lambda t: None if t is None else int(t.data_ptr())
        wq, wk, wiq, wik = self.weights
        kc, vc, ikc = self.caches
        pt_len = 0 if self.page_table is None else self.page_table.numel()
        for k, c0 in enumerate(range(0, T, self.chunk)):
            n = min(self.chunk, T - c0)
            st = self.slots[k % 2]
            with torch.cuda.stream(self.s_in):
                if st["used"]:
                    self.s_in.wait_event(st["comp"])      # the kernel is done reading the slot
                st["qkv"][:n].copy_(h_qkv[c0:c0 + n], non_blocking=True)
                st["pos"][:n].copy_(h_pos[c0:c0 + n], non_blocking=True)
                st["slot"][:n].copy_(h_slots[c0:c0 + n], non_blocking=True)
                st["h2d"].record(self.s_in)
            self.s_comp.wait_event(st["h2d"])
            if st["used"]:
                self.s_comp.wait_event(st["d2h"])         # last outputs of this slot copied out
            B.msa_producer_forward(self.cfg, n, p(st["qkv"]), self.row_stride, p(st["pos"]),
                                   p(st["slot"]), p(self.page_table), pt_len, p(wq), p(wk),
                                   p(wiq), p(wik), p(st["q"]), p(st["iq"]), kc, vc, ikc,
                                   p(self.scales), self.flags, self.s_comp.cuda_stream)
            st["comp"].record(self.s_comp)
            with torch.cuda.stream(self.s_out):
                self.s_out.wait_event(st["comp"])
                h_q[c0:c0 + n].copy_(st["q"][:n], non_blocking=True)
                h_iq[c0:c0 + n].copy_(st["iq"][:n], non_blocking=True)
                st["d2h"].record(self.s_out)
            st["used"] = True
        self.s_out.synchronize()

    def run_zero_copy(self, h_qkv, h_pos, h_slots, h_q, h_iq) -> None:
        """One producer launch that reads the rows, positions and slots from pinned host
        memory and writes compact Q / index-Q into pinned host memory directly (the
        caches stay on the device).  Raises if a buffer is not device-mapped host
        memory.  Returns once the outputs are on the host."""
        T = h_pos.shape[0]
        dev = []
        for name, t in (("rows", h_qkv), ("positions", h_pos), ("slots", h_slots),
                        ("q_out", h_q), ("idx_q_out", h_iq)):
            a = B.msa_host_buffer_device_address(int(t.data_ptr()))
            if a is None:
                raise ValueError(f"{name}: not pinned, device-mapped host memory")
            dev.append(a)
        p = lambda t: None if t is None else int(t.data_ptr())
        wq, wk, wiq, wik = self.weights
        kc, vc, ikc = self.caches
        pt_len = 0 if self.page_table is None else self.page_table.numel()
        B.msa_producer_forward(self.cfg, T, dev[0], self.row_stride, dev[1], dev[2],
                               p(self.page_table), pt_len, p(wq), p(wk), p(wiq), p(wik),
                               dev[3], dev[4], kc, vc, ikc, p(self.scales), self.flags,
                               self.s_comp.cuda_stream)
        self.s_comp.synchronize()
