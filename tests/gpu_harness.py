"""GPU-side comparison of the CUDA producer with the oracle (used by -m gpu tests).

For a workload, the producer runs twice on the device, on cache pools filled with
two different sentinel patterns (A and A xor 0x5A).  A byte was written by the
kernel exactly when it differs from its sentinel in either run, so the written
set is known without any tolerance; it must equal the cells the oracle's
placement gives.  Inside those cells the two runs must agree bit for bit and lie
within the stated tolerance of the oracle (fp8: one E4M3 step; bf16: 2e-2 +
1e-2*|ref|); the compact Q / index-Q outputs are compared element by element.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from harness import BF16_ATOL, BF16_RTOL, compare_bf16, e4m3_ulp_distance, run_oracle
from paged_kv_cache_msa_gb300 import workloads as wl
from paged_kv_cache_msa_gb300.device import DeviceWorkload

SENTINEL_XOR = 0x5A


def oracle_written_mask(w: wl.Workload) -> dict:
    """pool name -> bool array: bytes the oracle's placement says get written."""
    masks = {name: np.zeros(n, dtype=bool) for name, n in w.pools.items()}
    P = w.shape["page_size"]
    D = w.shape["head_dim"]
    pt = None if w.page_table is None else w.page_table.reshape(-1)
    slots = w.slot_mapping.tolist()
    for key in ("k", "v", "idx_k"):
        c = w.caches.get(key)
        if c is None:
            continue
        pages, offs = [], []
        for ls in slots:
            pl = oracle.place(ls, P, pt, c.num_pages)
            if pl is not None:
                pages.append(pl[0])
                offs.append(pl[1])
        if not pages:
            continue
        pages = np.asarray(pages, dtype=np.int64)
        offs = np.asarray(offs, dtype=np.int64)
        es = c.elem_size()
        heads = np.arange(c.num_heads, dtype=np.int64)
        e0 = (pages[:, None] * c.stride_page + heads[None, :] * c.stride_head
              + offs[:, None] * c.stride_token)                       # [n, H] elements
        start = c.offset + es * e0                                    # bytes
        row = np.arange(D * es, dtype=np.int64)
        for chunk in range(0, start.shape[0], 4096):
            cells = (start[chunk:chunk + 4096, :, None] + row[None, None, :]).reshape(-1)
            masks[c.pool][cells] = True
    return masks


def run_device(w: wl.Workload, pools_dev: dict, launch_flags: int, stream=None):
    dw = DeviceWorkload(w, pools_on_device=pools_dev)
    dw.run(launch_flags, stream=stream)
    return dw


def check_against_oracle(w: wl.Workload, launch_flags: int = 0, oracle_result=None,
                         check_outputs=True, device_run=None, check_cache_values=True):
    """Runs the CUDA producer on ``w`` and checks it against the oracle.  Returns
    the first DeviceWorkload (for further checks).  ``device_run(pools)``, when
    given, replaces the producer launch: it runs the CUDA path on the given device
    pools and returns an object with ``outputs_to_host()``."""
    if device_run is None:
        device_run = lambda pools: run_device(w, pools, launch_flags)
    host_a = wl.host_pools(w)
    if oracle_result is None:
        pools_o = {k: v.copy() for k, v in host_a.items()}
        q_o, iq_o, pools_o = run_oracle(w, pools=pools_o)
    else:
        q_o, iq_o, pools_o = oracle_result

    dev = torch.device("cuda")
    a_dev = {k: torch.from_numpy(v).to(dev) for k, v in host_a.items()}
    b_dev = {k: v ^ SENTINEL_XOR for k, v in a_dev.items()}
    run_a = {k: v.clone() for k, v in a_dev.items()}
    run_b = {k: v.clone() for k, v in b_dev.items()}
    dwa = device_run(run_a)
    dwb = device_run(run_b)
    torch.cuda.synchronize()

    if check_outputs:
        q_a, iq_a = dwa.outputs_to_host()
        q_b, iq_b = dwb.outputs_to_host()
        assert np.array_equal(q_a, q_b) and np.array_equal(iq_a, iq_b), "runs disagree on Q"
        compare_bf16(q_a, q_o, "q_out")
        compare_bf16(iq_a, iq_o, "idx_q_out")

    masks = oracle_written_mask(w)
    fp8_pools = {c.pool for c in w.caches.values() if c is not None and c.dtype == wl.DTYPE_E4M3}
    for name in w.pools:
        changed = (run_a[name] != a_dev[name]) | (run_b[name] != b_dev[name])
        m_dev = torch.from_numpy(masks[name]).to(dev)
        n_changed, n_expected = int(changed.sum()), int(masks[name].sum())
        if not torch.equal(changed, m_dev):
            extra = int((changed & ~m_dev).sum())
            missing = int((m_dev & ~changed).sum())
            raise AssertionError(f"pool {name}: written set differs from the oracle's placement "
                                 f"({n_changed} written, {n_expected} expected, {extra} stray, "
                                 f"{missing} missing)")
        got_a = run_a[name][m_dev].cpu().numpy()
        got_b = run_b[name][m_dev].cpu().numpy()
        assert np.array_equal(got_a, got_b), f"pool {name}: runs disagree"
        if not check_cache_values:
            continue
        exp = pools_o[name][masks[name]]
        if name in fp8_pools:
            d = e4m3_ulp_distance(got_a, exp)
            assert d.max(initial=0) <= 1, f"pool {name}: {int((d > 1).sum())} fp8 codes off by > 1 step"
        else:
            a16 = got_a.view(np.uint16)
            e16 = exp.view(np.uint16)
            compare_bf16(a16, e16, f"pool {name}")
    return dwa
