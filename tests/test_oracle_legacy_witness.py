"""A second witness for the oracle: the legacy unfused write path, in PyTorch CPU ops.

"[None][perf] Fuse MiniMax-M3 MSA per-layer KV-cache writes into one kernel"
("The problem") describes the path the fused producer replaces: per cache, a
division kernel (page), a remainder kernel (in-page offset), an index cast and an
index_put scatter.  This test composes that path from torch's own eager ops
(rms_norm, cos/sin, float8/bfloat16 casts, div/remainder, advanced-index
assignment into strided cache views) and checks that the oracle agrees with it:
the same bytes everywhere outside the written cells, fp8 codes within one step
and bf16 values within the stated tolerance inside them.  No GPU.
"""
import numpy as np
import pytest
import torch

from paged_kv_cache_msa_gb300 import workloads as wl
from harness import compare_bf16, e4m3_ulp_distance, run_oracle


def _rope_torch(y, pos, rd, theta, style):
    if rd == 0:
        return y
    k = torch.arange(rd // 2, dtype=torch.float64)
    inv = (1.0 / theta ** (2.0 * k / rd)).to(torch.float32)
    ang = pos.to(torch.float32)[:, None] * inv[None, :]            # [T, rd/2]
    c, s = torch.cos(ang)[:, None, :], torch.sin(ang)[:, None, :]
    y = y.clone()
    if style == wl.ROPE_NEOX:
        u, v = y[..., : rd // 2].clone(), y[..., rd // 2: rd].clone()
        y[..., : rd // 2] = u * c - v * s
        y[..., rd // 2: rd] = v * c + u * s
    else:
        u, v = y[..., 0:rd:2].clone(), y[..., 1:rd:2].clone()
        y[..., 0:rd:2] = u * c - v * s
        y[..., 1:rd:2] = v * c + u * s
    return y


def legacy_path(w: wl.Workload, pools: dict):
    s = w.shape
    D, P, rd = s["head_dim"], s["page_size"], s["rotary_dim"]
    Hq, Hkv, Hiq, Hik = s["num_q_heads"], s["num_kv_heads"], s["num_idx_q_heads"], s["num_idx_k_heads"]
    T = w.num_tokens
    x = torch.from_numpy(w.qkv.view(np.int16)).view(torch.bfloat16).float()[:, : w.width]
    bounds = np.cumsum([0, Hq, Hkv, Hkv, Hiq, Hik]) * D
    sec = {n: x[:, bounds[i]: bounds[i + 1]].reshape(T, -1, D)
           for i, n in enumerate(["q", "k", "v", "idx_q", "idx_k"])}
    wt = {k: torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).float() for k, v in w.weights.items()}
    pos = torch.from_numpy(w.positions)
    out = {}
    for n in ("q", "k", "idx_q", "idx_k"):
        y = torch.nn.functional.rms_norm(sec[n], (D,), wt[n], eps=s["rms_eps"])
        out[n] = _rope_torch(y, pos, rd, s["rope_theta"], s["rope_style"])
    out["v"] = sec["v"]
    q = out["q"].to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    iq = out["idx_q"].to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)

    slot = torch.from_numpy(w.slot_mapping)
    for key, which in (("k", 0), ("v", 1), ("idx_k", 2)):
        c = w.caches.get(key)
        if c is None:
            continue
        block = torch.div(slot, P, rounding_mode="floor")              # division kernel
        off = torch.remainder(slot, P)                                  # remainder kernel
        if w.page_table is not None:
            table = torch.from_numpy(w.page_table.reshape(-1)).long()   # index cast
            inside = (slot >= 0) & (block < table.numel())
            page = torch.where(inside, table[block.clamp(0, table.numel() - 1)], torch.full_like(block, -1))
        else:
            inside = slot >= 0
            page = block
        ok = inside & (page >= 0) & (page < c.num_pages)
        vals = out[key][ok]
        pool = torch.from_numpy(pools[c.pool])
        if c.dtype == wl.DTYPE_E4M3:
            enc = (vals * (1.0 / float(np.float32(w.scales[which])))).clamp(-448, 448)
            enc = enc.to(torch.float8_e4m3fn).view(torch.uint8)
            base = pool[c.offset:]
        else:
            enc = vals.to(torch.bfloat16).view(torch.int16)
            base = pool[c.offset:].view(torch.int16)
        view = torch.as_strided(base, (c.num_pages, c.num_heads, P, D),
                                (c.stride_page, c.stride_head, c.stride_token, 1))
        view[page[ok], :, off[ok], :] = enc                              # index_put scatter
    return q, iq


def _mixed_small(seed):
    """A small batch with padding, a page table with holes and strided caches."""
    rng = np.random.default_rng(seed)
    seq_positions = [[int(p)] for p in rng.integers(0, 256, size=6)] + [list(range(64, 100))]
    w = wl.make_batch("witness", seed, wl.BIG, seq_positions, max_blocks=4, num_pages=40,
                      rotary_dim=64, page_pad_bytes=256, row_pad=64, pad_frac=0.1)
    pt = np.array(w.page_table, copy=True)
    pt[0, :] = -1
    w.page_table = pt
    return w


@pytest.mark.parametrize("make", [wl.config1_tiny_decode, lambda: _mixed_small(77)],
                         ids=["config1_tiny_decode", "mixed_small"])
def test_oracle_matches_legacy_path(make):
    w = make()
    q_o, iq_o, pools_o = run_oracle(w)
    pools_l = wl.host_pools(w)
    q_l, iq_l = legacy_path(w, pools_l)
    compare_bf16(q_o, q_l, "q")
    compare_bf16(iq_o, iq_l, "idx_q")
    for name in pools_o:
        a, b = pools_o[name], pools_l[name]
        diff = np.nonzero(a != b)[0]
        if diff.size == 0:
            continue
        fp8_pools = {c.pool for c in w.caches.values() if c is not None and c.dtype == wl.DTYPE_E4M3}
        if name in fp8_pools:
            assert e4m3_ulp_distance(a[diff], b[diff]).max() <= 1
        else:
            # bf16 elements start at even byte offsets in these pools
            idx = np.unique(diff - diff % 2)
            av = np.frombuffer(a.tobytes(), dtype=np.uint16)[idx // 2]
            bv = np.frombuffer(b.tobytes(), dtype=np.uint16)[idx // 2]
            compare_bf16(av, bv, name)
