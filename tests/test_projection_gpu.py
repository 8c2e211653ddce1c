"""The projection GEMM with the producer in its epilogue, against the oracle (GPU).

The oracle side is the plain composition the fused kernel must equal: the
projection rows of the oracle (exact dot products rounded to fp32, then bf16),
then the producer oracle on those rows.  The CUDA side is one call of
msa_projection_forward.

Tolerance.  The kernel's bf16 rows are within one bf16 step plus the error of an
fp32 accumulation of the exact products, and almost all of them identical to the
oracle's.  A row element that differs by one bf16 step can move a cache value by
more than one E4M3 step where RoPE cancels (u cos - v sin near zero), so the
producer's own tolerances (bf16: 2e-2 + 1e-2*|ref|; fp8: one E4M3 step) are
widened, element by element, by the change the row bound can cause through the
norm factor, the weight and the RoPE partner; at least 99% of all values must meet
the unwidened tolerance.  The written cache bytes are checked exactly (two
sentinel runs).

The epilogue's own producer arithmetic is pinned separately and strictly: the
oracle producer run on the bf16 rows the kernel itself wrote (rows_out, the values
the epilogue normalises, rotates and encodes) must match every compact Q / index-Q
value within 2e-2 + 1e-2*|ref| and every fp8 code within one E4M3 step, with no
widening and no allowance (``check_epilogue_strict``).
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_harness import SENTINEL_XOR, check_against_oracle, oracle_written_mask
from harness import BF16_ATOL, BF16_RTOL, cache_cells, compare_bf16, e4m3_ulp_distance, run_oracle
from paged_kv_cache_msa_gb300 import binding as B
from paged_kv_cache_msa_gb300 import workloads as wl
from paged_kv_cache_msa_gb300.device import DeviceProjection

pytestmark = pytest.mark.gpu


def _bf16_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _operands_f64(a: np.ndarray) -> np.ndarray:
    """bf16 bits or E4M3 codes -> float64 (E4M3 through torch's float8 type)."""
    if a.dtype == np.uint16:
        return _bf16_f64(a)
    t = torch.from_numpy(np.ascontiguousarray(a)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def _exact_and_acc(pw: wl.ProjectionWorkload, idx):
    """Exact scaled dot products and the fp32-accumulation error bound of the
    kernel's value, K * 2^-24 * sum_k |x_k w_k| * |sx sw| plus the rounding of its
    two scale multiplications (2^-23 of the value)."""
    K = pw.hidden_size
    x = _operands_f64(pw.hidden[idx, :K])
    w = _operands_f64(pw.weight[:, :K])
    sx = np.ones(x.shape[0]) if pw.hidden_scales is None else pw.hidden_scales[idx].astype(np.float64)
    sw = np.ones(w.shape[0]) if pw.weight_scales is None else pw.weight_scales.astype(np.float64)
    s = sx[:, None] * sw[None, :]
    exact = (x @ w.T) * s
    acc = K * 2.0**-24 * (np.abs(x) @ np.abs(w).T) * np.abs(s) + 2.0**-23 * np.abs(exact)
    return exact, acc


def check_rows(got: np.ndarray, pw: wl.ProjectionWorkload, rows, idx=None):
    """The kernel's bf16 rows (of the tokens ``idx``, all by default) against the
    exact scaled dot products (float64 library matmul of the decoded operands):
    every one within the error of an fp32 accumulation of K products,
    K * 2^-24 * sum_k |x_k w_k|, plus one bf16 step of the exact value; and, when
    the oracle's rows are given, at least 99% identical to them."""
    idx = np.arange(pw.num_tokens) if idx is None else idx
    exact, acc = _exact_and_acc(pw, idx)
    a = np.abs(exact)
    step = np.where(a > 0, np.exp2(np.floor(np.log2(np.maximum(a, 1e-300))) - 7), 0.0)
    bound = step + acc
    err = np.abs(_bf16_f64(got) - exact)
    bad = err > bound
    assert not bad.any(), (f"projection rows: {int(bad.sum())} beyond the fp32 accumulation bound; "
                           f"first at {np.argwhere(bad)[:3].tolist()}")
    if rows is not None:
        assert (got == rows).mean() > 0.99, "projection rows: more than 1% not exactly rounded"


def oracle_rows(pw: wl.ProjectionWorkload, idx=None) -> np.ndarray:
    h = pw.hidden[:, :pw.hidden_size]
    sx = pw.hidden_scales
    if idx is not None:
        h = np.ascontiguousarray(h[idx])
        sx = None if sx is None else sx[idx]
    return oracle.projection(h, pw.weight[:, :pw.hidden_size], sx, pw.weight_scales)


def row_error_bound(pw: wl.ProjectionWorkload, idx) -> np.ndarray:
    """For the tokens ``idx`` and every projection output: how far the kernel's bf16
    row may lie from the oracle's.  The kernel rounds an fp32 sum that is within
    acc = K * 2^-24 * sum_k |x_k w_k| of the exact one, the oracle the exact sum
    itself (through fp32), so the two bf16 values are at most one bf16 step (at the
    larger magnitude) plus acc apart."""
    exact, acc = _exact_and_acc(pw, idx)
    a = np.abs(exact) + acc
    step = np.where(a > 0, np.exp2(np.floor(np.log2(np.maximum(a, 1e-300))) - 7), 2.0**-133)
    return step + acc


def value_bounds(pw: wl.ProjectionWorkload, rows: np.ndarray, e: np.ndarray) -> np.ndarray:
    """[n, heads, D]: the largest change of each value the producer encodes (after
    norm and RoPE, before the cache scale) that rows within ``e`` of the oracle's
    ``rows`` can cause, to first order: the change of the element itself times the
    norm factor and weight, the change of the norm factor, and the change of the
    RoPE partner (|cos|, |sin| <= 1); V values change by e itself."""
    s = pw.producer.shape
    D, rd, eps = s["head_dim"], s["rotary_dim"], s["rms_eps"]
    hq, hkv, hiq = s["num_q_heads"], s["num_kv_heads"], s["num_idx_q_heads"]
    H = pw.width // D
    R = _bf16_f64(rows)
    wts = {k: (np.ones(D) if v is None else _bf16_f64(v)) for k, v in pw.producer.weights.items()}
    partner = np.arange(D)
    rot = np.zeros(D, dtype=bool)
    rot[:rd] = True
    if s["rope_style"] == wl.ROPE_NEOX:
        half = rd // 2
        partner[:half] += half
        partner[half:rd] -= half
    else:
        partner[:rd] ^= 1
    out = np.empty((R.shape[0], H, D))
    for g in range(H):
        x = R[:, g * D:(g + 1) * D]
        eh = e[:, g * D:(g + 1) * D]
        if hq + hkv <= g < hq + 2 * hkv:      # V
            out[:, g] = eh
            continue
        key = ("q" if g < hq else "k" if g < hq + hkv else "idx_q" if g < hq + 2 * hkv + hiq
               else "idx_k")
        wv = np.abs(wts[key])
        ms = (x * x).mean(1) + eps
        r = 1.0 / np.sqrt(ms)
        drel = (np.abs(x) * eh).sum(1) / (D * ms)
        d = r[:, None] * wv * eh + np.abs(x) * r[:, None] * wv * drel[:, None]
        out[:, g] = d + np.where(rot, d[:, partner], 0.0)
    return out * 1.05 + 1e-7


_E4M3 = None


def e4m3_values(codes: np.ndarray) -> np.ndarray:
    global _E4M3
    if _E4M3 is None:
        _E4M3 = np.array([oracle.e4m3_decode(c) for c in range(256)], dtype=np.float64)
    return _E4M3[codes]


def e4m3_step(v: np.ndarray) -> np.ndarray:
    a = np.abs(v)
    return np.where(a < 2.0**-6, 2.0**-9, np.exp2(np.floor(np.log2(np.maximum(a, 2.0**-6))) - 3))


def check_values(pw, idx, rows, q_o, iq_o, pools_o, dp):
    """Every output of the tokens ``idx`` (the oracle's outputs are for exactly these
    tokens, in this order) against the oracle, within the producer's tolerance
    widened by the propagated row bound; at least 99% within the strict one."""
    s = pw.producer.shape
    D, hq, hkv, hiq = s["head_dim"], s["num_q_heads"], s["num_kv_heads"], s["num_idx_q_heads"]
    bound = value_bounds(pw, rows, row_error_bound(pw, idx))
    q_d, iq_d = dp.outputs_to_host()
    strict_ok, total = 0, 0
    for name, got, exp, b in (("q_out", q_d[idx], q_o, bound[:, :hq]),
                              ("idx_q_out", iq_d[idx], iq_o,
                               bound[:, hq + 2 * hkv:hq + 2 * hkv + hiq])):
        a, ev = _bf16_f64(got), _bf16_f64(exp)
        tol = BF16_ATOL + BF16_RTOL * np.abs(ev)
        assert (np.abs(a - ev) <= tol + b).all(), f"{name}: beyond the propagated bound"
        strict_ok += int((np.abs(a - ev) <= tol).sum())
        total += a.size
    w_p = pw.producer
    P = s["page_size"]
    pt = None if w_p.page_table is None else w_p.page_table.reshape(-1)
    slots = w_p.slot_mapping[idx]
    first = {"k": hq, "v": hq + hkv, "idx_k": hq + 2 * hkv + hiq}
    scale_idx = {"k": 0, "v": 1, "idx_k": 2}
    for key in ("k", "v", "idx_k"):
        c = w_p.caches.get(key)
        if c is None or c.num_heads == 0:
            continue
        pl = [oracle.place(int(ls), P, pt, c.num_pages) for ls in slots]
        take = np.array([p is not None for p in pl])
        if not take.any():
            continue
        cells = cache_cells(w_p, key, pl)                      # [n_valid, H, D*es]
        b = bound[take][:, first[key]:first[key] + c.num_heads]
        got = dp.pools[c.pool].cpu().numpy()[cells]
        exp = pools_o[c.pool][cells]
        if c.dtype == wl.DTYPE_E4M3:
            if s.get("scale_mode", 0) == 1:
                base = {"k": 0, "v": hkv, "idx_k": 2 * hkv}[key]
                sc = w_p.scales[base:base + c.num_heads].astype(np.float64)[None, :, None]
            else:
                sc = float(w_p.scales[scale_idx[key]])
            ga, ea = e4m3_values(got), e4m3_values(exp)
            step = np.maximum(e4m3_step(ga), e4m3_step(ea))
            ok = np.abs(ga - ea) <= step + b / sc
            assert ok.all(), f"{key}: {int((~ok).sum())} fp8 codes beyond the propagated bound"
            d = e4m3_ulp_distance(got.reshape(-1), exp.reshape(-1))
            strict_ok += int((d <= 1).sum())
            total += d.size
        else:
            a = _bf16_f64(got.reshape(-1).view(np.uint16)).reshape(b.shape)
            ev = _bf16_f64(exp.reshape(-1).view(np.uint16)).reshape(b.shape)
            tol = BF16_ATOL + BF16_RTOL * np.abs(ev)
            assert (np.abs(a - ev) <= tol + b).all(), f"{key}: beyond the propagated bound"
            strict_ok += int((np.abs(a - ev) <= tol).sum())
            total += a.size
    assert strict_ok >= 0.99 * total, f"only {strict_ok} of {total} within the producer's tolerance"


def _sub_workload(w_p: wl.Workload, idx, rows: np.ndarray, tag: str) -> wl.Workload:
    """The producer workload restricted to the tokens ``idx`` with the given rows."""
    meta = dict(w_p.meta)
    if "valid_mask" in meta:
        meta["valid_mask"] = meta["valid_mask"][idx]
    return wl.Workload(w_p.name + tag, w_p.shape, np.ascontiguousarray(rows), rows.shape[1],
                       w_p.positions[idx].copy(), w_p.slot_mapping[idx].copy(), w_p.page_table,
                       w_p.weights, w_p.scales, w_p.caches, w_p.pools, w_p.seed, meta)


def check_epilogue_strict(pw: wl.ProjectionWorkload, dp: DeviceProjection, idx=None):
    """The epilogue's producer arithmetic alone, at the producer's own tolerance.

    ``dp`` ran on cache pools filled with the workload's sentinel pattern A and wrote
    its bf16 rows (rows_out).  The oracle producer runs on exactly those rows for the
    tokens ``idx`` (all by default); every compact Q / index-Q value of those tokens
    must lie within 2e-2 + 1e-2*|ref|, every fp8 cache code within one E4M3 step and
    every bf16 cache value within the Q tolerance -- no widening, no allowance."""
    w_p = pw.producer
    T = pw.num_tokens
    idx = np.arange(T) if idx is None else np.asarray(idx, dtype=np.int64)
    dev = dp.device
    it = torch.from_numpy(idx).to(dev)
    rows_k = dp.rows_out.index_select(0, it).cpu().numpy().view(np.uint16)
    sub = _sub_workload(w_p, idx, rows_k, "[kernel rows]")
    q_o, iq_o, pools_o = run_oracle(sub, pools=wl.host_pools(w_p))
    q_d = dp.dw.q_out.index_select(0, it).cpu().numpy().view(np.uint16)
    iq_d = dp.dw.idx_q_out.index_select(0, it).cpu().numpy().view(np.uint16)
    compare_bf16(q_d, q_o, "q_out from the kernel's rows")
    compare_bf16(iq_d, iq_o, "idx_q_out from the kernel's rows")
    P = w_p.shape["page_size"]
    pt = None if w_p.page_table is None else w_p.page_table.reshape(-1)
    for key in ("k", "v", "idx_k"):
        c = w_p.caches.get(key)
        if c is None or c.num_heads == 0:
            continue
        pl = [oracle.place(int(ls), P, pt, c.num_pages) for ls in sub.slot_mapping]
        if not any(x is not None for x in pl):
            continue
        cells = cache_cells(w_p, key, pl).reshape(-1)
        got = dp.pools[c.pool].index_select(0, torch.from_numpy(cells).to(dev)).cpu().numpy()
        exp = pools_o[c.pool][cells]
        if c.dtype == wl.DTYPE_E4M3:
            d = e4m3_ulp_distance(got, exp)
            assert d.max(initial=0) <= 1, (f"{key} cache from the kernel's rows: "
                                           f"{int((d > 1).sum())} codes more than one E4M3 step off")
        else:
            compare_bf16(got.view(np.uint16), exp.view(np.uint16), f"{key} cache from the kernel's rows")


def tile_samples(T: int, seed: int, tile: int = 128) -> np.ndarray:
    """At least one token of every ``tile``-token tile (a random one), plus the first
    and last two tokens of the batch and of the first and last tiles."""
    rng = np.random.default_rng(seed)
    starts = np.arange(0, T, tile)
    pick = starts + rng.integers(0, tile, size=starts.shape[0])
    edges = [0, 1, tile - 1, tile, tile + 1, T - tile - 1, T - tile, T - 2, T - 1]
    return np.unique(np.clip(np.concatenate([pick, edges]), 0, T - 1))


def check_projection(pw: wl.ProjectionWorkload):
    rows = oracle_rows(pw)
    w_rows = pw.with_rows(rows)
    q_o, iq_o, pools_o = run_oracle(w_rows)
    statuses = []

    def device_run(pools):
        dp = DeviceProjection(pw, pools_on_device=pools, rows_out=True)
        dp.run()
        torch.cuda.synchronize()
        statuses.append(int(dp.status.item()))
        check_rows(dp.rows_to_host(), pw, rows)
        return dp

    # written set (exact) and agreement of the two sentinel runs
    dp = check_against_oracle(w_rows, oracle_result=(q_o, iq_o, pools_o), check_outputs=False,
                              device_run=device_run, check_cache_values=False)
    assert statuses == [0, 0]
    check_values(pw, np.arange(pw.num_tokens), rows, q_o, iq_o, pools_o, dp)
    check_epilogue_strict(pw, dp)


def _batch(seed, heads, T, hidden, **kw):
    mult = 16 if kw.get("operand_dtype") == wl.DTYPE_E4M3 else 8   # 16-byte row strides
    kw["hidden_pad"] = kw.get("hidden_pad", 0) + (-(hidden + kw.get("hidden_pad", 0))) % mult
    kw["weight_pad"] = kw.get("weight_pad", 0) + (-(hidden + kw.get("weight_pad", 0))) % mult
    rng = np.random.default_rng(seed)
    P = kw.get("page_size", 64)
    max_blocks = -(-(T + 64) // P)
    start = int(rng.integers(0, 64))
    seq_positions = [list(range(start, start + T))]
    kw.setdefault("num_pages", max_blocks + 3)
    return wl.make_projection_batch(f"proj{seed}", seed, heads, seq_positions, hidden,
                                    max_blocks=max_blocks, **kw)


OPERANDS = [wl.DTYPE_BF16, wl.DTYPE_E4M3]
OPERAND_IDS = ["bf16", "e4m3"]


@pytest.mark.parametrize("dt", OPERANDS, ids=OPERAND_IDS)
@pytest.mark.parametrize("T,hidden", [(1, 64), (127, 128), (300, 200), (513, 72), (40, 330)])
def test_tiny_shapes_ragged_tiles(T, hidden, dt):
    """Tiny shapes (15 heads of 64: 4 output tiles, the last one partly past the
    row), token counts and hidden sizes that leave ragged tiles (in tokens, outputs
    and K), NaN-padded row strides."""
    pw = _batch(10 + T, wl.TINY, T, hidden, hidden_pad=16, weight_pad=16, pad_frac=0.1,
                idx_k_dtype=wl.DTYPE_BF16, operand_dtype=dt)
    check_projection(pw)


@pytest.mark.parametrize("dt", OPERANDS, ids=OPERAND_IDS)
@pytest.mark.parametrize("T,hidden", [(64, 512), (200, 256), (257, 384)])
def test_big_shapes(T, hidden, dt):
    pw = _batch(20 + T, wl.BIG, T, hidden, pad_frac=0.1, page_pad_bytes=256, operand_dtype=dt)
    check_projection(pw)


@pytest.mark.parametrize("style,rd,D", [(wl.ROPE_NEOX, 32, 64), (wl.ROPE_GPTJ, 64, 64),
                                        (wl.ROPE_GPTJ, 40, 128), (wl.ROPE_NEOX, 0, 128),
                                        (wl.ROPE_NEOX, 96, 128)])
def test_rope_variants(style, rd, D):
    heads = wl.TINY if D == 64 else dict(wl.BIG, num_q_heads=6)
    pw = _batch(30 + rd + D, heads, 150, 192, rotary_dim=rd, rope_style=style)
    check_projection(pw)


def test_bf16_caches_per_head_scales_physical_slots():
    pw = _batch(41, dict(wl.BIG, num_q_heads=5), 140, 128, kv_dtype=wl.DTYPE_BF16,
                idx_k_dtype=wl.DTYPE_BF16, use_page_table=False)
    check_projection(pw)
    pw = _batch(42, wl.TINY, 140, 128, scale_mode=1, pad_frac=0.2)
    check_projection(pw)


def test_no_index_k_cache_and_odd_sections():
    heads = dict(num_q_heads=3, num_kv_heads=1, num_idx_q_heads=0, num_idx_k_heads=2, head_dim=128)
    pw = _batch(43, heads, 70, 136, with_idx_k=False)
    check_projection(pw)


@pytest.mark.parametrize("dt", OPERANDS, ids=OPERAND_IDS)
@pytest.mark.parametrize("T,hidden", [(1, 330), (33, 192), (96, 448), (128, 600), (128, 2100)])
def test_small_batches_split_over_k(T, hidden, dt):
    """At most 128 tokens with NeoX RoPE: the K blocks are shared out over a cluster
    of 2 to 8 CTAs whose partial sums one CTA adds up.  The hidden sizes give clusters
    of every size from 2 to 8 (bf16: ceil(K/64) blocks; E4M3: ceil(K/128)), with a
    ragged last block, and big heads in every output tile."""
    pw = _batch(50 + T + hidden, dict(wl.BIG, num_q_heads=6), T, hidden, pad_frac=0.1,
                hidden_pad=16, weight_pad=16, operand_dtype=dt)
    check_projection(pw)


@pytest.mark.parametrize("T", [40, 200])
def test_large_positions(T):
    """Positions in [2^16, 2^24): RoPE angles past 2^16 take the full-range sine and
    cosine instead of the 2pi reduction.  40 tokens run the split-over-K kernel
    (whose table is filled during the main loop), 200 the 2-SM kernel."""
    pw = _batch(60 + T, dict(wl.BIG, num_q_heads=6), T, 384)
    rng = np.random.default_rng(T)
    # positions only enter RoPE; the slots were fixed when the batch was built
    pw.producer.positions[:] = rng.integers(1 << 16, 1 << 24, size=T).astype(np.int32)
    check_projection(pw)


@pytest.mark.parametrize("dt", OPERANDS, ids=OPERAND_IDS)
def test_decode_batch_64_hidden_6144(dt):
    """The decode batch (64 tokens, big shapes, hidden 6,144): every output."""
    check_projection(wl.projection_decode(operand_dtype=dt))


def test_zero_tokens_launches_nothing():
    pw = _batch(44, wl.TINY, 5, 64)
    dp = DeviceProjection(pw)
    before = {k: v.clone() for k, v in dp.pools.items()}
    args = list(dp.args())
    args[1] = 0
    assert B.msa_projection_forward(*args, stream=torch.cuda.current_stream().cuda_stream) == B.MSA_OK
    torch.cuda.synchronize()
    for k in before:
        assert torch.equal(before[k], dp.pools[k])


def test_graph_replay_matches_direct_launch():
    pw = _batch(45, wl.BIG, 300, 256)
    direct = DeviceProjection(pw, rows_out=True)
    direct.run()
    torch.cuda.synchronize()
    dp = DeviceProjection(pw, rows_out=True)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        B.msa_projection_forward(*dp.args(), stream=s.cuda_stream)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(direct.rows_out, dp.rows_out)
    assert torch.equal(direct.dw.q_out, dp.dw.q_out)
    for k in direct.pools:
        assert torch.equal(direct.pools[k], dp.pools[k])
    assert int(dp.status.item()) == 0


@pytest.mark.parametrize("dt", OPERANDS, ids=OPERAND_IDS)
def test_prefill_65536_tokens_hidden_6144_sampled(dt):
    """The full-size prefill (65,536 tokens, hidden 6,144, 11,392 outputs): the
    written cache bytes exactly against the oracle's placement of every token
    (two sentinel runs), and sampled tokens -- a random one from every 128-token
    tile, the first and last tokens and tile edges -- element by element against
    the oracle, end to end and (on the kernel's own rows) strictly."""
    pw = wl.projection_prefill(operand_dtype=dt)
    T = pw.num_tokens
    rng = np.random.default_rng(77)
    # end to end through the oracle's own rows (about 2 s of oracle work per token)
    idx = np.unique(np.concatenate([[0, 1, 127, 128, 129, 255, 256, T - 129, T - 128, T - 1],
                                    rng.integers(0, T, size=22)]))
    # one token of every 128-token tile: rows against the exact products, epilogue strictly
    idx_tiles = tile_samples(T, 78)
    w_p = pw.producer
    host_a = wl.host_pools(w_p)
    dev = torch.device("cuda")
    a_dev = {k: torch.from_numpy(v).to(dev) for k, v in host_a.items()}
    runs = []
    for xor in (0, SENTINEL_XOR):
        pools = {k: (v ^ xor) for k, v in a_dev.items()}
        start = {k: v.clone() for k, v in pools.items()}
        dp = DeviceProjection(pw, pools_on_device=pools, rows_out=xor == 0)
        dp.run()
        torch.cuda.synchronize()
        assert int(dp.status.item()) == 0
        runs.append((dp, start))
    masks = oracle_written_mask(w_p)
    for name in w_p.pools:
        changed = torch.zeros_like(a_dev[name], dtype=torch.bool)
        for dp, start in runs:
            changed |= dp.pools[name] != start[name]
        assert torch.equal(changed, torch.from_numpy(masks[name]).to(dev)), f"pool {name}: written set"

    # sampled tokens against the oracle
    rows = oracle_rows(pw, idx)
    sub = wl.Workload(w_p.name + "[sample]", w_p.shape, rows, rows.shape[1], w_p.positions[idx].copy(),
                      w_p.slot_mapping[idx].copy(), w_p.page_table, w_p.weights, w_p.scales,
                      w_p.caches, w_p.pools, w_p.seed,
                      dict(w_p.meta, valid_mask=w_p.meta["valid_mask"][idx]))
    q_o, iq_o, pools_o = run_oracle(sub, pools=wl.host_pools(w_p))
    check_values(pw, idx, rows, q_o, iq_o, pools_o, runs[0][0])
    # every tile: the kernel's rows within the fp32 accumulation bound of the exact
    # products, and the epilogue alone, strictly, on the rows the kernel wrote (run A)
    dp_a = runs[0][0]
    it = torch.from_numpy(idx_tiles).to(dp_a.device)
    check_rows(dp_a.rows_out.index_select(0, it).cpu().numpy().view(np.uint16), pw, None, idx_tiles)
    check_epilogue_strict(pw, dp_a, idx_tiles)
