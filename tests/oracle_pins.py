"""Pins for the oracle: checks against things other than the oracle itself.

Each pin is a plain function that raises AssertionError on failure.  The test
modules call every pin against the oracle build (``test_oracle_pins.py``) and
against builds with a planted mistake (``test_oracle_mutants.py``), where at
least one pin must fail.

What pins what:
  * number formats: hand-worked golden points (tests/golden), torch's own
    float8_e4m3fn / bfloat16 casts, exhaustive code round trips and the
    ties-to-even midpoints of every adjacent code pair;
  * RMSNorm: torch.nn.functional.rms_norm in float64, exact invariance under
    power-of-two scaling, unit RMS with unit weight;
  * RoPE: identity at position 0, pair norms preserved, the relative-position
    property of q.k, and the textbook complex-rotation form in float64;
  * placement: hand-worked golden points and brute force (search, no division)
    over tiny pools;
  * the whole producer: Q / index-Q / K / index-K against a float64 textbook
    composition, V against torch's fp8 cast, and the exact set of written bytes
    (sentinels, page padding and guard bands unchanged).
"""
from __future__ import annotations

import math
import os

import numpy as np
import torch

import oracle
from paged_kv_cache_msa_gb300 import workloads as wl
from harness import (bf16_bits_to_f32, cache_cells, e4m3_ulp_distance, run_oracle)

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append(line.split())
    return rows


def _torch_e4m3(x: np.ndarray) -> np.ndarray:
    """torch's float8_e4m3fn cast (round to nearest even) after clamping to the
    largest finite magnitude, i.e. saturating."""
    t = torch.from_numpy(np.asarray(x, dtype=np.float32)).clamp(-448.0, 448.0)
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _torch_bf16(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.asarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------------------
# number formats
# ---------------------------------------------------------------------------

def pin_e4m3_golden():
    for v, code, *_ in _read_golden("e4m3_points.txt"):
        got = oracle.e4m3_encode(float(v))
        assert got == int(code, 16), f"e4m3({v}) = {got:#04x}, expected {code}"


def pin_e4m3_decode_vs_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    got = np.array([oracle.e4m3_decode(int(c)) for c in codes], dtype=np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def pin_e4m3_roundtrip_and_ties():
    finite = [c for c in range(256) if (c & 0x7F) != 0x7F]
    for c in finite:
        v = oracle.e4m3_decode(c)
        assert oracle.e4m3_encode(v) == c, f"round trip of {c:#04x}"
    # every adjacent pair of positive finite codes: the midpoint goes to the even
    # code; one float step either side of it goes to the nearer code
    for c in range(0, 0x7E):
        lo, hi = oracle.e4m3_decode(c), oracle.e4m3_decode(c + 1)
        mid = np.float32((np.float64(lo) + np.float64(hi)) / 2)
        assert float(mid) == (lo + hi) / 2
        even = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_encode(float(mid)) == even, f"tie between {c:#04x} and {c + 1:#04x}"
        assert oracle.e4m3_encode(float(np.nextafter(mid, np.float32(-1)))) == c
        assert oracle.e4m3_encode(float(np.nextafter(mid, np.float32(1e9)))) == c + 1
        assert oracle.e4m3_encode(-float(mid)) == 0x80 | even


def pin_e4m3_saturation():
    for v in (448.0, 448.5, 463.99, 464.0, 465.0, 480.0, 1e4, 3e38, math.inf):
        assert oracle.e4m3_encode(v) == 0x7E, v
        assert oracle.e4m3_encode(-v) == 0xFE, -v
    assert oracle.e4m3_encode(math.nan) & 0x7F == 0x7F


def pin_e4m3_vs_torch_random():
    rng = np.random.default_rng(7)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * 30,
        (rng.standard_normal(20000) * 1e-2).astype(np.float32),
        rng.uniform(-448, 448, 20000).astype(np.float32),
        rng.uniform(-2000, 2000, 5000).astype(np.float32),
    ])
    ref = _torch_e4m3(x)
    got = np.array([oracle.e4m3_encode(float(v)) for v in x], dtype=np.uint8)
    assert np.array_equal(got, ref), np.argwhere(got != ref)[:5]


def pin_bf16_golden():
    for v, code, *_ in _read_golden("bf16_points.txt"):
        got = oracle.bf16_encode(float(v))
        assert got == int(code, 16), f"bf16({v}) = {got:#06x}, expected {code}"


def pin_bf16_vs_torch():
    rng = np.random.default_rng(11)
    bits = rng.integers(0, 2**32, size=60000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    # exact ties: low 16 bits 0x8000
    ties = ((rng.integers(0, 2**16, 4000, dtype=np.uint32) << 16) | 0x8000).view(np.float32)
    x = np.concatenate([x, ties[np.isfinite(ties)]])
    ref = _torch_bf16(x)
    got = np.array([oracle.bf16_encode(float(v)) for v in x], dtype=np.uint16)
    assert np.array_equal(got, ref), np.argwhere(got != ref)[:5]
    for h in (0x3F80, 0xC000, 0x0001, 0x7F7F, 0x8000):
        assert oracle.bf16_decode(h) == float(bf16_bits_to_f32(np.array([h]))[0])


# ---------------------------------------------------------------------------
# RMSNorm
# ---------------------------------------------------------------------------

def pin_rmsnorm_vs_torch():
    rng = np.random.default_rng(3)
    for D in (64, 128):
        for scale in (1.0, 20.0, 1e-3):
            x = (rng.standard_normal(D) * scale).astype(np.float32)
            w = rng.uniform(0.5, 1.5, D).astype(np.float32)
            got = oracle.rmsnorm(x, w, eps=1e-6)
            ref = torch.nn.functional.rms_norm(torch.from_numpy(x).double(), (D,),
                                               torch.from_numpy(w).double(), eps=1e-6).numpy()
            assert np.allclose(got, ref, rtol=2e-6, atol=1e-7), (D, scale, np.abs(got - ref).max())


def pin_rmsnorm_unit_rms_and_scaling():
    rng = np.random.default_rng(4)
    for D in (64, 128):
        x = rng.standard_normal(D).astype(np.float32)
        y = oracle.rmsnorm(x, None, eps=1e-6).astype(np.float64)
        assert abs(math.sqrt(np.mean(y * y)) - 1.0) < 1e-5
        # with eps = 0 the norm is exactly invariant under power-of-two scaling
        y0 = oracle.rmsnorm(x, None, eps=0.0)
        y1 = oracle.rmsnorm(x * np.float32(8.0), None, eps=0.0)
        assert np.array_equal(y0, y1)


# ---------------------------------------------------------------------------
# RoPE
# ---------------------------------------------------------------------------

def _textbook_rope(y, rd, pos, theta, style):
    """Rotary embedding as a complex rotation of dim pairs, in float64."""
    y = np.array(y, dtype=np.float64)
    if rd == 0:
        return y
    k = np.arange(rd // 2)
    ang = pos * theta ** (-2.0 * k / rd)
    if style == oracle.ROPE_NEOX:
        iu, iv = k, k + rd // 2
    else:
        iu, iv = 2 * k, 2 * k + 1
    z = (y[iu] + 1j * y[iv]) * np.exp(1j * ang)
    y[iu], y[iv] = z.real, z.imag
    return y


def pin_rope_identity_and_passthrough():
    rng = np.random.default_rng(5)
    for style in (oracle.ROPE_NEOX, oracle.ROPE_GPTJ):
        for D, rd in ((64, 64), (128, 128), (128, 64), (128, 32)):
            x = rng.standard_normal(D).astype(np.float32)
            assert np.array_equal(oracle.rope(x, rd, 0, style=style), x)
            y = oracle.rope(x, rd, 777, style=style)
            assert np.array_equal(y[rd:], x[rd:])


def pin_rope_textbook():
    rng = np.random.default_rng(6)
    for style in (oracle.ROPE_NEOX, oracle.ROPE_GPTJ):
        for D, rd in ((64, 64), (128, 128), (128, 64)):
            for pos in (1, 2, 17, 511, 4097, 9215):
                x = rng.standard_normal(D).astype(np.float32)
                got = oracle.rope(x, rd, pos, theta=1e4, style=style)
                ref = _textbook_rope(x, rd, pos, 1e4, style)
                # the angle is a float32 product (relative error 2^-24), so large
                # positions carry up to pos * 6e-8 rad of angle error
                tol = 2e-6 + pos * 1.2e-7 * 4
                assert np.abs(got - ref).max() < tol, (style, D, rd, pos, np.abs(got - ref).max())


def pin_rope_norms_and_relative_position():
    rng = np.random.default_rng(8)
    for style in (oracle.ROPE_NEOX, oracle.ROPE_GPTJ):
        D = rd = 128
        q = rng.standard_normal(D).astype(np.float32)
        k = rng.standard_normal(D).astype(np.float32)
        qr = oracle.rope(q, rd, 300, style=style).astype(np.float64)
        half = rd // 2
        if style == oracle.ROPE_NEOX:
            pairs = [(i, i + half) for i in range(half)]
        else:
            pairs = [(2 * i, 2 * i + 1) for i in range(half)]
        q64 = q.astype(np.float64)
        for a, b in pairs:
            n0 = math.hypot(q64[a], q64[b])
            n1 = math.hypot(qr[a], qr[b])
            assert abs(n0 - n1) <= 1e-6 * max(1.0, n0)
        for m, n in ((5, 3), (100, 40), (260, 7)):
            d0 = float(np.dot(oracle.rope(q, rd, m, style=style).astype(np.float64),
                              oracle.rope(k, rd, n, style=style).astype(np.float64)))
            for shift in (1, 37, 150):
                d1 = float(np.dot(oracle.rope(q, rd, m + shift, style=style).astype(np.float64),
                                  oracle.rope(k, rd, n + shift, style=style).astype(np.float64)))
                assert abs(d0 - d1) < 1e-4 * max(1.0, abs(d0)), (m, n, shift, d0, d1)


# ---------------------------------------------------------------------------
# placement
# ---------------------------------------------------------------------------

def pin_placement_golden():
    tables = {"A": np.array([3, -1, 9, 1, 7], dtype=np.int32), "B": None}
    for case, slot, page, off in _read_golden("placement_points.txt"):
        got = oracle.place(int(slot), 4, tables[case], 8)
        exp = None if page == "none" else (int(page), int(off))
        assert got == exp, (case, slot, got, exp)


def _brute_place(ls, P, table, num_pages):
    """Search every (block, offset) whose slot is ls; no division."""
    if ls < 0:
        return None
    nblocks = len(table) if table is not None else num_pages
    for b in range(nblocks + 64):
        for o in range(P):
            if b * P + o == ls:
                if table is None:
                    page = b
                elif b < len(table):
                    page = int(table[b])
                else:
                    return None
                if 0 <= page < num_pages:
                    return (page, o)
                return None
    return None


def pin_placement_brute_force():
    rng = np.random.default_rng(9)
    P, npages = 4, 8
    for trial in range(20):
        table = rng.integers(-1, npages + 3, size=10).astype(np.int32)
        for ls in range(-2, 41):
            assert oracle.place(ls, P, table, npages) == _brute_place(ls, P, table, npages), (table, ls)
    for ls in range(-2, 41):
        assert oracle.place(ls, P, None, npages) == _brute_place(ls, P, None, npages)
    # a table whose buffer runs on past its stated length with valid pages: the
    # entries past the length must never be read
    buf = np.array([3, -1, 6, 1, 2, 2, 2, 2], dtype=np.int32)
    for ls in range(-2, 41):
        assert oracle.place(ls, P, buf, npages, table_len=4) == _brute_place(ls, P, buf[:4], npages)
    # 64-bit slots
    assert oracle.place(3 * 2**33 + 5, 64, None, 2**40) == (3 * 2**33 // 64, 5)


# ---------------------------------------------------------------------------
# the whole producer
# ---------------------------------------------------------------------------

def _tiny_pool_workload(seed, heads, rd=None, style=0, idx_k_dtype=wl.DTYPE_E4M3,
                        kv_dtype=wl.DTYPE_E4M3, page_pad=0, row_pad=0):
    """A small batch over tiny pools: P = 4, 8 pages, slots that cover padding,
    table entries of -1 and at or beyond the page count."""
    rng = np.random.default_rng(seed)
    P, npages, max_blocks = 4, 8, 3
    S = 4
    seq_positions = [[int(p)] for p in rng.integers(0, max_blocks * P, size=S)]
    seq_positions += [[0, 1, 2, 3, 4, 5]]          # a short prefill chunk
    w = wl.make_batch(f"tinypool{seed}", seed, heads, seq_positions, max_blocks=max_blocks,
                      num_pages=npages, rotary_dim=rd, rope_style=style, page_size=P,
                      kv_dtype=kv_dtype, idx_k_dtype=idx_k_dtype, page_pad_bytes=page_pad,
                      row_pad=row_pad, shuffle_pages=True)
    # make the table hold -1 and out-of-range entries, and add padded slots
    pt = np.array(w.page_table, copy=True)
    pt.reshape(-1)[::5] = -1
    pt.reshape(-1)[1::7] = npages + 2
    w.page_table = pt
    w.slot_mapping = np.array(w.slot_mapping, copy=True)
    w.slot_mapping[1] = -1
    return w


def _textbook_forward(w):
    """Float64 composition of the producer from library/textbook pieces:
    torch rms_norm, complex-rotation RoPE, torch casts."""
    s = w.shape
    D, rd = s["head_dim"], s["rotary_dim"]
    Hq, Hkv, Hiq, Hik = s["num_q_heads"], s["num_kv_heads"], s["num_idx_q_heads"], s["num_idx_k_heads"]
    x = bf16_bits_to_f32(w.qkv[:, :w.width]).astype(np.float64)
    wts = {k: bf16_bits_to_f32(v).astype(np.float64) for k, v in w.weights.items()}
    o = np.cumsum([0, Hq * D, Hkv * D, Hkv * D, Hiq * D, Hik * D])
    sec = {"q": (o[0], Hq), "k": (o[1], Hkv), "v": (o[2], Hkv), "idx_q": (o[3], Hiq), "idx_k": (o[4], Hik)}
    out = {}
    for name, (start, H) in sec.items():
        v = x[:, start:start + H * D].reshape(-1, H, D)
        if name != "v":
            v = torch.nn.functional.rms_norm(torch.from_numpy(v), (D,), torch.from_numpy(wts[name]),
                                             eps=s["rms_eps"]).numpy()
            v = np.stack([np.stack([_textbook_rope(v[t, h], rd, int(w.positions[t]), s["rope_theta"],
                                                   s["rope_style"]) for h in range(H)])
                          for t in range(v.shape[0])])
        out[name] = v
    return out


def _check_producer(w):
    q, iq, pools = run_oracle(w)
    init = wl.host_pools(w)
    ref = _textbook_forward(w)
    # compact outputs: one bf16 rounding of the float64 value, plus float32 noise
    for name, got in (("q", q), ("idx_q", iq)):
        g = bf16_bits_to_f32(got).astype(np.float64)
        r = ref[name]
        assert np.all(np.abs(g - r) <= 2.0 ** -8 * np.abs(r) + 2e-4), (name, np.abs(g - r).max())
    # placement from the brute-force search, not from the oracle
    P = w.shape["page_size"]
    pt = None if w.page_table is None else w.page_table.reshape(-1)
    touched = {p: np.zeros(n, dtype=bool) for p, n in w.pools.items()}
    for key in ("k", "v", "idx_k"):
        c = w.caches.get(key)
        if c is None:
            continue
        pls = [_brute_place(int(ls), P, pt, c.num_pages) for ls in w.slot_mapping]
        cells = cache_cells(w, key, pls)
        tok = [t for t, pl in enumerate(pls) if pl is not None]
        pool = pools[c.pool]
        if cells.size:
            assert not touched[c.pool][cells].any(), "two writes to one cell"
            touched[c.pool][cells] = True
        for i, t in enumerate(tok):
            for h in range(c.num_heads):
                got = pool[cells[i, h]]
                if c.dtype == wl.DTYPE_E4M3:
                    scale = np.float32(w.scales[{"k": 0, "v": 1, "idx_k": 2}[key]])
                    inv = np.float32(1.0) / scale
                    if key == "v":
                        # V: no norm, no RoPE: exactly the saturating cast of x * (1/s)
                        xv = bf16_bits_to_f32(w.qkv[t, (w.shape["num_q_heads"] + w.shape["num_kv_heads"]
                                                        + h) * w.shape["head_dim"]:][:w.shape["head_dim"]])
                        exp = _torch_e4m3(xv * inv)
                        assert np.array_equal(got, exp), (key, t, h)
                    else:
                        exp = _torch_e4m3((ref[key][t, h] * np.float64(inv)).astype(np.float32))
                        assert e4m3_ulp_distance(got, exp).max() <= 1, (key, t, h)
                else:
                    gv = bf16_bits_to_f32(got.view(np.uint16)).astype(np.float64)
                    r = ref[key][t, h]
                    assert np.all(np.abs(gv - r) <= 2.0 ** -8 * np.abs(r) + 2e-4), (key, t, h)
    # every byte outside the written cells is the sentinel it started as
    for p in pools:
        assert np.array_equal(pools[p][~touched[p]], init[p][~touched[p]]), f"stray write in pool {p}"


def pin_producer_tiny_shapes():
    _check_producer(_tiny_pool_workload(21, wl.TINY, idx_k_dtype=wl.DTYPE_BF16))


def pin_producer_big_shapes_partial_rope_strided():
    _check_producer(_tiny_pool_workload(22, wl.BIG, rd=64, page_pad=256, row_pad=64))


def pin_producer_gptj_bf16_caches():
    _check_producer(_tiny_pool_workload(23, wl.TINY, style=wl.ROPE_GPTJ, kv_dtype=wl.DTYPE_BF16,
                                       idx_k_dtype=wl.DTYPE_BF16))


def pin_producer_config1():
    _check_producer(wl.config1_tiny_decode())




# ---------------------------------------------------------------------------
# indexer
# ---------------------------------------------------------------------------

def _indexer_reference(w, pool):
    """Float64 composition from library pieces: dequantise the pool with torch's
    float8/bfloat16 views, gather each query's visible rows through the table,
    matrix-multiply with numpy, max over heads, np.maximum.at per block, and a
    stable lexsort for the ranking."""
    T, H, D = w.idx_q.shape
    c, P, BT = w.cache, w.page_size, w.block_tokens
    q = bf16_bits_to_f32(w.idx_q).astype(np.float64)
    base = torch.from_numpy(pool[c.offset:])
    if c.dtype == wl.DTYPE_E4M3:
        flat = base.view(torch.float8_e4m3fn).to(torch.float64).numpy() * np.float64(np.float32(w.k_scale))
    else:
        n = (base.numel() // 2) * 2
        flat = base[:n].view(torch.bfloat16).to(torch.float64).numpy()
    pt = w.page_table.reshape(-1)
    scores = np.full((T, w.max_blocks), -np.inf)
    for t in range(T):
        L = int(w.kv_len[t])
        j = np.arange(L)
        j = j[j // BT < w.max_blocks]
        ti = int(w.table_offset[t]) + j // P
        ok = (ti >= 0) & (ti < pt.size)
        j, ti = j[ok], ti[ok]
        page = pt[ti].astype(np.int64)
        ok = (page >= 0) & (page < c.num_pages)
        j, page = j[ok], page[ok]
        if j.size == 0:
            continue
        e = page * c.stride_page + (j % P) * c.stride_token
        kj = flat[e[:, None] + np.arange(D)[None, :]]
        tok = (q[t] @ kj.T).max(axis=0)
        np.maximum.at(scores[t], j // BT, tok)
    top = np.full((T, w.topk), -1, dtype=np.int64)
    for t in range(T):
        finite = np.nonzero(np.isfinite(scores[t]))[0]
        order = finite[np.lexsort((finite, -scores[t][finite]))]
        top[t, :min(w.topk, order.size)] = order[:w.topk]
    return scores, top


def _run_indexer_oracle(w, pool=None):
    pool = w.pool_fill if pool is None else pool
    return oracle.indexer(w.idx_q, w.kv_len, w.table_offset, w.page_table,
                          wl.indexer_cache_arg(w, pool), w.k_scale, w.page_size, w.block_tokens,
                          w.topk, w.max_blocks)


def check_indexer_against_reference(w, s, top, ref_s, ref_top):
    """Scores within fp32 accumulation error of the float64 reference; the ranking
    equal wherever the reference separates neighbours by more than that error."""
    fin = np.isfinite(ref_s)
    assert np.array_equal(np.isfinite(s), fin)
    tol = 1e-5 * (np.abs(ref_s[fin]).max(initial=1.0) + 1.0)
    assert np.abs(s[fin] - ref_s[fin]).max(initial=0.0) <= tol
    for t in range(s.shape[0]):
        for r in range(w.topk):
            a, b = int(top[t, r]), int(ref_top[t, r])
            if a == b:
                continue
            assert a >= 0 and b >= 0, (t, r, a, b)
            assert abs(ref_s[t, a] - ref_s[t, b]) <= 2 * tol, (t, r, a, b)


def same_indexer_results(w, a_scores, a_ids, b_scores, b_ids):
    """Two indexer entries agree: bit for bit, or (one of them on the tensor-core
    decode kernel, whose E4M3 query halves round differently) within the scores'
    tolerance, with the ids equal wherever the scores separate them."""
    if torch.equal(a_scores, b_scores) and torch.equal(a_ids, b_ids):
        return
    check_indexer_against_reference(w, a_scores.cpu().numpy(), a_ids.cpu().numpy(),
                                    b_scores.cpu().numpy().astype(np.float64), b_ids.cpu().numpy())


def pin_indexer_hand_worked():
    """H = 2 heads, D = 2, q = identity rows; bf16 cache of 2-token pages with the
    table [1, 0]; rows j0 = (3, -1), j1 = (-2, 5), j2 = (0.5, 0.5).  Token scores
    (max over heads) 3, 5, 0.5; 2-token blocks: block 0 = 5, block 1 = 0.5; top-3
    = [0, 1, -1]."""
    P, D = 2, 2
    rows = np.array([[0.5, 0.5], [0.0, 0.0], [3.0, -1.0], [-2.0, 5.0]], dtype=np.float32)
    pool = _torch_bf16(rows.reshape(-1)).view(np.uint8).copy()
    w = wl.IndexerWorkload("hand", _torch_bf16(np.array([[[1, 0], [0, 1]]], dtype=np.float32)),
                           np.array([3], dtype=np.int32), np.array([0], dtype=np.int64),
                           np.array([[1, 0]], dtype=np.int32),
                           wl.CacheSpec("idx_k", 0, wl.DTYPE_BF16, 2, 1, P * D, P * D, D),
                           pool.size, pool, 1.0, P, 2, 3, 3)
    s, top = _run_indexer_oracle(w)
    assert np.array_equal(s[0, :2], np.array([5.0, 0.5], dtype=np.float32)) and s[0, 2] == -np.inf
    assert top[0].tolist() == [0, 1, -1]


def pin_indexer_vs_reference():
    for dtype, D in ((wl.DTYPE_E4M3, 128), (wl.DTYPE_BF16, 64)):
        w = wl.make_indexer_batch("pin", 31 + D, [1, 63, 64, 65, 127, 128, 129, 700, 2048], heads=4,
                                  head_dim=D, dtype=dtype, topk=6)
        pt = np.array(w.page_table, copy=True)
        pt[7, 3] = -1                     # a hole: those tokens are skipped
        w.page_table = pt
        s, top = _run_indexer_oracle(w)
        ref_s, ref_top = _indexer_reference(w, w.pool_fill)
        check_indexer_against_reference(w, s, top, ref_s, ref_top)


def pin_indexer_ties_and_empty():
    w = wl.make_indexer_batch("ties", 41, [0, 256, 384], heads=2, head_dim=64,
                              dtype=wl.DTYPE_BF16, topk=4)
    pool = np.array(w.pool_fill, copy=True)
    # make block 2 of query 2 an exact copy of its block 0 (same rows, other pages)
    c = w.cache
    pt = w.page_table
    for j in range(128):
        src = c.offset + 2 * (int(pt[2, j // 64]) * c.stride_page + (j % 64) * c.stride_token)
        dst = c.offset + 2 * (int(pt[2, 4 + j // 64]) * c.stride_page + (j % 64) * c.stride_token)
        pool[dst:dst + 128] = pool[src:src + 128]
    s, top = _run_indexer_oracle(w, pool)
    assert np.all(s[0] == -np.inf) and top[0].tolist() == [-1] * 4
    assert s[2, 0] == s[2, 2]
    r0, r2 = top[2].tolist().index(0), top[2].tolist().index(2)
    assert r0 < r2 and (r2 == r0 + 1 or s[2, 1] == s[2, 0])
    assert top[1, 2:].tolist() == [-1, -1]


def pin_indexer_page_relabelling():
    w = wl.make_indexer_batch("relabel", 43, [300, 1000], heads=8, head_dim=128, topk=8)
    s0, t0 = _run_indexer_oracle(w)
    rng = np.random.default_rng(5)
    c = w.cache
    perm = rng.permutation(c.num_pages)
    pool = np.array(w.pool_fill, copy=True)
    for old, new in enumerate(perm):
        a = c.offset + old * c.stride_page
        b = c.offset + int(new) * c.stride_page
        pool[b:b + c.stride_page] = w.pool_fill[a:a + c.stride_page]
    w.page_table = np.where(w.page_table >= 0, perm[np.maximum(w.page_table, 0)], -1).astype(np.int32)
    s1, t1 = _run_indexer_oracle(w, pool)
    assert np.array_equal(s0, s1) and np.array_equal(t0, t1)


# ---------------------------------------------------------------------------
# the projection that feeds the producer
# ---------------------------------------------------------------------------

_BF16_NAN = 0x7FC0


def _round_significant(a: int, bits: int) -> int:
    """The non-negative integer a rounded to ``bits`` significant bits, ties to even."""
    shift = max(0, a.bit_length() - bits)
    q, r = divmod(a, 1 << shift)
    half = (1 << shift) >> 1
    if shift and (r > half or (r == half and (q & 1))):
        q += 1
    return q << shift


def _bf16_rne_of_int(n: int) -> int:
    """bf16 bits of the integer n after rounding to fp32 (24 significant bits) and
    then to bf16 (8 significant bits), each with ties to even, by integer
    arithmetic alone."""
    if n == 0:
        return 0
    sign = 0x8000 if n < 0 else 0
    v = _round_significant(_round_significant(abs(n), 24), 8)
    e = v.bit_length() - 1
    mant = (v >> (e - 7)) if e >= 7 else (v << (7 - e))
    return sign | ((e + 127) << 7) | (mant & 0x7F)


def _int_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Exact bf16 bits of small integers (|a| <= 256)."""
    out = np.array([_bf16_rne_of_int(int(v)) for v in a.reshape(-1)], dtype=np.uint16)
    assert all(bf16_bits_to_f32(np.array([b], dtype=np.uint16))[0] == float(v)
               for b, v in zip(out, a.reshape(-1)))
    return out.reshape(a.shape)


def _padded(bits: np.ndarray, pad: int) -> np.ndarray:
    """The same matrix inside a wider one whose extra columns hold NaN."""
    out = np.full((bits.shape[0], bits.shape[1] + pad), _BF16_NAN, dtype=np.uint16)
    out[:, :bits.shape[1]] = bits
    return out[:, :bits.shape[1]]


def pin_projection_exact_integers():
    """Small-integer operands: every dot product is an integer computed exactly in
    int64, then rounded to bf16 by integer arithmetic.  Row strides wider than the
    hidden size with NaN in the gap, magnitudes that force rounding, and a row whose
    exact sum needs cancellation beyond fp32 (2^25 + 1 - 2^25 = 1)."""
    rng = np.random.default_rng(71)
    T, K, W = 7, 40, 24
    h = rng.integers(-8, 9, size=(T, K))
    w = rng.integers(-8, 9, size=(W, K))
    w[5] = rng.integers(-128, 129, size=K)        # sums up to ~40k: rounded to 8 bits
    h[3] = rng.integers(-128, 129, size=K)
    w[0] = 1
    h[6] = 0
    hb = _int_to_bf16_bits(h)
    wb = _int_to_bf16_bits(w)
    # cancellation row: hidden [2^25, 1, -2^25, 0, ...]
    hb[6, 0], hb[6, 1], hb[6, 2] = 0x4C00, 0x3F80, 0xCC00
    h6 = np.zeros(K, dtype=object)
    h6[0], h6[1], h6[2] = 2**25, 1, -(2**25)
    exact = [[int(v) for v in row] for row in h.astype(np.int64) @ w.astype(np.int64).T]
    exact[6] = [int(sum(int(a) * int(b) for a, b in zip(h6, w[j]))) for j in range(W)]
    expect = np.array([[_bf16_rne_of_int(v) for v in row] for row in exact], dtype=np.uint16)
    got = oracle.projection(_padded(hb, 8), _padded(wb, 16))
    assert got[6, 0] == 0x3F80, "cancellation: the sum must be exact before rounding"
    assert np.array_equal(got, expect), np.argwhere(got != expect)[:5]


def pin_projection_signed_permutation():
    """Weight rows that are signed unit vectors pick (and negate) single hidden
    columns, so every output equals one input bit for bit: output j of token t is
    sign_j * hidden[t, perm_j], which fixes which operand is indexed by what."""
    rng = np.random.default_rng(72)
    T, K, W = 5, 48, 64
    x = rng.standard_normal((T, K)).astype(np.float32)
    x[np.abs(x) < 1e-3] = 0.5
    hb = np.asarray(torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy()).view(np.uint16)
    perm = rng.integers(0, K, size=W)
    sign = rng.choice([1, -1], size=W)
    wb = np.zeros((W, K), dtype=np.uint16)
    wb[np.arange(W), perm] = np.where(sign > 0, 0x3F80, 0xBF80)
    got = oracle.projection(_padded(hb, 24), wb)
    expect = hb[:, perm] ^ np.where(sign > 0, 0, 0x8000).astype(np.uint16)[None, :]
    assert np.array_equal(got, expect)


def _round_sig_frac(v, bits: int):
    """The rational v rounded to ``bits`` significant bits, ties to even (exact)."""
    from fractions import Fraction
    v = Fraction(v)
    if v == 0:
        return Fraction(0)
    sign = -1 if v < 0 else 1
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    unit = Fraction(2) ** (e - bits + 1)       # the spacing at this magnitude
    q, r = divmod(a, unit)
    q = int(q)
    if r > unit / 2 or (r == unit / 2 and (q & 1)):
        q += 1
    return sign * q * unit


def _bf16_bits_of_fraction(v) -> int:
    """bf16 bits of the rational v after rounding to fp32 and then to bf16 (RNE),
    by exact rational arithmetic (normal range only)."""
    from fractions import Fraction
    r = _round_sig_frac(_round_sig_frac(v, 24), 8)
    if r == 0:
        return 0
    sign = 0x8000 if r < 0 else 0
    a = abs(r)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    mant = int(a / Fraction(2) ** (e - 7)) & 0x7F
    return sign | ((e + 127) << 7) | mant


def _e4m3_codes(x: np.ndarray) -> np.ndarray:
    """E4M3 codes of values that E4M3 holds exactly, through torch's cast."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.float8_e4m3fn)
    codes = t.view(torch.uint8).numpy().copy()
    back = t.to(torch.float32).numpy()
    assert np.array_equal(back, x.astype(np.float32)), "value not exact in E4M3"
    return codes


def pin_projection_e4m3_exact_integers_and_scales():
    """E4M3 operands holding small integers, dyadic per-token and per-output scales:
    every output is an exact rational, rounded to fp32 then bf16 by exact rational
    arithmetic.  Distinct scales per token and per output fix which scale goes
    where."""
    from fractions import Fraction
    rng = np.random.default_rng(73)
    T, K, W = 6, 48, 20
    h = rng.integers(-8, 9, size=(T, K))
    w = rng.integers(-8, 9, size=(W, K))
    sx = np.array([0.5, 0.375, 1.25, 3.0, 0.0625, 1.0][:T], dtype=np.float32)
    sw = (np.array([0.25, 1.5, 0.625, 2.0, 0.75], dtype=np.float32)[np.arange(W) % 5]
          * np.float32(2.0) ** (np.arange(W) // 5)).astype(np.float32)
    hb = _e4m3_codes(h.astype(np.float32))
    wb = _e4m3_codes(w.astype(np.float32))
    pad_h = np.full((T, K + 16), 0x7F, dtype=np.uint8)
    pad_h[:, :K] = hb
    dots = h.astype(np.int64) @ w.astype(np.int64).T
    expect = np.array([[_bf16_bits_of_fraction(Fraction(int(dots[t, j])) * Fraction(float(sx[t]))
                                               * Fraction(float(sw[j])))
                        for j in range(W)] for t in range(T)], dtype=np.uint16)
    got = oracle.projection(pad_h[:, :K], wb, sx, sw)
    assert np.array_equal(got, expect), np.argwhere(got != expect)[:5]


def pin_projection_e4m3_signed_permutation():
    """E4M3 weights that are signed unit vectors: each output is one E4M3 hidden
    value, negated or not, which bf16 holds exactly."""
    rng = np.random.default_rng(74)
    T, K, W = 4, 64, 40
    codes = rng.integers(0, 256, size=(T, K)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x38          # no NaN codes
    codes[(codes & 0x7F) == 0x00] = 0x38          # no zeros (signed zeros would blur the check)
    vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float32)
    vbits = vals.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    perm = rng.integers(0, K, size=W)
    sign = rng.choice([1, -1], size=W)
    wb = np.zeros((W, K), dtype=np.uint8)
    wb[np.arange(W), perm] = np.where(sign > 0, 0x38, 0xB8)   # +-1.0
    got = oracle.projection(codes, wb)
    expect = vbits[:, perm] ^ np.where(sign > 0, 0, 0x8000).astype(np.uint16)[None, :]
    assert np.array_equal(got, expect)


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_") and callable(v)]
