"""The C-ABI library on the host, with no GPU: it builds for sm_103a, loads, exports
every function the header declares, and its host-side checks accept well-formed
arguments and reject malformed ones without touching the GPU.

Pointers here are made-up aligned addresses: the checks only look at pointer
values, never at the memory behind them, and a rejected call launches nothing.
"""
import ctypes
import os
import re

import pytest

from paged_kv_cache_msa_gb300 import binding as B
from paged_kv_cache_msa_gb300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return B.load()


def declared_functions():
    names = set()
    inc = os.path.join(ROOT, "include")
    for h in sorted(os.listdir(inc)):
        if not h.endswith(".h"):
            continue
        with open(os.path.join(inc, h)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"\b(msa_[a-z_]+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_binding_surface():
    assert declared_functions() == sorted(B.EXPORTED)


def test_library_exports_every_declared_function(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings(lib):
    names = ["MSA_OK", "MSA_ERR_INVALID_ARGUMENT", "MSA_ERR_UNSUPPORTED", "MSA_ERR_MISALIGNED",
             "MSA_ERR_OFFSET_OVERFLOW", "MSA_ERR_CUDA"]
    for i, n in enumerate(names):
        assert B.status_string(i) == n
    assert B.status_string(99) == "MSA_ERR_UNKNOWN"


# ---------------------------------------------------------------------------
# a well-formed call (the big shapes, one HND fp8 pool per cache)
# ---------------------------------------------------------------------------

BASE = 0x7F0000000000


def good_call(T=16, **over):
    Hq, Hkv, Hiq, Hik, D, P = 64, 8, 8, 1, 128, 64
    cfg = B.make_cfg(Hq, Hkv, Hiq, Hik, D, 128, B.MSA_ROPE_NEOX, P)
    W = (Hq + 2 * Hkv + Hiq + Hik) * D
    npages = 1024

    def cache(i, heads, dtype=B.MSA_DTYPE_FP8_E4M3):
        return B.make_cache(BASE + (i + 10) * 2**34, dtype, npages, heads, heads * P * D, P * D, D)

    a = dict(cfg=cfg, num_tokens=T, qkv=BASE, qkv_row_stride=W, positions=BASE + 2**32,
             slot_mapping=BASE + 2**33, page_table=BASE + 3 * 2**32, page_table_len=1024,
             q_norm_w=BASE + 5 * 2**32, k_norm_w=BASE + 5 * 2**32 + 256,
             idx_q_norm_w=BASE + 5 * 2**32 + 512, idx_k_norm_w=BASE + 5 * 2**32 + 768,
             q_out=BASE + 6 * 2**32, idx_q_out=BASE + 7 * 2**32, k_cache=cache(0, Hkv),
             v_cache=cache(1, Hkv), idx_k_cache=cache(2, Hik), scales=BASE + 8 * 2**32,
             launch_flags=0)
    a.update(over)
    return a


def validate(a):
    return B.msa_producer_validate(**a)


def test_well_formed_call_passes(lib):
    assert validate(good_call()) == B.MSA_OK
    assert validate(good_call(launch_flags=B.MSA_LAUNCH_PERSISTENT | B.MSA_LAUNCH_PDL)) == B.MSA_OK
    assert validate(good_call(page_table=None, page_table_len=0)) == B.MSA_OK
    assert validate(good_call(idx_k_cache=None)) == B.MSA_OK


def test_zero_tokens_is_ok_without_launch(lib):
    # with zero tokens even the pointers may be null; forward returns before any CUDA call
    a = good_call(T=0, qkv=None, positions=None, slot_mapping=None)
    assert validate(a) == B.MSA_OK
    assert B.msa_producer_forward(**a, stream=0, check=False) == B.MSA_OK


def _cfg(**kw):
    base = dict(num_q_heads=64, num_kv_heads=8, num_idx_q_heads=8, num_idx_k_heads=1,
                head_dim=128, rotary_dim=128, rope_style=0, page_size=64)
    base.update(kw)
    return B.make_cfg(**base)


@pytest.mark.parametrize("over,status", [
    (dict(cfg=None), B.MSA_ERR_INVALID_ARGUMENT),
    (dict(num_tokens=-1), B.MSA_ERR_INVALID_ARGUMENT),
    (dict(qkv=None), B.MSA_ERR_INVALID_ARGUMENT),
    (dict(positions=None), B.MSA_ERR_INVALID_ARGUMENT),
    (dict(slot_mapping=None), B.MSA_ERR_INVALID_ARGUMENT),
    (dict(qkv_row_stride=89 * 128 - 8), B.MSA_ERR_INVALID_ARGUMENT),
    (dict(qkv=BASE + 8), B.MSA_ERR_MISALIGNED),
    (dict(qkv_row_stride=89 * 128 + 4), B.MSA_ERR_MISALIGNED),
    (dict(positions=BASE + 2**32 + 2), B.MSA_ERR_MISALIGNED),
    (dict(slot_mapping=BASE + 2**33 + 4), B.MSA_ERR_MISALIGNED),
    (dict(page_table_len=0), B.MSA_ERR_INVALID_ARGUMENT),
    (dict(page_table=BASE + 3 * 2**32 + 2), B.MSA_ERR_MISALIGNED),
    (dict(q_out=None), B.MSA_ERR_INVALID_ARGUMENT),
    (dict(q_out=BASE + 6 * 2**32 + 8), B.MSA_ERR_MISALIGNED),
    (dict(idx_q_out=None), B.MSA_ERR_INVALID_ARGUMENT),
    (dict(q_norm_w=None), B.MSA_ERR_INVALID_ARGUMENT),
    (dict(k_norm_w=None), B.MSA_ERR_INVALID_ARGUMENT),
    (dict(k_cache=None), B.MSA_ERR_INVALID_ARGUMENT),
    (dict(v_cache=None), B.MSA_ERR_INVALID_ARGUMENT),
    (dict(scales=None), B.MSA_ERR_INVALID_ARGUMENT),
    (dict(launch_flags=4), B.MSA_ERR_INVALID_ARGUMENT),
    (dict(cfg=_cfg(head_dim=96, rotary_dim=96)), B.MSA_ERR_UNSUPPORTED),
    (dict(cfg=_cfg(head_dim=0)), B.MSA_ERR_INVALID_ARGUMENT),
    (dict(cfg=_cfg(rotary_dim=136)), B.MSA_ERR_INVALID_ARGUMENT),
    (dict(cfg=_cfg(rotary_dim=-16)), B.MSA_ERR_INVALID_ARGUMENT),
    (dict(cfg=_cfg(rotary_dim=63)), B.MSA_ERR_INVALID_ARGUMENT),
    (dict(cfg=_cfg(rotary_dim=72)), B.MSA_ERR_UNSUPPORTED),
    (dict(cfg=_cfg(rope_style=7)), B.MSA_ERR_UNSUPPORTED),
    (dict(cfg=_cfg(page_size=0)), B.MSA_ERR_INVALID_ARGUMENT),
    (dict(cfg=_cfg(num_q_heads=-1)), B.MSA_ERR_INVALID_ARGUMENT),
    (dict(cfg=_cfg(num_q_heads=0, num_kv_heads=0, num_idx_q_heads=0, num_idx_k_heads=0)),
     B.MSA_ERR_INVALID_ARGUMENT),
    (dict(cfg=_cfg(num_kv_heads=4)), B.MSA_ERR_INVALID_ARGUMENT),   # cache num_heads mismatch
])
def test_malformed_call_is_rejected(lib, over, status):
    a = good_call(**over)
    got = validate(a)
    assert got == status, (B.status_string(got), B.last_error_detail())
    # forward returns the same status before touching the GPU
    assert B.msa_producer_forward(**a, stream=0, check=False) == status


def test_cfg_scalar_checks(lib):
    for kw, st in ((dict(rope_theta=0.0), B.MSA_ERR_INVALID_ARGUMENT),
                   (dict(rope_theta=float("inf")), B.MSA_ERR_INVALID_ARGUMENT),
                   (dict(rms_eps=-1e-6), B.MSA_ERR_INVALID_ARGUMENT),
                   (dict(rms_eps=float("nan")), B.MSA_ERR_INVALID_ARGUMENT),
                   (dict(scale_mode=5), B.MSA_ERR_UNSUPPORTED)):
        c = _cfg()
        for k, v in kw.items():
            setattr(c, k, v)
        assert validate(good_call(cfg=c)) == st, kw
    c = _cfg()
    c.reserved = 1
    assert validate(good_call(cfg=c)) == B.MSA_ERR_INVALID_ARGUMENT
    # GPT-J needs rotary_dim % 8, NeoX % 16; rotary_dim 0 needs no theta
    assert validate(good_call(cfg=_cfg(rope_style=1, rotary_dim=72))) == B.MSA_OK
    c = _cfg(rotary_dim=0)
    c.rope_theta = 0.0
    assert validate(good_call(cfg=c)) == B.MSA_OK


def _cache(**kw):
    d = dict(data_ptr=BASE + 10 * 2**34, dtype=B.MSA_DTYPE_FP8_E4M3, num_pages=1024, num_heads=8,
             stride_page=8 * 64 * 128, stride_head=64 * 128, stride_token=128)
    d.update(kw)
    return B.make_cache(**d)


@pytest.mark.parametrize("kw,status", [
    (dict(data_ptr=0), B.MSA_ERR_INVALID_ARGUMENT),
    (dict(data_ptr=BASE + 10 * 2**34 + 8), B.MSA_ERR_MISALIGNED),
    (dict(dtype=9), B.MSA_ERR_UNSUPPORTED),
    (dict(num_pages=-1), B.MSA_ERR_INVALID_ARGUMENT),
    (dict(stride_token=-128), B.MSA_ERR_INVALID_ARGUMENT),
    (dict(stride_token=132), B.MSA_ERR_MISALIGNED),
    (dict(stride_token=64), B.MSA_ERR_INVALID_ARGUMENT),            # rows overlap
    (dict(stride_head=64 * 128 - 8), B.MSA_ERR_INVALID_ARGUMENT),   # heads overlap
    (dict(stride_page=4 * 64 * 128), B.MSA_ERR_INVALID_ARGUMENT),   # pages overlap
    (dict(stride_page=2**62), B.MSA_ERR_OFFSET_OVERFLOW),
    (dict(num_pages=2**40, stride_page=2**30), B.MSA_ERR_OFFSET_OVERFLOW),
    (dict(data_ptr=2**64 - 2**20), B.MSA_ERR_OFFSET_OVERFLOW),     # wraps the address space
    (dict(num_heads=4), B.MSA_ERR_INVALID_ARGUMENT),
])
def test_malformed_cache_is_rejected(lib, kw, status):
    a = good_call(k_cache=_cache(**kw))
    got = validate(a)
    assert got == status, (B.status_string(got), B.last_error_detail())


def test_layouts_that_are_accepted(lib):
    P, D = 64, 128
    # K and V interleaved in one pool [pages, 2, 8, P, D]: page stride 2*8*P*D
    kv = dict(stride_page=2 * 8 * P * D, stride_head=P * D, stride_token=D)
    assert validate(good_call(k_cache=_cache(**kv), v_cache=_cache(**kv))) == B.MSA_OK
    # NHD pages [P, 8, D]
    assert validate(good_call(k_cache=_cache(stride_page=8 * P * D, stride_head=D,
                                             stride_token=8 * D))) == B.MSA_OK
    # padded pages; bf16 cache; a pool over 2^31 elements
    assert validate(good_call(k_cache=_cache(stride_page=8 * P * D + 256))) == B.MSA_OK
    assert validate(good_call(idx_k_cache=_cache(dtype=B.MSA_DTYPE_BF16, num_heads=1,
                                                 stride_page=P * D, stride_head=P * D))) == B.MSA_OK
    assert validate(good_call(k_cache=_cache(num_pages=24576, stride_page=2 * 8 * P * D))) == B.MSA_OK
    # a cache with zero pages is accepted (it takes no token)
    assert validate(good_call(k_cache=_cache(num_pages=0))) == B.MSA_OK


def test_bf16_only_caches_need_no_scales(lib):
    P, D = 64, 128
    bf = lambda h: _cache(dtype=B.MSA_DTYPE_BF16, num_heads=h, stride_page=h * P * D,
                          stride_head=P * D)
    a = good_call(k_cache=bf(8), v_cache=bf(8), idx_k_cache=bf(1), scales=None)
    assert validate(a) == B.MSA_OK


def test_per_head_scale_limit(lib):
    c = _cfg(scale_mode=B.MSA_SCALE_PER_HEAD)
    assert validate(good_call(cfg=c)) == B.MSA_OK
    c = _cfg(scale_mode=B.MSA_SCALE_PER_HEAD, num_kv_heads=200)
    a = good_call(cfg=c, k_cache=_cache(num_heads=200, stride_page=200 * 64 * 128),
                  v_cache=_cache(num_heads=200, stride_page=200 * 64 * 128))
    assert validate(a) == B.MSA_ERR_UNSUPPORTED


def test_host_buffer_helper_rejects_null(lib):
    out = ctypes.c_void_p()
    assert lib.msa_host_buffer_device_address(None, ctypes.byref(out)) == B.MSA_ERR_INVALID_ARGUMENT
    assert lib.msa_host_buffer_device_address(ctypes.c_void_p(BASE), None) == B.MSA_ERR_INVALID_ARGUMENT


# ---------------------------------------------------------------------------
# the indexer's host checks
# ---------------------------------------------------------------------------

def good_indexer_call(**over):
    cfg = B.make_indexer_cfg(8, 128, 64, 128, 16, 72)
    cache = B.make_cache(BASE + 20 * 2**34, B.MSA_DTYPE_FP8_E4M3, 9216, 1, 64 * 128, 64 * 128, 128)
    a = dict(cfg=cfg, num_queries=64, idx_q=BASE, kv_len=BASE + 2**32, table_offset=BASE + 2**33,
             page_table=BASE + 3 * 2**32, page_table_len=9216, idx_k_cache=cache,
             k_scale=BASE + 5 * 2**32, block_scores=BASE + 6 * 2**32, topk_ids=BASE + 7 * 2**32)
    a.update(over)
    return a


def _icfg(**kw):
    base = dict(num_heads=8, head_dim=128, page_size=64, block_tokens=128, topk=16, max_blocks=72)
    base.update(kw)
    return B.make_indexer_cfg(**base)


@pytest.mark.parametrize("over,status", [
    (dict(num_queries=0, idx_q=None), B.MSA_OK),
    (dict(cfg=None), B.MSA_ERR_INVALID_ARGUMENT),
    (dict(num_queries=-1), B.MSA_ERR_INVALID_ARGUMENT),
    (dict(idx_q=None), B.MSA_ERR_INVALID_ARGUMENT),
    (dict(block_scores=None), B.MSA_ERR_INVALID_ARGUMENT),
    (dict(k_scale=None), B.MSA_ERR_INVALID_ARGUMENT),
    (dict(page_table_len=0), B.MSA_ERR_INVALID_ARGUMENT),
    (dict(idx_q=BASE + 8), B.MSA_ERR_MISALIGNED),
    (dict(table_offset=BASE + 2**33 + 4), B.MSA_ERR_MISALIGNED),
    (dict(cfg=_icfg(num_heads=17)), B.MSA_ERR_UNSUPPORTED),
    (dict(cfg=_icfg(head_dim=96)), B.MSA_ERR_UNSUPPORTED),
    (dict(cfg=_icfg(block_tokens=100)), B.MSA_ERR_UNSUPPORTED),
    (dict(cfg=_icfg(topk=0)), B.MSA_ERR_UNSUPPORTED),
    (dict(cfg=_icfg(max_blocks=0)), B.MSA_ERR_UNSUPPORTED),
    (dict(cfg=_icfg(page_size=0)), B.MSA_ERR_INVALID_ARGUMENT),
    (dict(num_queries=2**30), B.MSA_ERR_UNSUPPORTED),
    (dict(idx_k_cache=B.make_cache(BASE + 20 * 2**34, B.MSA_DTYPE_FP8_E4M3, 9216, 1, 64 * 128 + 8,
                                   64 * 128, 128)), B.MSA_ERR_MISALIGNED),
    (dict(idx_k_cache=B.make_cache(BASE + 20 * 2**34, B.MSA_DTYPE_FP8_E4M3, 9216, 2, 64 * 128,
                                   64 * 128, 128)), B.MSA_ERR_INVALID_ARGUMENT),
    (dict(launch_flags=B.MSA_LAUNCH_PERSISTENT), B.MSA_ERR_INVALID_ARGUMENT),
    (dict(launch_flags=8), B.MSA_ERR_INVALID_ARGUMENT),
])
def test_indexer_host_checks(lib, over, status):
    a = good_indexer_call(**over)
    # rejected calls (and an empty one) return before touching the GPU
    got = B.msa_indexer_forward(**a, stream=0, check=False)
    assert got == status, (B.status_string(got), B.last_error_detail())
    # the single-launch entry checks the same arguments the same way
    got = B.msa_indexer_forward_fused(**a, counters=BASE + 30 * 2**32, stream=0, check=False)
    assert got == status, (B.status_string(got), B.last_error_detail())


@pytest.mark.parametrize("counters,status", [
    (None, B.MSA_ERR_INVALID_ARGUMENT),
    (BASE + 30 * 2**32 + 2, B.MSA_ERR_MISALIGNED),
])
def test_indexer_fused_counter_checks(lib, counters, status):
    for nq in (64, 0):   # the counters are checked before an empty call returns
        a = good_indexer_call(num_queries=nq)
        got = B.msa_indexer_forward_fused(**a, counters=counters, stream=0, check=False)
        assert got == status, (B.status_string(got), B.last_error_detail())


# ---------------------------------------------------------------------------
# the projection entry point: host-side checks
# ---------------------------------------------------------------------------

def good_projection(**over):
    a = good_call()
    for k in ("qkv", "qkv_row_stride", "launch_flags"):
        a.pop(k)
    a.update(hidden=BASE + 9 * 2**32, hidden_size=6144, hidden_row_stride=6144,
             weight=BASE + 10 * 2**32, weight_row_stride=6144, operand_dtype=B.MSA_DTYPE_BF16,
             hidden_scales=None, weight_scales=None, rows_out=None, rows_out_stride=0,
             status=BASE + 11 * 2**32)
    a.update(over)
    return a


def test_projection_well_formed_calls_pass(lib):
    assert B.msa_projection_validate(**good_projection()) == B.MSA_OK
    assert B.msa_projection_validate(**good_projection(status=None)) == B.MSA_OK
    assert B.msa_projection_validate(**good_projection(hidden_size=200, hidden_row_stride=208,
                                                       weight_row_stride=200)) == B.MSA_OK
    assert B.msa_projection_validate(**good_projection(rows_out=BASE + 12 * 2**32,
                                                       rows_out_stride=89 * 128)) == B.MSA_OK
    fp8 = dict(operand_dtype=B.MSA_DTYPE_FP8_E4M3, hidden_scales=BASE + 13 * 2**32,
               weight_scales=BASE + 14 * 2**32)
    assert B.msa_projection_validate(**good_projection(**fp8)) == B.MSA_OK
    assert B.msa_projection_validate(**good_projection(**fp8, hidden_row_stride=6160)) == B.MSA_OK


def test_projection_zero_tokens_is_ok_without_launch(lib):
    a = good_projection(num_tokens=0, hidden=None, weight=None, positions=None, slot_mapping=None)
    assert B.msa_projection_validate(**a) == B.MSA_OK
    assert B.msa_projection_forward(**a, stream=0, check=False) == B.MSA_OK


@pytest.mark.parametrize("over,status", [
    (dict(hidden=None), B.MSA_ERR_INVALID_ARGUMENT),
    (dict(weight=None), B.MSA_ERR_INVALID_ARGUMENT),
    (dict(hidden_size=0), B.MSA_ERR_INVALID_ARGUMENT),
    (dict(hidden_row_stride=6136), B.MSA_ERR_INVALID_ARGUMENT),
    (dict(weight_row_stride=6136), B.MSA_ERR_INVALID_ARGUMENT),
    (dict(hidden=BASE + 9 * 2**32 + 8), B.MSA_ERR_MISALIGNED),
    (dict(weight=BASE + 10 * 2**32 + 2), B.MSA_ERR_MISALIGNED),
    (dict(hidden_row_stride=6148), B.MSA_ERR_MISALIGNED),
    (dict(weight_row_stride=6150), B.MSA_ERR_MISALIGNED),
    (dict(rows_out=BASE + 12 * 2**32, rows_out_stride=89 * 128 - 8), B.MSA_ERR_INVALID_ARGUMENT),
    (dict(rows_out=BASE + 12 * 2**32 + 4, rows_out_stride=89 * 128), B.MSA_ERR_MISALIGNED),
    (dict(status=BASE + 11 * 2**32 + 2), B.MSA_ERR_MISALIGNED),
    (dict(num_tokens=2**31), B.MSA_ERR_UNSUPPORTED),
    (dict(positions=None), B.MSA_ERR_INVALID_ARGUMENT),
    (dict(q_out=None), B.MSA_ERR_INVALID_ARGUMENT),
    (dict(k_cache=None), B.MSA_ERR_INVALID_ARGUMENT),
    (dict(scales=None), B.MSA_ERR_INVALID_ARGUMENT),
    (dict(cfg=_cfg(head_dim=96, rotary_dim=96)), B.MSA_ERR_UNSUPPORTED),
    (dict(operand_dtype=7), B.MSA_ERR_UNSUPPORTED),
    (dict(operand_dtype=B.MSA_DTYPE_FP8_E4M3, hidden_row_stride=6152), B.MSA_ERR_MISALIGNED),
    (dict(operand_dtype=B.MSA_DTYPE_FP8_E4M3, weight_row_stride=6152), B.MSA_ERR_MISALIGNED),
    (dict(hidden_scales=BASE + 13 * 2**32 + 2), B.MSA_ERR_MISALIGNED),
    (dict(weight_scales=BASE + 14 * 2**32 + 1), B.MSA_ERR_MISALIGNED),
])
def test_projection_malformed_call_is_rejected(lib, over, status):
    a = good_projection(**over)
    assert B.msa_projection_validate(**a) == status, B.last_error_detail()
    assert B.msa_projection_forward(**a, stream=0, check=False) == status


def test_build_reuse_is_keyed_on_source_content(tmp_path):
    """A library on disk is reused only when the digest of its sources, build
    script, command line and defines matches the one recorded beside it; any
    change of a source byte or a define makes build() compile again."""
    build_mod.build()
    d0 = build_mod.source_digest(())
    assert build_mod.up_to_date(())
    assert build_mod.source_digest(("MSA_STAGES=3",)) != d0
    assert not build_mod.up_to_date(("MSA_STAGES=3",))
    # a copy of the sources with one byte changed hashes differently
    src = build_mod.SOURCES[0]
    saved = list(build_mod.DEPENDENCIES)
    changed = tmp_path / os.path.basename(src)
    with open(src, "rb") as f:
        data = f.read()
    changed.write_bytes(data + b"\n")
    try:
        build_mod.DEPENDENCIES[build_mod.DEPENDENCIES.index(src)] = str(changed)
        assert build_mod.source_digest(()) != d0
    finally:
        build_mod.DEPENDENCIES[:] = saved
    assert build_mod.source_digest(()) == d0
