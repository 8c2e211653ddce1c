"""Python binding of the producer's C ABI (argument marshalling only).

Every step of the producer runs in the CUDA library ``lib/libmsa_producer.so``;
this module only turns Python/torch arguments into the C call.  There is no CPU
or eager fallback: if the library has not been built, every call raises.

Names follow ``include/msa_producer.h``.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

MSA_OK = 0
MSA_ERR_INVALID_ARGUMENT = 1
MSA_ERR_UNSUPPORTED = 2
MSA_ERR_MISALIGNED = 3
MSA_ERR_OFFSET_OVERFLOW = 4
MSA_ERR_CUDA = 5

MSA_DTYPE_BF16 = 0
MSA_DTYPE_FP8_E4M3 = 1
MSA_ROPE_NEOX = 0
MSA_ROPE_GPTJ = 1
MSA_SCALE_PER_TENSOR = 0
MSA_SCALE_PER_HEAD = 1
MSA_LAUNCH_PERSISTENT = 1
MSA_LAUNCH_PDL = 2
MSA_LAUNCH_QUERY_RUNS = 4

# every function the header declares
EXPORTED = ("msa_producer_forward", "msa_producer_validate", "msa_producer_launch_shape",
            "msa_indexer_forward", "msa_indexer_forward_fused", "msa_indexer_forward_fused_noalloc",
            "msa_host_buffer_device_address",
            "msa_status_string",
            "msa_last_error_detail", "msa_projection_forward", "msa_projection_validate",
            "msa_checked_violations")

MSA_STATUS_WAIT_TIMEOUT = 1


class MsaError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}: {detail}")


class MsaCacheDesc(ctypes.Structure):
    _fields_ = [
        ("data", ctypes.c_void_p),
        ("dtype", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
        ("num_pages", ctypes.c_int64),
        ("num_heads", ctypes.c_int64),
        ("stride_page", ctypes.c_int64),
        ("stride_head", ctypes.c_int64),
        ("stride_token", ctypes.c_int64),
    ]


class MsaProducerCfg(ctypes.Structure):
    _fields_ = [
        ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("num_idx_q_heads", ctypes.c_int32),
        ("num_idx_k_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("rotary_dim", ctypes.c_int32),
        ("rope_style", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("rope_theta", ctypes.c_float),
        ("rms_eps", ctypes.c_float),
        ("scale_mode", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
    ]


class MsaIndexerCfg(ctypes.Structure):
    _fields_ = [
        ("num_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("block_tokens", ctypes.c_int32),
        ("topk", ctypes.c_int32),
        ("max_blocks", ctypes.c_int32),
        ("reserved", ctypes.c_int32 * 2),
    ]


_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return _build.LIB_PATH


def load(path: str | None = None) -> ctypes.CDLL:
    """Loads the CUDA library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or _build.LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                f"the CUDA producer library is not built ({p}); build it with "
                "`python -m paged_kv_cache_msa_gb300.build` (there is no CPU fallback)")
        L = ctypes.CDLL(p)
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
        cfgp, cachep = ctypes.POINTER(MsaProducerCfg), ctypes.POINTER(MsaCacheDesc)
        common = [cfgp, i64, vp, i64, vp, vp, vp, i64, vp, vp, vp, vp, vp, vp,
                  cachep, cachep, cachep, vp, i32]
        L.msa_producer_forward.argtypes = common + [vp]
        L.msa_producer_forward.restype = ctypes.c_int
        L.msa_producer_validate.argtypes = common
        L.msa_producer_validate.restype = ctypes.c_int
        L.msa_producer_launch_shape.argtypes = [cfgp, i64, i32, ctypes.POINTER(i32),
                                                ctypes.POINTER(i32), ctypes.POINTER(i32)]
        L.msa_producer_launch_shape.restype = ctypes.c_int
        L.msa_indexer_forward.argtypes = [ctypes.POINTER(MsaIndexerCfg), i64, vp, vp, vp, vp, i64,
                                          cachep, vp, vp, vp, i32, vp]
        L.msa_indexer_forward.restype = ctypes.c_int
        L.msa_indexer_forward_fused.argtypes = [ctypes.POINTER(MsaIndexerCfg), i64, vp, vp, vp, vp,
                                                i64, cachep, vp, vp, vp, vp, i32, vp]
        L.msa_indexer_forward_fused.restype = ctypes.c_int
        L.msa_indexer_forward_fused_noalloc.argtypes = [ctypes.POINTER(MsaIndexerCfg), i64, vp, vp,
                                                        vp, vp, i64, cachep, vp, vp, vp, i32, vp]
        L.msa_indexer_forward_fused_noalloc.restype = ctypes.c_int
        proj = [cfgp, i64, vp, i64, i64, vp, i64, ctypes.c_int, vp, vp, vp, vp, vp, i64, vp, vp,
                vp, vp, vp, vp, cachep, cachep, cachep, vp, vp, i64, vp]
        L.msa_projection_forward.argtypes = proj + [vp]
        L.msa_projection_forward.restype = ctypes.c_int
        L.msa_projection_validate.argtypes = proj
        L.msa_projection_validate.restype = ctypes.c_int
        L.msa_host_buffer_device_address.argtypes = [vp, ctypes.POINTER(ctypes.c_void_p)]
        L.msa_host_buffer_device_address.restype = ctypes.c_int
        L.msa_checked_violations.argtypes = [ctypes.POINTER(ctypes.c_uint64), i32]
        L.msa_checked_violations.restype = ctypes.c_int
        L.msa_status_string.argtypes = [ctypes.c_int]
        L.msa_status_string.restype = ctypes.c_char_p
        L.msa_last_error_detail.argtypes = []
        L.msa_last_error_detail.restype = ctypes.c_char_p
        if path is None:
            _lib = L
        return L


def status_string(status: int) -> str:
    return load().msa_status_string(int(status)).decode()


def last_error_detail() -> str:
    return load().msa_last_error_detail().decode()


def make_cfg(num_q_heads, num_kv_heads, num_idx_q_heads, num_idx_k_heads, head_dim,
             rotary_dim=None, rope_style=MSA_ROPE_NEOX, page_size=64, rope_theta=1e4,
             rms_eps=1e-6, scale_mode=MSA_SCALE_PER_TENSOR) -> MsaProducerCfg:
    c = MsaProducerCfg()
    c.num_q_heads, c.num_kv_heads = int(num_q_heads), int(num_kv_heads)
    c.num_idx_q_heads, c.num_idx_k_heads = int(num_idx_q_heads), int(num_idx_k_heads)
    c.head_dim = int(head_dim)
    c.rotary_dim = int(head_dim if rotary_dim is None else rotary_dim)
    c.rope_style, c.page_size = int(rope_style), int(page_size)
    c.rope_theta, c.rms_eps = float(rope_theta), float(rms_eps)
    c.scale_mode, c.reserved = int(scale_mode), 0
    return c


def make_cache(data_ptr: int, dtype: int, num_pages: int, num_heads: int, stride_page: int,
               stride_head: int, stride_token: int) -> MsaCacheDesc:
    d = MsaCacheDesc()
    d.data, d.dtype, d.reserved = int(data_ptr), int(dtype), 0
    d.num_pages, d.num_heads = int(num_pages), int(num_heads)
    d.stride_page, d.stride_head, d.stride_token = int(stride_page), int(stride_head), int(stride_token)
    return d


def _ref(x):
    return None if x is None else ctypes.byref(x)


def _args(cfg, num_tokens, qkv, qkv_row_stride, positions, slot_mapping, page_table,
          page_table_len, q_norm_w, k_norm_w, idx_q_norm_w, idx_k_norm_w, q_out, idx_q_out,
          k_cache, v_cache, idx_k_cache, scales, launch_flags):
    return (ctypes.byref(cfg) if cfg is not None else None, int(num_tokens), qkv,
            int(qkv_row_stride), positions, slot_mapping, page_table, int(page_table_len),
            q_norm_w, k_norm_w, idx_q_norm_w, idx_k_norm_w, q_out, idx_q_out,
            _ref(k_cache), _ref(v_cache), _ref(idx_k_cache), scales, int(launch_flags))


def msa_producer_forward(cfg, num_tokens, qkv, qkv_row_stride, positions, slot_mapping,
                         page_table, page_table_len, q_norm_w, k_norm_w, idx_q_norm_w,
                         idx_k_norm_w, q_out, idx_q_out, k_cache, v_cache, idx_k_cache, scales,
                         launch_flags=0, stream=0, check=True) -> int:
    """The C entry point; pointers are integers (device addresses) or None, the
    stream a ``cudaStream_t`` as an integer.  Raises MsaError unless the call
    returns MSA_OK (``check=False`` returns the status instead)."""
    L = load()
    s = L.msa_producer_forward(*_args(cfg, num_tokens, qkv, qkv_row_stride, positions,
                                      slot_mapping, page_table, page_table_len, q_norm_w,
                                      k_norm_w, idx_q_norm_w, idx_k_norm_w, q_out, idx_q_out,
                                      k_cache, v_cache, idx_k_cache, scales, launch_flags),
                               stream)
    if check and s != MSA_OK:
        raise MsaError(s, "msa_producer_forward", last_error_detail())
    return s


def msa_producer_validate(cfg, num_tokens, qkv, qkv_row_stride, positions, slot_mapping,
                          page_table, page_table_len, q_norm_w, k_norm_w, idx_q_norm_w,
                          idx_k_norm_w, q_out, idx_q_out, k_cache, v_cache, idx_k_cache, scales,
                          launch_flags=0) -> int:
    """The host-side checks alone; returns the status (no GPU needed)."""
    return load().msa_producer_validate(*_args(cfg, num_tokens, qkv, qkv_row_stride, positions,
                                               slot_mapping, page_table, page_table_len, q_norm_w,
                                               k_norm_w, idx_q_norm_w, idx_k_norm_w, q_out,
                                               idx_q_out, k_cache, v_cache, idx_k_cache, scales,
                                               launch_flags))


def _projection_args(cfg, num_tokens, hidden, hidden_size, hidden_row_stride, weight,
                     weight_row_stride, operand_dtype, hidden_scales, weight_scales, positions,
                     slot_mapping, page_table, page_table_len, q_norm_w, k_norm_w, idx_q_norm_w,
                     idx_k_norm_w, q_out, idx_q_out, k_cache, v_cache, idx_k_cache, scales,
                     rows_out, rows_out_stride, status):
    return (ctypes.byref(cfg) if cfg is not None else None, int(num_tokens), hidden,
            int(hidden_size), int(hidden_row_stride), weight, int(weight_row_stride),
            int(operand_dtype), hidden_scales, weight_scales, positions, slot_mapping, page_table,
            int(page_table_len), q_norm_w, k_norm_w, idx_q_norm_w, idx_k_norm_w, q_out, idx_q_out,
            _ref(k_cache), _ref(v_cache), _ref(idx_k_cache), scales, rows_out,
            int(rows_out_stride), status)


def msa_projection_forward(cfg, num_tokens, hidden, hidden_size, hidden_row_stride, weight,
                           weight_row_stride, operand_dtype, hidden_scales, weight_scales,
                           positions, slot_mapping, page_table, page_table_len, q_norm_w,
                           k_norm_w, idx_q_norm_w, idx_k_norm_w, q_out, idx_q_out, k_cache,
                           v_cache, idx_k_cache, scales, rows_out=None, rows_out_stride=0,
                           status=None, stream=0, check=True) -> int:
    """The projection GEMM with the producer in its epilogue (one launch); pointers
    are integers (device addresses) or None.  Raises MsaError unless MSA_OK
    (``check=False`` returns the status)."""
    L = load()
    s = L.msa_projection_forward(*_projection_args(
        cfg, num_tokens, hidden, hidden_size, hidden_row_stride, weight, weight_row_stride,
        operand_dtype, hidden_scales, weight_scales, positions, slot_mapping, page_table,
        page_table_len, q_norm_w, k_norm_w, idx_q_norm_w, idx_k_norm_w, q_out, idx_q_out, k_cache,
        v_cache, idx_k_cache, scales, rows_out, rows_out_stride, status), stream)
    if check and s != MSA_OK:
        raise MsaError(s, "msa_projection_forward", last_error_detail())
    return s


def msa_projection_validate(cfg, num_tokens, hidden, hidden_size, hidden_row_stride, weight,
                            weight_row_stride, operand_dtype, hidden_scales, weight_scales,
                            positions, slot_mapping, page_table, page_table_len, q_norm_w,
                            k_norm_w, idx_q_norm_w, idx_k_norm_w, q_out, idx_q_out, k_cache,
                            v_cache, idx_k_cache, scales, rows_out=None, rows_out_stride=0,
                            status=None) -> int:
    """The checks of msa_projection_forward alone; returns the status."""
    return load().msa_projection_validate(*_projection_args(
        cfg, num_tokens, hidden, hidden_size, hidden_row_stride, weight, weight_row_stride,
        operand_dtype, hidden_scales, weight_scales, positions, slot_mapping, page_table,
        page_table_len, q_norm_w, k_norm_w, idx_q_norm_w, idx_k_norm_w, q_out, idx_q_out, k_cache,
        v_cache, idx_k_cache, scales, rows_out, rows_out_stride, status))


def make_indexer_cfg(num_heads, head_dim, page_size=64, block_tokens=128, topk=16,
                     max_blocks=72) -> MsaIndexerCfg:
    c = MsaIndexerCfg()
    c.num_heads, c.head_dim, c.page_size = int(num_heads), int(head_dim), int(page_size)
    c.block_tokens, c.topk, c.max_blocks = int(block_tokens), int(topk), int(max_blocks)
    c.reserved[0] = c.reserved[1] = 0
    return c


def msa_indexer_forward(cfg, num_queries, idx_q, kv_len, table_offset, page_table,
                        page_table_len, idx_k_cache, k_scale, block_scores, topk_ids,
                        launch_flags=0, stream=0, check=True) -> int:
    """The C entry point; pointers are integers or None.  Raises MsaError unless the
    call returns MSA_OK (``check=False`` returns the status)."""
    s = load().msa_indexer_forward(ctypes.byref(cfg) if cfg is not None else None,
                                   int(num_queries), idx_q, kv_len, table_offset, page_table,
                                   int(page_table_len), _ref(idx_k_cache), k_scale,
                                   block_scores, topk_ids, int(launch_flags), stream)
    if check and s != MSA_OK:
        raise MsaError(s, "msa_indexer_forward", last_error_detail())
    return s


def msa_indexer_forward_fused(cfg, num_queries, idx_q, kv_len, table_offset, page_table,
                              page_table_len, idx_k_cache, k_scale, block_scores, topk_ids,
                              counters, launch_flags=0, stream=0, check=True) -> int:
    """The single-launch C entry point (``counters``: device int32 per query, zero on
    entry); pointers are integers or None.  Raises MsaError unless the call returns
    MSA_OK (``check=False`` returns the status)."""
    s = load().msa_indexer_forward_fused(ctypes.byref(cfg) if cfg is not None else None,
                                         int(num_queries), idx_q, kv_len, table_offset, page_table,
                                         int(page_table_len), _ref(idx_k_cache), k_scale,
                                         block_scores, topk_ids, counters, int(launch_flags), stream)
    if check and s != MSA_OK:
        raise MsaError(s, "msa_indexer_forward_fused", last_error_detail())
    return s


def msa_indexer_forward_fused_noalloc(cfg, num_queries, idx_q, kv_len, table_offset, page_table,
                                      page_table_len, idx_k_cache, k_scale, block_scores,
                                      topk_ids, launch_flags=0, stream=0, check=True) -> int:
    """The single-launch C entry point on the library's own counters; pointers are
    integers or None.  Raises MsaError unless the call returns MSA_OK (``check=False``
    returns the status)."""
    s = load().msa_indexer_forward_fused_noalloc(
        ctypes.byref(cfg) if cfg is not None else None, int(num_queries), idx_q, kv_len,
        table_offset, page_table, int(page_table_len), _ref(idx_k_cache), k_scale, block_scores,
        topk_ids, int(launch_flags), stream)
    if check and s != MSA_OK:
        raise MsaError(s, "msa_indexer_forward_fused_noalloc", last_error_detail())
    return s


def msa_checked_violations(reset: bool = True):
    """Stores skipped by a checked build since the last reset (synchronises the
    device); None for a normal build."""
    n = ctypes.c_uint64(0)
    s = load().msa_checked_violations(ctypes.byref(n), 1 if reset else 0)
    if s == MSA_ERR_UNSUPPORTED:
        return None
    if s != MSA_OK:
        raise MsaError(s, "msa_checked_violations", last_error_detail())
    return int(n.value)


def msa_host_buffer_device_address(host_ptr: int):
    """Device address of pinned, mapped host memory, or None when the buffer is not
    device-accessible."""
    out = ctypes.c_void_p()
    st = load().msa_host_buffer_device_address(host_ptr, ctypes.byref(out))
    return out.value if st == MSA_OK else None


def msa_producer_launch_shape(cfg, num_tokens, launch_flags=0):
    """(grid, block, dynamic smem bytes) the forward call would use."""
    g, b, s = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    st = load().msa_producer_launch_shape(ctypes.byref(cfg), int(num_tokens), int(launch_flags),
                                          ctypes.byref(g), ctypes.byref(b), ctypes.byref(s))
    if st != MSA_OK:
        raise MsaError(st, "msa_producer_launch_shape", last_error_detail())
    return g.value, b.value, s.value


# ---------------------------------------------------------------------------
# torch tensors -> C arguments
# ---------------------------------------------------------------------------

def _ptr(t):
    return None if t is None else int(t.data_ptr())


def cache_from_tensor(t, dtype: int | None = None) -> MsaCacheDesc:
    """Descriptor of a cache given as a (possibly non-contiguous) tensor view
    [num_pages, num_heads, page_size, head_dim] with unit dim stride.  The dtype
    comes from the tensor (bfloat16, float8_e4m3fn) unless given (for uint8 views
    of fp8 bytes)."""
    import torch
    assert t.dim() == 4 and t.stride(3) == 1, "cache view must be [pages, heads, P, D], dim stride 1"
    if dtype is None:
        if t.dtype == torch.bfloat16:
            dtype = MSA_DTYPE_BF16
        elif t.dtype in (torch.float8_e4m3fn, torch.uint8):
            dtype = MSA_DTYPE_FP8_E4M3
        else:
            raise TypeError(f"unsupported cache dtype {t.dtype}")
    return make_cache(t.data_ptr(), dtype, t.shape[0], t.shape[1], t.stride(0), t.stride(1),
                      t.stride(2))


def forward_tensors(cfg: MsaProducerCfg, qkv, positions, slot_mapping, page_table, norm_weights,
                    q_out, idx_q_out, k_cache, v_cache, idx_k_cache, scales, launch_flags=0,
                    stream=None) -> None:
    """msa_producer_forward on torch CUDA tensors.  ``qkv`` is [T, >= width] bf16
    with unit column stride; ``norm_weights`` a 4-tuple (q, k, idx_q, idx_k);
    caches are MsaCacheDesc (or None).  Runs on ``stream`` or the current stream."""
    import torch
    assert qkv.dim() == 2 and qkv.stride(1) == 1
    if stream is None:
        stream = torch.cuda.current_stream(qkv.device)
    pt_len = 0 if page_table is None else page_table.numel()
    wq, wk, wiq, wik = norm_weights
    msa_producer_forward(cfg, qkv.shape[0], _ptr(qkv), qkv.stride(0), _ptr(positions),
                         _ptr(slot_mapping), _ptr(page_table), pt_len, _ptr(wq), _ptr(wk),
                         _ptr(wiq), _ptr(wik), _ptr(q_out), _ptr(idx_q_out), k_cache, v_cache,
                         idx_k_cache, _ptr(scales), launch_flags, stream.cuda_stream)
