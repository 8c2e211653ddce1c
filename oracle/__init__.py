"""CPU oracle for the MiniMax-M3 MSA fused producer and paged-cache write.

TEST INFRASTRUCTURE ONLY.  The definition lives in ``msa_oracle.c`` (single-threaded
C99, single precision, no fast-math, no contraction).  This module compiles it with
gcc and exposes it through ctypes.  Only the test suite, the smoke check and the
benchmark's CPU-baseline leg import it; the CUDA product path does not, and shares
no code with it.

The pages the oracle follows are cited in ``msa_oracle.c``:
"[None][perf] Fuse MiniMax-M3 QKV and index projection" (TensorRT-LLM PR 18205,
Description), "[None][perf] Fuse MiniMax-M3 MSA per-layer KV-cache writes into one
kernel" (PR 18614, "The problem" / "The fix") and "Wire in custom decode kernels
for MinimaxM3" (PR 18611, merge commit message).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "msa_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libmsa_oracle.so")

DTYPE_BF16 = 0
DTYPE_E4M3 = 1
ROPE_NEOX = 0
ROPE_GPTJ = 1
SCALE_PER_TENSOR = 0
SCALE_PER_HEAD = 1

# Flags: plain C99, no fast-math, no floating-point contraction, so that the
# x86-64 and AArch64 builds compute the same bits.
CFLAGS = ["-std=c99", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]


def build(force: bool = False) -> str:
    """Compiles the oracle with gcc into ``oracle/_build`` and returns the path."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    subprocess.run(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class OracleShape(ctypes.Structure):
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


class OracleCache(ctypes.Structure):
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


_lib = None
_lock = threading.Lock()


def load(path: str) -> ctypes.CDLL:
    """Loads an oracle build from ``path`` and declares its exported signatures."""
    L = ctypes.CDLL(path)
    L.oracle_bf16_decode.argtypes = [ctypes.c_uint16]
    L.oracle_bf16_decode.restype = ctypes.c_float
    L.oracle_bf16_encode.argtypes = [ctypes.c_float]
    L.oracle_bf16_encode.restype = ctypes.c_uint16
    L.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
    L.oracle_e4m3_decode.restype = ctypes.c_float
    L.oracle_e4m3_encode.argtypes = [ctypes.c_float]
    L.oracle_e4m3_encode.restype = ctypes.c_uint8
    fp = ctypes.POINTER(ctypes.c_float)
    L.oracle_rmsnorm.argtypes = [fp, fp, ctypes.c_int32, ctypes.c_float, fp]
    L.oracle_rmsnorm.restype = None
    L.oracle_rope.argtypes = [fp, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                              ctypes.c_float, ctypes.c_int32]
    L.oracle_rope.restype = None
    L.oracle_place.argtypes = [ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p,
                               ctypes.c_int64, ctypes.c_int64,
                               ctypes.POINTER(ctypes.c_int64),
                               ctypes.POINTER(ctypes.c_int64)]
    L.oracle_place.restype = ctypes.c_int
    vp = ctypes.c_void_p
    L.oracle_forward.argtypes = [
        ctypes.POINTER(OracleShape), ctypes.c_int64,
        vp, ctypes.c_int64,
        vp, vp, vp, ctypes.c_int64,
        vp, vp, vp, vp,
        vp, vp,
        ctypes.POINTER(OracleCache), ctypes.POINTER(OracleCache),
        ctypes.POINTER(OracleCache), vp,
    ]
    L.oracle_forward.restype = ctypes.c_int
    L.oracle_indexer.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                 ctypes.c_int32, ctypes.c_int64, vp, vp, vp, vp, ctypes.c_int64,
                                 ctypes.POINTER(OracleCache), ctypes.c_float, ctypes.c_int32,
                                 vp, vp]
    L.oracle_indexer.restype = ctypes.c_int
    L.oracle_projection.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int32, vp,
                                    ctypes.c_int64, vp, ctypes.c_int64, vp, ctypes.c_int64, vp,
                                    vp, ctypes.c_int64]
    L.oracle_projection.restype = ctypes.c_int
    return L


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            _lib = load(build())
    return _lib


# --------------------------------------------------------------------------
# scalar helpers (for the pins)
# --------------------------------------------------------------------------

def bf16_encode(x: float) -> int:
    return int(lib().oracle_bf16_encode(float(x)))


def bf16_decode(h: int) -> float:
    return float(lib().oracle_bf16_decode(int(h)))


def e4m3_encode(x: float) -> int:
    return int(lib().oracle_e4m3_encode(float(x)))


def e4m3_decode(c: int) -> float:
    return float(lib().oracle_e4m3_decode(int(c)))


def _fptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_float))


def rmsnorm(x, w=None, eps: float = 1e-6) -> np.ndarray:
    """One head: y = (x * r) * w, r = 1/sqrt(mean(x^2) + eps); float32 in and out."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty_like(x)
    if w is None:
        wp = ctypes.cast(None, ctypes.POINTER(ctypes.c_float))
    else:
        w = np.ascontiguousarray(w, dtype=np.float32)
        wp = _fptr(w)
    lib().oracle_rmsnorm(_fptr(x), wp, x.size, float(eps), _fptr(y))
    return y


def rope(y, rotary_dim: int, pos: int, theta: float = 1e4, style: int = ROPE_NEOX) -> np.ndarray:
    """One head, rotated in a copy; float32 in and out."""
    y = np.array(y, dtype=np.float32, copy=True)
    lib().oracle_rope(_fptr(y), y.size, int(rotary_dim), int(style), float(theta), int(pos))
    return y


def place(ls: int, page_size: int, page_table, num_pages: int, table_len: int | None = None):
    """Returns (page, off) or None for a slot that writes nothing.  ``table_len``
    (default: the array's size) is the table length the oracle is told."""
    page = ctypes.c_int64(-1)
    off = ctypes.c_int64(-1)
    if page_table is None:
        ptp, ptl = None, 0
    else:
        page_table = np.ascontiguousarray(page_table, dtype=np.int32)
        ptp = page_table.ctypes.data
        ptl = page_table.size if table_len is None else int(table_len)
        assert 0 <= ptl <= page_table.size
    ok = lib().oracle_place(int(ls), int(page_size), ptp, ptl, int(num_pages),
                            ctypes.byref(page), ctypes.byref(off))
    return (page.value, off.value) if ok else None


# --------------------------------------------------------------------------
# the whole producer over host arrays
# --------------------------------------------------------------------------

def _cache_struct(c):
    """c: None or dict(data=np.uint8 array (the whole allocation), offset=bytes to
    element 0, dtype, num_pages, num_heads, stride_page, stride_head, stride_token)."""
    if c is None:
        return None
    s = OracleCache()
    s.data = c["data"].ctypes.data + int(c.get("offset", 0))
    s.dtype = int(c["dtype"])
    s.num_pages = int(c["num_pages"])
    s.num_heads = int(c["num_heads"])
    s.stride_page = int(c["stride_page"])
    s.stride_head = int(c["stride_head"])
    s.stride_token = int(c["stride_token"])
    return s


def forward(shape: dict, qkv: np.ndarray, row_stride: int, positions: np.ndarray,
            slot_mapping: np.ndarray, page_table, weights: dict, q_out: np.ndarray,
            idx_q_out: np.ndarray, k_cache, v_cache, idx_k_cache, scales: np.ndarray,
            num_tokens: int | None = None, token_offset: int = 0) -> None:
    """Runs the oracle in place on host arrays.

    qkv: uint16 (bf16 bits), at least [T, row_stride]; positions int32 [T];
    slot_mapping int64 [T]; page_table int32 (any shape, flattened) or None;
    weights: dict q/k/idx_q/idx_k -> uint16 [D] (bf16 bits) or None (unit);
    q_out uint16 [T, Hq, D]; idx_q_out uint16 [T, Hiq, D];
    caches: see ``_cache_struct``; scales float32.
    ``num_tokens``/``token_offset`` run a sub-range of tokens (for timing samples).
    """
    sh = OracleShape()
    for k in ("num_q_heads", "num_kv_heads", "num_idx_q_heads", "num_idx_k_heads",
              "head_dim", "rotary_dim", "rope_style", "page_size"):
        setattr(sh, k, int(shape[k]))
    sh.rope_theta = float(shape["rope_theta"])
    sh.rms_eps = float(shape["rms_eps"])
    sh.scale_mode = int(shape.get("scale_mode", SCALE_PER_TENSOR))

    T = positions.shape[0] if num_tokens is None else int(num_tokens)
    t0 = int(token_offset)
    assert qkv.dtype == np.uint16 and qkv.flags.c_contiguous
    assert positions.dtype == np.int32 and slot_mapping.dtype == np.int64
    assert q_out.dtype == np.uint16 and idx_q_out.dtype == np.uint16
    D = sh.head_dim
    if page_table is None:
        ptp, ptl = None, 0
    else:
        assert page_table.dtype == np.int32 and page_table.flags.c_contiguous
        ptp, ptl = page_table.ctypes.data, page_table.size

    def wp(name):
        w = weights.get(name)
        if w is None:
            return None
        assert w.dtype == np.uint16 and w.size == D
        return w.ctypes.data

    kc, vc, ic = (_cache_struct(c) for c in (k_cache, v_cache, idx_k_cache))
    scales = np.ascontiguousarray(scales, dtype=np.float32)
    qkv_ptr = qkv.ctypes.data + 2 * t0 * int(row_stride)
    rc = lib().oracle_forward(
        ctypes.byref(sh), T,
        qkv_ptr, int(row_stride),
        positions.ctypes.data + 4 * t0, slot_mapping.ctypes.data + 8 * t0, ptp, ptl,
        wp("q"), wp("k"), wp("idx_q"), wp("idx_k"),
        q_out.ctypes.data + 2 * t0 * sh.num_q_heads * D,
        idx_q_out.ctypes.data + 2 * t0 * sh.num_idx_q_heads * D,
        ctypes.byref(kc) if kc else None, ctypes.byref(vc) if vc else None,
        ctypes.byref(ic) if ic else None, scales.ctypes.data)
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (rc={rc})")


def indexer(idx_q: np.ndarray, kv_len: np.ndarray, table_offset: np.ndarray, page_table,
            idx_k_cache: dict, k_scale: float, page_size: int, block_tokens: int, topk: int,
            max_blocks: int):
    """Block scores [T, max_blocks] (float32) and top-k block ids [T, topk] (int32).
    idx_q: uint16 (bf16 bits) [T, H, D]; kv_len int32 [T]; table_offset int64 [T];
    page_table int32 (flattened); idx_k_cache: see ``_cache_struct`` (one head)."""
    T, H, D = idx_q.shape
    assert idx_q.dtype == np.uint16 and idx_q.flags.c_contiguous
    kv_len = np.ascontiguousarray(kv_len, dtype=np.int32)
    table_offset = np.ascontiguousarray(table_offset, dtype=np.int64)
    pt = np.ascontiguousarray(page_table, dtype=np.int32).reshape(-1)
    scores = np.empty((T, max_blocks), dtype=np.float32)
    top = np.empty((T, topk), dtype=np.int32)
    c = _cache_struct(idx_k_cache)
    rc = lib().oracle_indexer(H, D, int(page_size), int(block_tokens), int(topk), T,
                              idx_q.ctypes.data, kv_len.ctypes.data, table_offset.ctypes.data,
                              pt.ctypes.data, pt.size, ctypes.byref(c), float(k_scale),
                              int(max_blocks), scores.ctypes.data, top.ctypes.data)
    if rc != 0:
        raise ValueError("oracle rejected the indexer arguments")
    return scores, top


def projection(hidden: np.ndarray, weight: np.ndarray, hidden_scales=None,
               weight_scales=None) -> np.ndarray:
    """The projection rows [T, W] (uint16, bf16 bits) of hidden [T, K] and the
    output-major weight [W, K]: both uint16 (bf16 bits) or both uint8 (E4M3
    codes).  Row strides may exceed K (pass a column slice of a wider array).
    ``hidden_scales`` float32 [T] and ``weight_scales`` float32 [W] (or None: 1)."""
    assert hidden.dtype == weight.dtype and hidden.dtype in (np.uint16, np.uint8)
    assert hidden.ndim == 2 and weight.ndim == 2
    es = hidden.itemsize
    dtype = DTYPE_BF16 if es == 2 else DTYPE_E4M3
    T, K = hidden.shape
    W, K2 = weight.shape
    assert K == K2
    assert hidden.strides[1] == es and weight.strides[1] == es
    sx = None if hidden_scales is None else np.ascontiguousarray(hidden_scales, dtype=np.float32)
    sw = None if weight_scales is None else np.ascontiguousarray(weight_scales, dtype=np.float32)
    assert sx is None or sx.shape == (T,)
    assert sw is None or sw.shape == (W,)
    rows = np.empty((T, W), dtype=np.uint16)
    rc = lib().oracle_projection(T, K, dtype, hidden.ctypes.data, hidden.strides[0] // es,
                                 None if sx is None else sx.ctypes.data, W,
                                 weight.ctypes.data, weight.strides[0] // es,
                                 None if sw is None else sw.ctypes.data, rows.ctypes.data, W)
    if rc != 0:
        raise ValueError("oracle rejected the projection arguments")
    return rows
