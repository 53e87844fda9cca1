"""CPU oracle for the paged KV cache decode path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The library (``paged_kv_cache_261_gb300``)
never does, and the two share no code: this package holds a float64 C program
(``pagedattn_oracle.c``, loaded with ctypes) and a Python model of the block
manager (``allocator_model.py``).

What it computes and where that is defined (web pages, by title and section):
  - scatter of new tokens into cache slots: "PagedAttention实现", write_kv;
    "04 - Paged Attention 实现进度", B.2 (slot_mapping);
  - whole-block copy for copy-on-write: "PagedAttention实现", cow_write;
  - decode attention: "CS349E lecture 7: 01_paged_attention.py", demo 2,
    paper eq. 4 (block-wise scores, one softmax over the whole context,
    block-wise V accumulation, equal to contiguous attention);
  - chunked-prefill attention: the same per query position, each seeing the
    positions up to its own (demo 1/demo 2 paged steps; "04 - Paged Attention
    实现进度", B.2 and D.2, cu_seqlens_q / query_start_loc);
  - 8-bit cache (a reading of this project, not on the pages): OCP FP8 E4M3
    codes with one float32 scale for K and one for V; scatter = nearest code of
    x / scale (float32 division), decode attention = the float64 attention over
    decoded(code) * scale (pinned in ``tests/test_oracle_fp8_pins.py``);
  - block manager: see ``allocator_model.py``.

Every function is pinned by tests in ``tests/test_oracle_pins.py`` against
values printed on the pages, closed forms, a library routine (torch's
scaled_dot_product_attention in float64 on contiguous K/V) and hand-made
fixtures under ``tests/golden/``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

from .allocator_model import AllocatorError, BlockPoolModel, OutOfBlocks, UnknownSequence  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pagedattn_oracle.c")
_LIB = os.path.join(_HERE, "_build", "liboracle.so")

OR_F32, OR_F16, OR_BF16, OR_F64, OR_E4M3 = 0, 1, 2, 3, 4
_CODES = {"f32": OR_F32, "f16": OR_F16, "bf16": OR_BF16, "f64": OR_F64, "e4m3": OR_E4M3}
_NP_STORAGE = {"f32": np.float32, "f16": np.float16, "bf16": np.uint16, "f64": np.float64,
               "e4m3": np.uint8}

_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc into oracle/_build/liboracle.so."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        vp, i32p, i64, c_int = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        lib.oracle_kv_write.argtypes = [vp, vp, i32p, i64, vp, vp, i64, c_int, i64, c_int]
        lib.oracle_kv_write.restype = i64
        lib.oracle_copy_blocks.argtypes = [vp, vp, i32p, i64, i64, i64, c_int]
        lib.oracle_copy_blocks.restype = i64
        lib.oracle_paged_attention.argtypes = [vp, vp, c_int, vp, vp, c_int, i32p, c_int, i32p,
                                               c_int, c_int, c_int, c_int, c_int, i64,
                                               ctypes.c_double, c_int]
        lib.oracle_paged_attention.restype = c_int
        lib.oracle_attention_weights.argtypes = [vp, vp, vp, c_int, vp, vp, c_int, i32p, c_int,
                                                 i32p, c_int, c_int, c_int, c_int, c_int, i64,
                                                 ctypes.c_double, c_int, c_int]
        lib.oracle_attention_weights.restype = c_int
        lib.oracle_paged_prefill.argtypes = [vp, vp, vp, vp, c_int, i32p, c_int, i32p, i32p, c_int, c_int,
                                             c_int, c_int, c_int, i64, ctypes.c_double, c_int]
        lib.oracle_paged_prefill.restype = c_int
        lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_to_double.restype = ctypes.c_double
        lib.oracle_e4m3_from_float.argtypes = [ctypes.c_float]
        lib.oracle_e4m3_from_float.restype = ctypes.c_uint8
        lib.oracle_kv_write_fp8.argtypes = [vp, vp, c_int, i32p, i64, vp, vp, i64, c_int, i64,
                                            ctypes.c_float, ctypes.c_float]
        lib.oracle_kv_write_fp8.restype = i64
        lib.oracle_paged_attention_fp8.argtypes = [vp, vp, c_int, vp, vp, i32p, c_int, i32p, c_int, c_int,
                                                   c_int, c_int, c_int, i64, ctypes.c_double, ctypes.c_float,
                                                   ctypes.c_float, c_int]
        lib.oracle_paged_attention_fp8.restype = c_int
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _check_storage(a: np.ndarray, dtype: str) -> np.ndarray:
    want = _NP_STORAGE[dtype]
    if a.dtype != want:
        raise TypeError(f"{dtype} data must be stored as {np.dtype(want)}, got {a.dtype}")
    return np.ascontiguousarray(a)


def kv_write(k, v, slot_mapping, key_cache, value_cache, dtype: str) -> int:
    """In place: key_cache/value_cache [NB, bs, Hk, D] get rows k/v [T, Hk, D].

    Returns the number of invalid (non -1, out of range) slots skipped."""
    lib = _load()
    k = _check_storage(k, dtype)
    v = _check_storage(v, dtype)
    for c in (key_cache, value_cache):
        _check_storage(c, dtype)
        if not c.flags.c_contiguous:
            raise ValueError("caches must be C-contiguous")
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int32)
    nb, bs = key_cache.shape[0], key_cache.shape[1]
    row = int(np.prod(key_cache.shape[2:]))
    rc = lib.oracle_kv_write(_ptr(k), _ptr(v), _ptr(sm), sm.shape[0], _ptr(key_cache),
                             _ptr(value_cache), nb, bs, row, _CODES[dtype])
    if rc < 0:
        raise ValueError(f"oracle_kv_write: {rc}")
    return int(rc)


def copy_blocks(key_cache, value_cache, pairs, dtype: str) -> int:
    """In place: for each (src, dst) row of pairs, block dst := block src (K and V)."""
    lib = _load()
    for c in (key_cache, value_cache):
        _check_storage(c, dtype)
        if not c.flags.c_contiguous:
            raise ValueError("caches must be C-contiguous")
    p = np.ascontiguousarray(np.asarray(pairs, dtype=np.int32).reshape(-1, 2))
    nb = key_cache.shape[0]
    be = int(np.prod(key_cache.shape[1:]))
    rc = lib.oracle_copy_blocks(_ptr(key_cache), _ptr(value_cache), _ptr(p), p.shape[0], nb, be,
                                _CODES[dtype])
    if rc < 0:
        raise ValueError(f"oracle_copy_blocks: {rc}")
    return int(rc)


def paged_attention(q, key_cache, value_cache, block_tables, context_lens, scale: float,
                    dtype: str, q_dtype: str | None = None, num_threads: int = 1) -> np.ndarray:
    """float64 out [B, H, D] of single-query decode attention over a paged cache."""
    lib = _load()
    q_dtype = q_dtype or dtype
    q = _check_storage(q, q_dtype)
    kc = _check_storage(key_cache, dtype)
    vc = _check_storage(value_cache, dtype)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    B, H, D = q.shape
    nb, bs, hk, d2 = kc.shape
    if d2 != D or vc.shape != kc.shape or bt.shape[0] != B or cl.shape[0] != B:
        raise ValueError("shape mismatch")
    out = np.zeros((B, H, D), dtype=np.float64)
    rc = lib.oracle_paged_attention(_ptr(out), _ptr(q), _CODES[q_dtype], _ptr(kc), _ptr(vc),
                                    _CODES[dtype], _ptr(bt), bt.shape[1] if bt.ndim == 2 else 0,
                                    _ptr(cl), B, H, hk, D, bs, nb, float(scale), int(num_threads))
    if rc != 0:
        raise ValueError(f"oracle_paged_attention: {rc}")
    return out


def attention_weights(q, key_cache, value_cache, block_tables, context_lens, scale: float,
                      dtype: str, b: int, h: int, q_dtype: str | None = None):
    """(weights [ctx_b], out [B, H, D]) with the softmax weights of (b, h)."""
    lib = _load()
    q_dtype = q_dtype or dtype
    q = _check_storage(q, q_dtype)
    kc = _check_storage(key_cache, dtype)
    vc = _check_storage(value_cache, dtype)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    B, H, D = q.shape
    nb, bs, hk, _ = kc.shape
    w = np.zeros(max(int(cl[b]), 1), dtype=np.float64)
    out = np.zeros((B, H, D), dtype=np.float64)
    rc = lib.oracle_attention_weights(_ptr(w), _ptr(out), _ptr(q), _CODES[q_dtype], _ptr(kc),
                                      _ptr(vc), _CODES[dtype], _ptr(bt), bt.shape[1], _ptr(cl),
                                      B, H, hk, D, bs, nb, float(scale), int(b), int(h))
    if rc != 0:
        raise ValueError(f"oracle_attention_weights: {rc}")
    return w[: int(cl[b])], out


def paged_prefill(q, key_cache, value_cache, block_tables, context_lens, query_start_loc, scale: float,
                  dtype: str, num_threads: int = 1) -> np.ndarray:
    """float64 out [total_q, H, D] of causal chunked-prefill attention over a paged cache."""
    lib = _load()
    q = _check_storage(q, dtype)
    kc = _check_storage(key_cache, dtype)
    vc = _check_storage(value_cache, dtype)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    qs = np.ascontiguousarray(query_start_loc, dtype=np.int32)
    T, H, D = q.shape
    nb, bs, hk, d2 = kc.shape
    B = cl.shape[0]
    if d2 != D or vc.shape != kc.shape or bt.shape[0] != B or qs.shape[0] != B + 1 or qs[-1] != T:
        raise ValueError("shape mismatch")
    out = np.zeros((T, H, D), dtype=np.float64)
    rc = lib.oracle_paged_prefill(_ptr(out), _ptr(q), _ptr(kc), _ptr(vc), _CODES[dtype], _ptr(bt), bt.shape[1],
                                  _ptr(cl), _ptr(qs), B, H, hk, D, bs, nb, float(scale), int(num_threads))
    if rc != 0:
        raise ValueError(f"oracle_paged_prefill: {rc}")
    return out


def e4m3_to_float64(codes) -> np.ndarray:
    """float64 values of E4M3 codes (NaN for the two NaN codes)."""
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8)
    flat = [lib.oracle_e4m3_to_double(int(x)) for x in c.reshape(-1)]
    return np.asarray(flat, dtype=np.float64).reshape(c.shape)


def e4m3_from_float32(x) -> np.ndarray:
    """Nearest E4M3 codes (ties to even, saturating at 448) of float32 values."""
    lib = _load()
    a = np.asarray(x, dtype=np.float32)
    flat = [lib.oracle_e4m3_from_float(float(v)) for v in a.reshape(-1)]
    return np.asarray(flat, dtype=np.uint8).reshape(a.shape)


def kv_write_fp8(k, v, slot_mapping, key_cache, value_cache, k_scale: float, v_scale: float,
                 src_dtype: str) -> int:
    """In place: uint8 E4M3 caches [NB, bs, Hk, D] get rows k/v [T, Hk, D] quantised
    as code(x / scale) in float32. Returns the number of invalid slots skipped."""
    lib = _load()
    k = _check_storage(k, src_dtype)
    v = _check_storage(v, src_dtype)
    for c in (key_cache, value_cache):
        _check_storage(c, "e4m3")
        if not c.flags.c_contiguous:
            raise ValueError("caches must be C-contiguous")
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int32)
    nb, bs = key_cache.shape[0], key_cache.shape[1]
    row = int(np.prod(key_cache.shape[2:]))
    rc = lib.oracle_kv_write_fp8(_ptr(k), _ptr(v), _CODES[src_dtype], _ptr(sm), sm.shape[0], _ptr(key_cache),
                                 _ptr(value_cache), nb, bs, row, float(k_scale), float(v_scale))
    if rc < 0:
        raise ValueError(f"oracle_kv_write_fp8: {rc}")
    return int(rc)


def paged_attention_fp8(q, key_cache, value_cache, block_tables, context_lens, scale: float,
                        k_scale: float, v_scale: float, q_dtype: str, num_threads: int = 1) -> np.ndarray:
    """float64 out [B, H, D] of decode attention over uint8 E4M3 caches, element =
    decoded(code) * k_scale (K) or * v_scale (V)."""
    lib = _load()
    q = _check_storage(q, q_dtype)
    kc = _check_storage(key_cache, "e4m3")
    vc = _check_storage(value_cache, "e4m3")
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    B, H, D = q.shape
    nb, bs, hk, d2 = kc.shape
    if d2 != D or vc.shape != kc.shape or bt.shape[0] != B or cl.shape[0] != B:
        raise ValueError("shape mismatch")
    out = np.zeros((B, H, D), dtype=np.float64)
    rc = lib.oracle_paged_attention_fp8(_ptr(out), _ptr(q), _CODES[q_dtype], _ptr(kc), _ptr(vc), _ptr(bt),
                                        bt.shape[1], _ptr(cl), B, H, hk, D, bs, nb, float(scale),
                                        float(k_scale), float(v_scale), int(num_threads))
    if rc != 0:
        raise ValueError(f"oracle_paged_attention_fp8: {rc}")
    return out


def num_host_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1
