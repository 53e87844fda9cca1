"""Paged KV cache decode path for GB300 (sm_103a): Python binding of libpagedattn.

A thin ctypes layer over the C ABI in ``include/pagedattn.h``: it reads shapes,
dtypes and pointers off torch tensors and calls the library. Every step of the
computation runs in the library's CUDA kernels; there is no fallback. Importing
this package fails when ``_build/libpagedattn.so`` has not been built (run
``python paged_kv_cache_261_gb300/build.py``).

Entry points (same names as the C ABI, without the ``pa_`` prefix):
  paged_kv_write(k, v, slot_mapping, key_cache, value_cache)
  paged_attention_decode(out, q, key_cache, value_cache, block_tables,
                         context_lens, scale, block_size, num_kv_heads)
  paged_attention_prefill(out, q, key_cache, value_cache, block_tables,
                          context_lens, query_start_loc, scale, max_query_len)
  paged_attention_decode_shared(out, q, key_cache, value_cache, block_tables,
                                context_lens, prefix_lens, group_members, scale)
  prefix_groups(block_tables, context_lens, block_size)   (host)
  copy_blocks(key_cache, value_cache, src_dst_pairs)
  paged_kv_write_fp8(k, v, slot_mapping, key_cache, value_cache, k_scale, v_scale)
  paged_attention_decode_fp8(out, q, key_cache, value_cache, block_tables,
                             context_lens, scale, k_scale, v_scale)
  get_device_error()
  BlockAllocator: the host block manager (free list, reference counts, fork,
  copy-on-write, block-table and slot-mapping export).
Cache layout: [num_blocks, block_size, num_kv_heads, head_dim]. The _fp8 calls
take 8-bit caches (torch.uint8 or torch.float8_e4m3fn) holding OCP FP8 E4M3
codes with one float32 scale for K and one for V.
"""
from __future__ import annotations

import contextlib
import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libpagedattn.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"libpagedattn.so is missing at {LIB_PATH}; build it with "
        "`python paged_kv_cache_261_gb300/build.py` (needs nvcc)")

_lib = ctypes.CDLL(LIB_PATH)

PA_OK = 0
PA_ERR_INVALID_ARG = -1
PA_ERR_UNSUPPORTED = -2
PA_ERR_OUT_OF_BLOCKS = -3
PA_ERR_CUDA = -4
PA_ERR_DEVICE_INDEX = -5
PA_ERR_UNKNOWN_SEQ = -6
PA_ERR_WORKSPACE = -7
PA_ERR_EXISTS = -8

PA_DTYPE_F32, PA_DTYPE_F16, PA_DTYPE_BF16, PA_DTYPE_E4M3 = 0, 1, 2, 3

PA_DEVERR_SLOT = 0x1
PA_DEVERR_BLOCK_ID = 0x2
PA_DEVERR_CONTEXT = 0x4
PA_DEVERR_COPY_PAIR = 0x8
PA_DEVERR_WAIT = 0x10

_vp, _i32, _i64, _sz, _f = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float


def _decl(name, args, res=ctypes.c_int):
    fn = getattr(_lib, name)
    fn.argtypes = args
    fn.restype = res
    return fn


_decl("pa_status_string", [_i32], ctypes.c_char_p)
_decl("pa_version", [])
_decl("pa_paged_kv_write", [_vp, _vp, _vp, _i64, _vp, _vp, _i64, _i32, _i32, _i32, _i32, _vp])
_decl("pa_decode_workspace_bytes", [_i32, _i32, _i32, _i32, _i32], _sz)
_decl("pa_decode_partition_size", [_i32, _i32, _i32])
_decl("pa_decode_shared_partition_size", [_i32, _i32, _i32, _i32, _i32, _i32])
_decl("pa_paged_attention_decode", [_vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _i32,
                                    _i64, _f, _i32, _i32, _vp, _sz, _i32, _vp])
_decl("pa_paged_attention_decode_append", [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32,
                                           _i32, _i32, _i64, _f, _i32, _i32, _vp, _sz, _i32, _vp])
_decl("pa_copy_blocks", [_vp, _vp, _vp, _i64, _i64, _i32, _i32, _i32, _i32, _vp])
_decl("pa_get_device_error", [_vp, ctypes.POINTER(ctypes.c_uint32)])
_decl("pa_check_bounded_wait", [_i64, _vp, _vp])
_decl("pa_decode_shared_workspace_bytes", [_i32, _i32, _i32, _i32, _i32], _sz)
_decl("pa_paged_attention_decode_shared", [_vp, _vp, _vp, _vp, _vp, _i32, _vp, _vp, _vp, _i32, _i32, _i32, _i32,
                                           _i32, _i32, _i32, _i32, _i64, _f, _i32, _i32, _vp, _sz, _i32, _vp])
_decl("pa_prefix_groups", [_vp, _vp, _i32, _i32, _i32, _i32, _i32, _vp, _vp, ctypes.POINTER(ctypes.c_int)])
_decl("pa_paged_kv_write_fp8", [_vp, _vp, _vp, _i64, _vp, _vp, _i64, _i32, _i32, _i32, _f, _f, _i32, _vp])
_decl("pa_paged_attention_decode_fp8", [_vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _i32,
                                        _i64, _f, _f, _f, _i32, _i32, _vp, _sz, _i32, _vp])
_decl("pa_paged_attention_decode_fp8_append", [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32,
                                               _i32, _i32, _i32, _i64, _f, _f, _f, _i32, _i32, _vp, _sz, _i32, _vp])
_decl("pa_paged_attention_prefill", [_vp, _vp, _vp, _vp, _vp, _i32, _vp, _vp, _i32, _i64, _i32, _i32, _i32, _i32,
                                     _i32, _i64, _f, _i32, _vp])


class PagedAttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


def status_string(status: int) -> str:
    return _lib.pa_status_string(int(status)).decode()


def version() -> int:
    return int(_lib.pa_version())


def lib() -> ctypes.CDLL:
    """The loaded C library (raw ABI access)."""
    return _lib


def _check(rc: int, what: str) -> None:
    if rc != PA_OK:
        raise PagedAttnError(rc, what)


# ---------------------------------------------------------------------------
# torch glue
# ---------------------------------------------------------------------------

def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    m = {torch.float32: PA_DTYPE_F32, torch.float16: PA_DTYPE_F16, torch.bfloat16: PA_DTYPE_BF16}
    if t.dtype not in m:
        raise TypeError(f"unsupported dtype {t.dtype}")
    return m[t.dtype]


def _is_fp8_cache(t) -> bool:
    torch = _torch()
    return t.dtype == torch.uint8 or t.dtype == getattr(torch, "float8_e4m3fn", None)


def _storage_code(t) -> int:
    """Element code of a cache tensor, 8-bit caches included."""
    return PA_DTYPE_E4M3 if _is_fp8_cache(t) else _dtype_code(t)


_SAME_DEVICE = contextlib.nullcontext()


def _on(device):
    """The tensors' device made current for a library call: the library launches on,
    and sizes its grids for, the current device (no switch when it already is)."""
    torch = _torch()
    idx = device.index
    if idx is None or idx == torch.cuda.current_device():
        return _SAME_DEVICE
    return torch.cuda.device(idx)


def _stream_ptr(stream, device) -> int:
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return int(stream.cuda_stream)


def _cuda(t, name: str, dtype=None, device=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    return t


def paged_kv_write(k, v, slot_mapping, key_cache, value_cache, stream=None) -> None:
    """Scatter k/v [T, Hk, D] into key_cache/value_cache [NB, bs, Hk, D] at slot_mapping[T]."""
    torch = _torch()
    dev = key_cache.device
    _cuda(key_cache, "key_cache")
    _cuda(value_cache, "value_cache", key_cache.dtype, dev)
    _cuda(k, "k", key_cache.dtype, dev)
    _cuda(v, "v", key_cache.dtype, dev)
    _cuda(slot_mapping, "slot_mapping", torch.int32, dev)
    nb, bs, hk, d = key_cache.shape
    if value_cache.shape != key_cache.shape:
        raise ValueError("value_cache shape differs from key_cache")
    T = slot_mapping.shape[0]
    if tuple(k.shape) != (T, hk, d) or tuple(v.shape) != (T, hk, d):
        raise ValueError(f"k/v must be [{T}, {hk}, {d}]")
    with _on(dev):
        rc = _lib.pa_paged_kv_write(k.data_ptr(), v.data_ptr(), slot_mapping.data_ptr(), T,
                                    key_cache.data_ptr(), value_cache.data_ptr(), nb, bs, hk, d,
                                    _dtype_code(key_cache), _stream_ptr(stream, dev))
    _check(rc, "pa_paged_kv_write")


def decode_workspace_bytes(num_seqs: int, num_heads: int, head_dim: int, max_context_len: int,
                           partition_size: int = 0) -> int:
    return int(_lib.pa_decode_workspace_bytes(num_seqs, num_heads, head_dim, max_context_len,
                                              partition_size))


_ws_cache: dict = {}


def decode_partition_size(num_seqs: int, max_context_len: int, partition_size: int = 0) -> int:
    """Partition size (tokens) a decode call uses: partition_size, or the automatic choice for 0."""
    return int(_lib.pa_decode_partition_size(num_seqs, max_context_len, partition_size))


def decode_shared_partition_size(num_seqs: int, num_groups: int, num_kv_heads: int, max_prefix_len: int,
                                 max_context_len: int, partition_size: int = 0) -> int:
    """Partition size (tokens) a sharing-aware decode call uses: partition_size, or the automatic choice for 0."""
    return int(_lib.pa_decode_shared_partition_size(num_seqs, num_groups, num_kv_heads, max_prefix_len,
                                                    max_context_len, partition_size))


def _workspace(device, stream_ptr: int, nbytes: int):
    """Cached per (device, stream) workspace buffer, grown on demand."""
    torch = _torch()
    key = (device, stream_ptr)
    buf = _ws_cache.get(key)
    if buf is None or buf.numel() < nbytes:
        buf = torch.empty(max(nbytes, 1 << 20), dtype=torch.uint8, device=device)
        _ws_cache[key] = buf
    return buf


def paged_attention_decode(out, q, key_cache, value_cache, block_tables, context_lens, scale: float,
                           block_size: int | None = None, num_kv_heads: int | None = None,
                           max_context_len: int = 0, partition_size: int = 0, workspace=None,
                           stream=None) -> None:
    """out[b, h] = softmax(scale * q[b, h] . K_b^T) V_b over the paged cache.

    q, out [B, H, D]; caches [NB, bs, Hk, D]; block_tables int32 [B, MB];
    context_lens int32 [B]. max_context_len: host upper bound on the lengths
    (0 = MB * bs). workspace: optional uint8 CUDA tensor; by default a cached
    per-stream buffer is used."""
    torch = _torch()
    dev = key_cache.device
    _cuda(key_cache, "key_cache")
    _cuda(value_cache, "value_cache", key_cache.dtype, dev)
    _cuda(q, "q", key_cache.dtype, dev)
    _cuda(out, "out", key_cache.dtype, dev)
    _cuda(block_tables, "block_tables", torch.int32, dev)
    _cuda(context_lens, "context_lens", torch.int32, dev)
    nb, bs, hk, d = key_cache.shape
    if block_size is not None and block_size != bs:
        raise ValueError(f"block_size {block_size} != cache block size {bs}")
    if num_kv_heads is not None and num_kv_heads != hk:
        raise ValueError(f"num_kv_heads {num_kv_heads} != cache kv heads {hk}")
    if value_cache.shape != key_cache.shape:
        raise ValueError("value_cache shape differs from key_cache")
    B, H, D = q.shape
    if D != d or tuple(out.shape) != (B, H, D):
        raise ValueError("q/out must be [B, H, head_dim]")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or tuple(context_lens.shape) != (B,):
        raise ValueError("block_tables must be [B, MB] and context_lens [B]")
    mb = block_tables.shape[1]
    sp = _stream_ptr(stream, dev)
    need = decode_workspace_bytes(B, H, D, max_context_len or mb * bs, partition_size)
    ws_ptr, ws_bytes = None, 0
    if need:
        if workspace is None:
            workspace = _workspace(dev, sp, need)
        _cuda(workspace, "workspace", torch.uint8, dev)
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel()
    with _on(dev):
        rc = _lib.pa_paged_attention_decode(out.data_ptr(), q.data_ptr(), key_cache.data_ptr(),
                                            value_cache.data_ptr(), block_tables.data_ptr(), mb,
                                            context_lens.data_ptr(), B, H, hk, D, bs, nb, float(scale),
                                            int(max_context_len), int(partition_size), ws_ptr, ws_bytes,
                                            _dtype_code(key_cache), sp)
    _check(rc, "pa_paged_attention_decode")


def paged_attention_decode_append(out, q, k_new, v_new, slot_mapping, key_cache, value_cache, block_tables,
                                  context_lens, scale: float, max_context_len: int = 0, partition_size: int = 0,
                                  workspace=None, stream=None) -> None:
    """One decode step: each sequence's new token (k_new, v_new [B, Hk, D]) goes to
    slot_mapping[b] -- the slot of position context_lens[b] - 1, or -1 -- and
    then paged_attention_decode. The same result and caches as paged_kv_write
    followed by paged_attention_decode; the tensor-core decode writes the tokens
    itself instead of a separate launch."""
    torch = _torch()
    dev = key_cache.device
    _cuda(key_cache, "key_cache")
    _cuda(value_cache, "value_cache", key_cache.dtype, dev)
    _cuda(q, "q", key_cache.dtype, dev)
    _cuda(out, "out", key_cache.dtype, dev)
    _cuda(k_new, "k_new", key_cache.dtype, dev)
    _cuda(v_new, "v_new", key_cache.dtype, dev)
    _cuda(slot_mapping, "slot_mapping", torch.int32, dev)
    _cuda(block_tables, "block_tables", torch.int32, dev)
    _cuda(context_lens, "context_lens", torch.int32, dev)
    nb, bs, hk, d = key_cache.shape
    if value_cache.shape != key_cache.shape:
        raise ValueError("value_cache shape differs from key_cache")
    B, H, D = q.shape
    if D != d or tuple(out.shape) != (B, H, D):
        raise ValueError("q/out must be [B, H, head_dim]")
    if tuple(k_new.shape) != (B, hk, D) or tuple(v_new.shape) != (B, hk, D) or tuple(slot_mapping.shape) != (B,):
        raise ValueError("k_new/v_new must be [B, num_kv_heads, head_dim] and slot_mapping [B]")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or tuple(context_lens.shape) != (B,):
        raise ValueError("block_tables must be [B, MB] and context_lens [B]")
    mb = block_tables.shape[1]
    sp = _stream_ptr(stream, dev)
    need = decode_workspace_bytes(B, H, D, max_context_len or mb * bs, partition_size)
    ws_ptr, ws_bytes = None, 0
    if need:
        if workspace is None:
            workspace = _workspace(dev, sp, need)
        _cuda(workspace, "workspace", torch.uint8, dev)
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel()
    with _on(dev):
        rc = _lib.pa_paged_attention_decode_append(out.data_ptr(), q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(),
                                                   slot_mapping.data_ptr(), key_cache.data_ptr(),
                                                   value_cache.data_ptr(), block_tables.data_ptr(), mb,
                                                   context_lens.data_ptr(), B, H, hk, D, bs, nb, float(scale),
                                                   int(max_context_len), int(partition_size), ws_ptr, ws_bytes,
                                                   _dtype_code(key_cache), sp)
    _check(rc, "pa_paged_attention_decode_append")


def paged_attention_prefill(out, q, key_cache, value_cache, block_tables, context_lens, query_start_loc,
                            scale: float, max_query_len: int, stream=None) -> None:
    """Causal chunked-prefill attention: q, out [T, H, D] packed by query_start_loc [B + 1];
    row i of sequence b sits at position context_lens[b] - q_len_b + i and sees
    positions up to its own. max_query_len: host bound on every chunk length."""
    torch = _torch()
    dev = key_cache.device
    _cuda(key_cache, "key_cache")
    _cuda(value_cache, "value_cache", key_cache.dtype, dev)
    _cuda(q, "q", key_cache.dtype, dev)
    _cuda(out, "out", key_cache.dtype, dev)
    _cuda(block_tables, "block_tables", torch.int32, dev)
    _cuda(context_lens, "context_lens", torch.int32, dev)
    _cuda(query_start_loc, "query_start_loc", torch.int32, dev)
    nb, bs, hk, d = key_cache.shape
    if value_cache.shape != key_cache.shape:
        raise ValueError("value_cache shape differs from key_cache")
    T, H, D = q.shape
    B = context_lens.shape[0]
    if D != d or tuple(out.shape) != (T, H, D):
        raise ValueError("q/out must be [T, H, head_dim]")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or tuple(query_start_loc.shape) != (B + 1,):
        raise ValueError("block_tables must be [B, MB] and query_start_loc [B + 1]")
    with _on(dev):
        rc = _lib.pa_paged_attention_prefill(out.data_ptr(), q.data_ptr(), key_cache.data_ptr(),
                                             value_cache.data_ptr(), block_tables.data_ptr(), block_tables.shape[1],
                                             context_lens.data_ptr(), query_start_loc.data_ptr(), B, T,
                                             int(max_query_len), H, hk, D, bs, nb, float(scale),
                                             _dtype_code(key_cache), _stream_ptr(stream, dev))
    _check(rc, "pa_paged_attention_prefill")


def prefix_groups(block_tables, context_lens, block_size: int, max_members: int = 8,
                  min_shared_blocks: int = 1):
    """Host: groups of sequences whose tables start with the same full blocks.

    Returns (prefix_lens int32 [B], group_members int32 [num_groups, max_members])."""
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    B = cl.shape[0]
    pl = np.zeros(max(B, 1), np.int32)
    gm = np.full((max(B, 1), max_members), -1, np.int32)
    ng = ctypes.c_int(0)
    _check(_lib.pa_prefix_groups(bt.ctypes.data, cl.ctypes.data, B, bt.shape[1] if bt.ndim == 2 else 0,
                                 block_size, max_members, min_shared_blocks, pl.ctypes.data, gm.ctypes.data,
                                 ctypes.byref(ng)), "pa_prefix_groups")
    return pl[:B].copy(), gm[: ng.value].copy()


def decode_shared_workspace_bytes(num_seqs: int, num_heads: int, head_dim: int, max_context_len: int,
                                  partition_size: int = 0) -> int:
    return int(_lib.pa_decode_shared_workspace_bytes(num_seqs, num_heads, head_dim, max_context_len,
                                                     partition_size))


def paged_attention_decode_shared(out, q, key_cache, value_cache, block_tables, context_lens, prefix_lens,
                                  group_members, scale: float, max_context_len: int = 0,
                                  max_prefix_len: int | None = None, partition_size: int = 0, workspace=None,
                                  stream=None) -> None:
    """Decode that reads each group's shared prefix once for all its members.

    prefix_lens int32 [B] and group_members int32 [G, M] as from prefix_groups
    (device tensors). Same result as paged_attention_decode."""
    torch = _torch()
    dev = key_cache.device
    _cuda(key_cache, "key_cache")
    _cuda(value_cache, "value_cache", key_cache.dtype, dev)
    _cuda(q, "q", key_cache.dtype, dev)
    _cuda(out, "out", key_cache.dtype, dev)
    for t, n in ((block_tables, "block_tables"), (context_lens, "context_lens"), (prefix_lens, "prefix_lens"),
                 (group_members, "group_members")):
        _cuda(t, n, torch.int32, dev)
    nb, bs, hk, d = key_cache.shape
    B, H, D = q.shape
    if D != d or tuple(out.shape) != (B, H, D) or block_tables.shape[0] != B or prefix_lens.shape[0] != B:
        raise ValueError("shape mismatch")
    if group_members.dim() != 2:
        raise ValueError("group_members must be [num_groups, max_members]")
    mb = block_tables.shape[1]
    mctx = max_context_len or mb * bs
    mpre = mctx if max_prefix_len is None else int(max_prefix_len)
    sp = _stream_ptr(stream, dev)
    need = decode_shared_workspace_bytes(B, H, D, mctx, partition_size)
    if workspace is None:
        workspace = _workspace(dev, sp, need)
    _cuda(workspace, "workspace", torch.uint8, dev)
    ng, mm = group_members.shape
    with _on(dev):
        rc = _lib.pa_paged_attention_decode_shared(out.data_ptr(), q.data_ptr(), key_cache.data_ptr(),
                                                   value_cache.data_ptr(), block_tables.data_ptr(), mb,
                                                   context_lens.data_ptr(), prefix_lens.data_ptr(),
                                                   group_members.data_ptr() if ng else None, ng, max(mm, 1), mpre,
                                                   B, H, hk, D, bs, nb, float(scale), int(max_context_len),
                                                   int(partition_size), workspace.data_ptr(), workspace.numel(),
                                                   _dtype_code(key_cache), sp)
    _check(rc, "pa_paged_attention_decode_shared")


def copy_blocks(key_cache, value_cache, src_dst_pairs, stream=None) -> None:
    """key_cache[dst] = key_cache[src] (and V) for each row (src, dst) of src_dst_pairs [P, 2]."""
    torch = _torch()
    dev = key_cache.device
    _cuda(key_cache, "key_cache")
    _cuda(value_cache, "value_cache", key_cache.dtype, dev)
    _cuda(src_dst_pairs, "src_dst_pairs", torch.int32, dev)
    if src_dst_pairs.dim() != 2 or src_dst_pairs.shape[1] != 2:
        raise ValueError("src_dst_pairs must be [P, 2]")
    nb, bs, hk, d = key_cache.shape
    with _on(dev):
        rc = _lib.pa_copy_blocks(key_cache.data_ptr(), value_cache.data_ptr(), src_dst_pairs.data_ptr(),
                                 src_dst_pairs.shape[0], nb, bs, hk, d, _storage_code(key_cache),
                                 _stream_ptr(stream, dev))
    _check(rc, "pa_copy_blocks")


def _fp8_caches(key_cache, value_cache, dev):
    _cuda(key_cache, "key_cache")
    _cuda(value_cache, "value_cache", key_cache.dtype, dev)
    if not _is_fp8_cache(key_cache):
        raise TypeError(f"8-bit caches must be torch.uint8 or torch.float8_e4m3fn, got {key_cache.dtype}")
    if value_cache.shape != key_cache.shape:
        raise ValueError("value_cache shape differs from key_cache")
    return key_cache.shape


def paged_kv_write_fp8(k, v, slot_mapping, key_cache, value_cache, k_scale: float, v_scale: float,
                       stream=None) -> None:
    """Scatter k/v [T, Hk, D] (fp32/fp16/bf16) into 8-bit caches [NB, bs, Hk, D] as the
    E4M3 codes of k / k_scale and v / v_scale, at slot_mapping[T]."""
    torch = _torch()
    dev = key_cache.device
    nb, bs, hk, d = _fp8_caches(key_cache, value_cache, dev)
    _cuda(k, "k", None, dev)
    _cuda(v, "v", k.dtype, dev)
    _cuda(slot_mapping, "slot_mapping", torch.int32, dev)
    T = slot_mapping.shape[0]
    if tuple(k.shape) != (T, hk, d) or tuple(v.shape) != (T, hk, d):
        raise ValueError(f"k/v must be [{T}, {hk}, {d}]")
    with _on(dev):
        rc = _lib.pa_paged_kv_write_fp8(k.data_ptr(), v.data_ptr(), slot_mapping.data_ptr(), T, key_cache.data_ptr(),
                                        value_cache.data_ptr(), nb, bs, hk, d, float(k_scale), float(v_scale),
                                        _dtype_code(k), _stream_ptr(stream, dev))
    _check(rc, "pa_paged_kv_write_fp8")


def paged_attention_decode_fp8(out, q, key_cache, value_cache, block_tables, context_lens, scale: float,
                               k_scale: float, v_scale: float, max_context_len: int = 0,
                               partition_size: int = 0, workspace=None, stream=None) -> None:
    """Decode attention over 8-bit caches: K = code * k_scale, V = code * v_scale.

    q, out [B, H, 128] bf16 or fp16; other arguments as paged_attention_decode."""
    torch = _torch()
    dev = key_cache.device
    nb, bs, hk, d = _fp8_caches(key_cache, value_cache, dev)
    _cuda(q, "q", None, dev)
    _cuda(out, "out", q.dtype, dev)
    _cuda(block_tables, "block_tables", torch.int32, dev)
    _cuda(context_lens, "context_lens", torch.int32, dev)
    B, H, D = q.shape
    if D != d or tuple(out.shape) != (B, H, D):
        raise ValueError("q/out must be [B, H, head_dim]")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or tuple(context_lens.shape) != (B,):
        raise ValueError("block_tables must be [B, MB] and context_lens [B]")
    mb = block_tables.shape[1]
    sp = _stream_ptr(stream, dev)
    need = decode_workspace_bytes(B, H, D, max_context_len or mb * bs, partition_size)
    ws_ptr, ws_bytes = None, 0
    if need:
        if workspace is None:
            workspace = _workspace(dev, sp, need)
        _cuda(workspace, "workspace", torch.uint8, dev)
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel()
    with _on(dev):
        rc = _lib.pa_paged_attention_decode_fp8(out.data_ptr(), q.data_ptr(), key_cache.data_ptr(),
                                                value_cache.data_ptr(), block_tables.data_ptr(), mb,
                                                context_lens.data_ptr(), B, H, hk, D, bs, nb, float(scale),
                                                float(k_scale), float(v_scale), int(max_context_len),
                                                int(partition_size), ws_ptr, ws_bytes, _dtype_code(q), sp)
    _check(rc, "pa_paged_attention_decode_fp8")


def paged_attention_decode_fp8_append(out, q, k_new, v_new, slot_mapping, key_cache, value_cache, block_tables,
                                      context_lens, scale: float, k_scale: float, v_scale: float,
                                      max_context_len: int = 0, partition_size: int = 0, workspace=None,
                                      stream=None) -> None:
    """One decode step over 8-bit caches: each sequence's new token (k_new, v_new
    [B, Hk, D] in q's dtype) is quantised into slot_mapping[b] -- the slot of
    position context_lens[b] - 1, or -1 -- by the decode kernel itself, then the
    decode runs. The same result and caches as paged_kv_write_fp8 followed by
    paged_attention_decode_fp8."""
    torch = _torch()
    dev = key_cache.device
    nb, bs, hk, d = _fp8_caches(key_cache, value_cache, dev)
    _cuda(q, "q", None, dev)
    _cuda(out, "out", q.dtype, dev)
    _cuda(k_new, "k_new", q.dtype, dev)
    _cuda(v_new, "v_new", q.dtype, dev)
    _cuda(slot_mapping, "slot_mapping", torch.int32, dev)
    _cuda(block_tables, "block_tables", torch.int32, dev)
    _cuda(context_lens, "context_lens", torch.int32, dev)
    B, H, D = q.shape
    if D != d or tuple(out.shape) != (B, H, D):
        raise ValueError("q/out must be [B, H, head_dim]")
    if tuple(k_new.shape) != (B, hk, D) or tuple(v_new.shape) != (B, hk, D) or tuple(slot_mapping.shape) != (B,):
        raise ValueError("k_new/v_new must be [B, num_kv_heads, head_dim] and slot_mapping [B]")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or tuple(context_lens.shape) != (B,):
        raise ValueError("block_tables must be [B, MB] and context_lens [B]")
    mb = block_tables.shape[1]
    sp = _stream_ptr(stream, dev)
    need = decode_workspace_bytes(B, H, D, max_context_len or mb * bs, partition_size)
    ws_ptr, ws_bytes = None, 0
    if need:
        if workspace is None:
            workspace = _workspace(dev, sp, need)
        _cuda(workspace, "workspace", torch.uint8, dev)
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel()
    with _on(dev):
        rc = _lib.pa_paged_attention_decode_fp8_append(out.data_ptr(), q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(),
                                                       slot_mapping.data_ptr(), key_cache.data_ptr(),
                                                       value_cache.data_ptr(), block_tables.data_ptr(), mb,
                                                       context_lens.data_ptr(), B, H, hk, D, bs, nb, float(scale),
                                                       float(k_scale), float(v_scale), int(max_context_len),
                                                       int(partition_size), ws_ptr, ws_bytes, _dtype_code(q), sp)
    _check(rc, "pa_paged_attention_decode_fp8_append")


def get_device_error(stream=None, device=None) -> int:
    """Synchronise the stream; return and clear the PA_DEVERR_* bits of the device."""
    torch = _torch()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    bits = ctypes.c_uint32(0)
    with _on(dev):
        rc = _lib.pa_get_device_error(_stream_ptr(stream, dev), ctypes.byref(bits))
    if rc not in (PA_OK, PA_ERR_DEVICE_INDEX):
        raise PagedAttnError(rc, "pa_get_device_error")
    return int(bits.value)


def check_bounded_wait(limit_ns: int, report=None, stream=None) -> None:
    """Run the bounded-wait failure check (pa_check_bounded_wait): one warp waits
    limit_ns on an mbarrier phase nothing completes, then sets PA_DEVERR_WAIT.
    report: optional int64 CUDA tensor of 4 elements (see the C header)."""
    torch = _torch()
    dev = torch.device("cuda", torch.cuda.current_device())
    ptr = None
    if report is not None:
        report = _cuda(report, "report", dtype=torch.int64)
        if report.numel() < 4:
            raise ValueError("report needs 4 int64 elements")
        dev = report.device
        ptr = report.data_ptr()
    with _on(dev):
        _check(_lib.pa_check_bounded_wait(int(limit_ns), ptr, _stream_ptr(stream, dev)), "pa_check_bounded_wait")


from .allocator import AllocStats, BlockAllocator  # noqa: E402,F401
