"""The allocation-free decode entry point against the regular one (GPU).

Some callers cannot allocate device memory at all -- their device memory is
owned by a host runtime that forbids libraries to allocate, or an allocation on
their serving path is not acceptable -- and have no buffer to lend either.
pa_paged_attention_decode_noalloc keeps the split-K scratch in a fixed array
inside the library instead. This file checks, through the C ABI, that two calls
in a row on different batches give bit for bit the results of
pa_paged_attention_decode (the same kernels run; only the scratch address
differs, so any stale scratch read would show), and that a request larger than
the built-in scratch is refused.

It sits in a file of its own that pytest collects last, and it builds and loads
everything it needs itself, so it runs alone in a fresh process too.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from __graft_entry__ import build
    build()
    import paged_kv_cache_261_gb300 as pa
    L = pa.lib()
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    L.pa_paged_attention_decode_noalloc.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32,
                                                    i64, ctypes.c_float, i32, i32, i32, vp]
    L.pa_paged_attention_decode_noalloc.restype = i32
    return pa, L


def _inputs(w):
    d = torch.device("cuda", 0)
    dt = workloads.torch_dtype(w.dtype)
    kc = torch.zeros((w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim), dtype=dt, device=d)
    vc = torch.zeros_like(kc)
    w.fill_cache_torch(kc, vc, include_newest=True)
    q = w.q_values(like=kc).to(dt).contiguous()
    bt = torch.as_tensor(w.block_tables, device=d)
    cl = torch.as_tensor(w.context_lens, device=d)
    return q, kc, vc, bt, cl


def _call(L, fn, w, out, q, kc, vc, bt, cl, partition, extra=()):
    stream = torch.cuda.current_stream().cuda_stream
    args = [out.data_ptr(), q.data_ptr(), kc.data_ptr(), vc.data_ptr(), bt.data_ptr(), bt.shape[1],
            cl.data_ptr(), w.num_seqs, w.num_heads, w.num_kv_heads, w.head_dim, w.block_size,
            w.num_blocks, w.scale, int(w.context_lens.max()), partition]
    return fn(*args, *extra, 2, stream)


def test_noalloc_decode_matches_the_regular_entry_point_twice(lib):
    pa, L = lib
    cases = [workloads.llama8b_decode(num_seqs=24), workloads.long_context(num_seqs=2)]
    prepared = []
    for w in cases:
        q, kc, vc, bt, cl = _inputs(w)
        need = pa.decode_workspace_bytes(w.num_seqs, w.num_heads, w.head_dim, int(w.context_lens.max()), 256)
        assert 0 < need <= (32 << 20)
        ws = torch.empty(need, dtype=torch.uint8, device=q.device)
        ref = torch.empty_like(q)
        assert _call(L, L.pa_paged_attention_decode, w, ref, q, kc, vc, bt, cl, 256,
                     extra=(ws.data_ptr(), need)) == 0
        prepared.append((w, q, kc, vc, bt, cl, ref))
    # two calls in a row; the second one finds the first one's leftovers in the scratch
    outs = []
    for w, q, kc, vc, bt, cl, _ in prepared:
        got = torch.full_like(q, float("nan"))
        assert _call(L, L.pa_paged_attention_decode_noalloc, w, got, q, kc, vc, bt, cl, 256) == 0
        outs.append(got)
    torch.cuda.synchronize()
    for (w, *_, ref), got in zip(prepared, outs):
        assert torch.isfinite(got.float()).all()
        assert torch.equal(got, ref), w.name
    assert pa.get_device_error() == 0


def test_noalloc_decode_refuses_requests_beyond_its_scratch(lib):
    pa, L = lib
    w = workloads.long_context(num_seqs=8)            # 8 x 64 heads x 256 partitions needs ~68 MB
    d = torch.device("cuda", 0)
    q = torch.zeros((8, 64, 128), dtype=torch.bfloat16, device=d)
    out = torch.zeros_like(q)
    kc = torch.zeros((16, 16, 8, 128), dtype=torch.bfloat16, device=d)
    bt = torch.zeros((8, 8192), dtype=torch.int32, device=d)
    cl = torch.ones(8, dtype=torch.int32, device=d)
    stream = torch.cuda.current_stream().cuda_stream
    rc = L.pa_paged_attention_decode_noalloc(out.data_ptr(), q.data_ptr(), kc.data_ptr(), kc.data_ptr(),
                                             bt.data_ptr(), 8192, cl.data_ptr(), 8, 64, 8, 128, 16, 16,
                                             0.1, 131072, 512, 2, stream)
    assert rc == pa.PA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert float(out.float().abs().sum()) == 0.0       # nothing was launched
    assert w.num_seqs == 8
