"""GPU parity of chunked-prefill attention against the CPU oracle.

The chunk's K/V go into the cache through paged_kv_write, then every chunk row
attends causally; bf16/fp16 outputs within max 2e-2 / mean 2e-3 of the float64
oracle. Unused cache slots hold NaN, so a read outside the visible keys shows up.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_cases import assert_close, dev, pa_mod, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _free_memory():
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


@pytest.fixture(scope="module")
def pa():
    return pa_mod()


def gpu_prefill(pa, pw, poison=True):
    w = pw.base
    d = dev()
    dt = workloads.torch_dtype(w.dtype)
    shape = (w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim)
    fill = float("nan") if poison else 0.0
    kc = torch.full(shape, fill, dtype=dt, device=d)
    vc = torch.full(shape, fill, dtype=dt, device=d)
    workloads.fill_prior_torch(pw, kc, vc)
    k, v = pw.chunk_kv(like=kc)
    pa.paged_kv_write(k.to(dt).contiguous(), v.to(dt).contiguous(),
                      torch.as_tensor(pw.chunk_slots(), device=d), kc, vc)
    q = pw.q_values(like=kc).to(dt).contiguous()
    out = torch.full_like(q, float("nan"))
    pa.paged_attention_prefill(out, q, kc, vc, torch.as_tensor(w.block_tables, device=d),
                               torch.as_tensor(w.context_lens, device=d),
                               torch.as_tensor(pw.query_start_loc, device=d), w.scale, int(pw.q_lens.max()))
    torch.cuda.synchronize()
    return out, kc, vc


def oracle_prefill(pw):
    w = pw.base
    view = w.compact_host_view(range(w.num_seqs), include_newest=True)
    kc = workloads.to_storage_numpy(view["key_cache"], w.dtype)
    vc = workloads.to_storage_numpy(view["value_cache"], w.dtype)
    q = workloads.to_storage_numpy(pw.q_values(), w.dtype)
    return oracle.paged_prefill(q, kc, vc, view["block_tables"], view["context_lens"], pw.query_start_loc,
                                w.scale, w.dtype, num_threads=oracle.num_host_threads())


@pytest.mark.parametrize("H,Hk,bs,dtype", [
    (32, 8, 16, "bf16"),     # G = 4
    (64, 8, 16, "bf16"),     # G = 8
    (8, 8, 32, "f16"),       # G = 1
    (12, 4, 8, "bf16"),      # G = 3, padded to 4
    (32, 2, 128, "f16"),     # G = 16
    (16, 4, 64, "bf16"),     # G = 4, block size 64
])
def test_chunked_prefill_against_oracle(pa, H, Hk, bs, dtype):
    prior = np.array([0, 5, 130, 700, 31, 0, 1000], np.int32)
    q_lens = np.array([1, 17, 64, 128, 200, 300, 33], np.int32)
    pw = workloads.make_prefill("prefill", 21 + H, prior, q_lens, H, Hk, 128, bs, dtype)
    out, _, _ = gpu_prefill(pa, pw)
    ref = oracle_prefill(pw)
    assert_close(to_f64(out), ref, dtype, f"prefill H{H}/{Hk} bs{bs} {dtype}")
    assert pa.get_device_error() == 0


def test_prefill_beyond_the_sort_keeps_index_order(pa):
    """More (sequence, query tile) entries than the kernel's item sort takes
    (16384): the items are dealt in index order, with the same results. G = 16
    makes a query tile 8 tokens, so one 2048-token chunk and 129 one-token chunks
    give 130 x 256 entries."""
    q_lens = np.array([2048] + [1] * 129, np.int32)
    prior = (np.arange(130) % 40).astype(np.int32)
    pw = workloads.make_prefill("prefill_many", 77, prior, q_lens, 32, 2, 128, 16, "bf16")
    assert pw.base.num_seqs * (2048 // 8) > 16384
    out, _, _ = gpu_prefill(pa, pw)
    assert_close(to_f64(out), oracle_prefill(pw), "bf16", "prefill in index order")
    assert pa.get_device_error() == 0


def test_chunked_prefill_workload(pa):
    pw = workloads.chunked_prefill(num_seqs=6)
    out, _, _ = gpu_prefill(pa, pw)
    ref = oracle_prefill(pw)
    assert_close(to_f64(out), ref, "bf16", "chunked_prefill")
    assert pa.get_device_error() == 0


def test_single_token_chunks_match_the_decode_kernel(pa):
    prior = np.array([0, 40, 511, 2000], np.int32)
    pw = workloads.make_prefill("one", 7, prior, np.ones(4, np.int32), 32, 8, 128, 16, "bf16")
    out, kc, vc = gpu_prefill(pa, pw)
    q = pw.q_values(like=kc).to(torch.bfloat16).contiguous()
    dec = torch.empty_like(q)
    d = dev()
    pa.paged_attention_decode(dec, q, kc, vc, torch.as_tensor(pw.base.block_tables, device=d),
                              torch.as_tensor(pw.base.context_lens, device=d), pw.base.scale)
    torch.cuda.synchronize()
    assert float((out.double() - dec.double()).abs().max()) <= 2e-2


def test_inconsistent_lengths_are_reported(pa):
    pw = workloads.make_prefill("bad", 3, np.array([10, 10], np.int32), np.array([8, 8], np.int32),
                                8, 2, 128, 16, "bf16")
    d = dev()
    kc = torch.zeros((pw.base.num_blocks, 16, 2, 128), dtype=torch.bfloat16, device=d)
    q = torch.zeros((16, 8, 128), dtype=torch.bfloat16, device=d)
    out = torch.zeros_like(q)
    lens = torch.tensor([18, 5], dtype=torch.int32, device=d)          # second chunk longer than its context
    pa.paged_attention_prefill(out, q, kc, kc, torch.as_tensor(pw.base.block_tables, device=d), lens,
                               torch.as_tensor(pw.query_start_loc, device=d), 0.1, 8)
    assert pa.get_device_error() & pa.PA_DEVERR_CONTEXT
    assert torch.isfinite(out.float()).all()
