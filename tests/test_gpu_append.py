"""Decode with append (pa_paged_attention_decode_append) against the two calls it
stands for -- paged_kv_write of each sequence's new token, then the decode -- and
against the oracle, in the launch configuration the bench times.

Outputs and caches must be bit-identical to the separate calls: the tensor-core
decode writes the tokens itself (the CTA that reads a token's block writes it
first), the other paths run the scatter first. A slot that is not that of
position ctx - 1 is reported (PA_DEVERR_SLOT) and not written."""
import numpy as np
import pytest
import torch

import workloads
from gpu_cases import assert_close, check_newest_rows, dev, oracle_decode, pa_mod, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _free_memory():
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


@pytest.fixture(scope="module")
def pa():
    return pa_mod()


def _both(pa, w, slots=None, partition_size=0):
    """(out, key cache, value cache) of the fused call and of write + decode."""
    d = dev()
    dt = workloads.torch_dtype(w.dtype)
    shape = (w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim)
    kc = torch.full(shape, float("nan"), dtype=dt, device=d)
    vc = torch.full(shape, float("nan"), dtype=dt, device=d)
    w.fill_cache_torch(kc, vc, include_newest=False)
    kn, vn = w.newest_kv(like=kc)
    kn, vn = kn.to(dt).contiguous(), vn.to(dt).contiguous()
    q = w.q_values(like=kc).to(dt).contiguous()
    sl = torch.as_tensor(w.slot_mapping if slots is None else slots, device=d)
    bt = torch.as_tensor(w.block_tables, device=d)
    cl = torch.as_tensor(w.context_lens, device=d)
    res = []
    for fused in (True, False):
        k2, v2 = kc.clone(), vc.clone()
        out = torch.full_like(q, float("nan"))
        if fused:
            pa.paged_attention_decode_append(out, q, kn, vn, sl, k2, v2, bt, cl, w.scale,
                                             partition_size=partition_size)
        else:
            pa.paged_kv_write(kn, vn, sl, k2, v2)
            pa.paged_attention_decode(out, q, k2, v2, bt, cl, w.scale, partition_size=partition_size)
        torch.cuda.synchronize()
        res.append((out, k2, v2, pa.get_device_error()))
    return res


def _append(pa, w, max_context_len=0, partition_size=0):
    """Decode with append over a NaN-poisoned cache that lacks each sequence's
    newest token, in the launch configuration the bench uses (a workspace and the
    host bound on the context length)."""
    d = dev()
    dt = workloads.torch_dtype(w.dtype)
    shape = (w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim)
    kc = torch.full(shape, float("nan"), dtype=dt, device=d)
    vc = torch.full(shape, float("nan"), dtype=dt, device=d)
    w.fill_cache_torch(kc, vc, include_newest=False)
    kn, vn = w.newest_kv(like=kc)
    q = w.q_values(like=kc).to(dt).contiguous()
    out = torch.full_like(q, float("nan"))
    mc = max_context_len or int(w.context_lens.max())
    ws = torch.empty(max(pa.decode_workspace_bytes(w.num_seqs, w.num_heads, w.head_dim, mc, partition_size), 16),
                     dtype=torch.uint8, device=d)
    pa.paged_attention_decode_append(out, q, kn.to(dt).contiguous(), vn.to(dt).contiguous(),
                                     torch.as_tensor(w.slot_mapping, device=d), kc, vc,
                                     torch.as_tensor(w.block_tables, device=d),
                                     torch.as_tensor(w.context_lens, device=d), w.scale, max_context_len=mc,
                                     partition_size=partition_size, workspace=ws)
    torch.cuda.synchronize()
    return out, kc, vc


def test_append_ragged_against_the_oracle(pa):
    ctx = np.array([1, 2, 127, 128, 129, 511, 512, 513, 1000, 3000, 77], np.int32)
    w = workloads.make_decode("append_oracle", 606, ctx, 32, 8, 128, 16, "bf16")
    out, kc, vc = _append(pa, w)
    check_newest_rows(w, kc, vc)
    assert_close(to_f64(out), oracle_decode(w, range(w.num_seqs)), "bf16", "append ragged")
    assert pa.get_device_error() == 0


def test_append_llama8b_full_batch_against_the_oracle(pa):
    w = workloads.llama8b_decode()
    out, kc, vc = _append(pa, w)
    check_newest_rows(w, kc, vc)
    assert_close(to_f64(out), oracle_decode(w, range(w.num_seqs)), "bf16", "append llama8b_decode")
    assert pa.get_device_error() == 0


def test_append_long_context_sampled_against_the_oracle(pa):
    w = workloads.long_context()
    out, kc, vc = _append(pa, w)
    check_newest_rows(w, kc, vc)
    seqs = [int(np.argmin(w.context_lens)), int(np.argmax(w.context_lens))]
    assert_close(to_f64(out)[seqs], oracle_decode(w, seqs), "bf16", "append long_context")
    assert pa.get_device_error() == 0


def _same(a, b):
    # NaN-aware bitwise equality (unused cache slots hold NaN)
    return torch.equal(a.view(torch.int16) if a.element_size() == 2 else a.view(torch.int32),
                       b.view(torch.int16) if b.element_size() == 2 else b.view(torch.int32))


@pytest.mark.parametrize("dtype,bs,H,Hk", [("bf16", 16, 32, 8), ("f16", 32, 64, 8), ("bf16", 64, 16, 2),
                                            ("bf16", 8, 8, 8)])
def test_append_equals_write_then_decode(pa, dtype, bs, H, Hk):
    ctx = np.array([1, 2, 127, 128, 129, 511, 512, 513, 1000, 3000, 0, 77], np.int32)
    w = workloads.make_decode("append", 601, ctx, H, Hk, 128, bs, dtype)
    (o1, k1, v1, e1), (o2, k2, v2, e2) = _both(pa, w)
    assert e1 == 0 and e2 == 0
    assert _same(o1, o2) and _same(k1, k2) and _same(v1, v2)


def test_append_long_context_partitions(pa):
    w = workloads.long_context(num_seqs=3)
    (o1, k1, v1, e1), (o2, k2, v2, e2) = _both(pa, w, partition_size=512)
    assert e1 == 0 and e2 == 0
    assert _same(o1, o2) and _same(k1, k2) and _same(v1, v2)


def test_append_batch_above_one_launch(pa):
    """More sequences than one partition launch takes: the launch for sequences
    512.. writes their own tokens."""
    rng = np.random.default_rng(5)
    w = workloads.make_decode("append_many", 602, rng.integers(1, 300, size=700).astype(np.int32), 8, 2, 128, 16,
                              "bf16")
    (o1, k1, v1, e1), (o2, k2, v2, e2) = _both(pa, w)
    assert e1 == 0 and e2 == 0
    assert _same(o1, o2) and _same(k1, k2) and _same(v1, v2)


def test_append_fp32_takes_the_scatter_then_the_simt_decode(pa):
    w = workloads.make_decode("append_f32", 603, np.array([5, 17, 300, 0], np.int32), 8, 4, 64, 8, "f32")
    (o1, k1, v1, e1), (o2, k2, v2, e2) = _both(pa, w)
    assert e1 == 0 and e2 == 0
    assert _same(o1, o2) and _same(k1, k2) and _same(v1, v2)


def test_append_skips_minus_one_slots(pa):
    w = workloads.make_decode("append_skip", 604, np.array([40, 600, 1300, 9], np.int32), 16, 4, 128, 16, "bf16")
    slots = w.slot_mapping.copy()
    slots[1] = -1
    slots[3] = -1
    (o1, k1, v1, e1), (o2, k2, v2, e2) = _both(pa, w, slots=slots)
    assert e1 == 0 and e2 == 0
    assert _same(o1, o2) and _same(k1, k2) and _same(v1, v2)


def test_append_reports_a_slot_that_is_not_the_last_position(pa):
    w = workloads.make_decode("append_bad", 605, np.array([40, 600, 0], np.int32), 16, 4, 128, 16, "bf16")
    good = w.slot_mapping.copy()
    bad = good.copy()
    bad[0] = good[0] - 1                 # the slot before the sequence's last position
    bad[2] = good[1] + 1                 # an empty context takes only -1
    d = dev()
    dt = workloads.torch_dtype(w.dtype)
    shape = (w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim)
    kc = torch.zeros(shape, dtype=dt, device=d)
    vc = torch.zeros_like(kc)
    w.fill_cache_torch(kc, vc, include_newest=False)
    before = kc.clone()
    kn, vn = w.newest_kv(like=kc)
    q = w.q_values(like=kc).to(dt).contiguous()
    out = torch.empty_like(q)
    pa.paged_attention_decode_append(out, q, kn.to(dt).contiguous(), vn.to(dt).contiguous(),
                                     torch.as_tensor(bad, device=d), kc, vc, torch.as_tensor(w.block_tables, device=d),
                                     torch.as_tensor(w.context_lens, device=d), w.scale)
    torch.cuda.synchronize()
    assert pa.get_device_error() & pa.PA_DEVERR_SLOT
    flat_b, flat_k = before.view(-1, w.num_kv_heads * w.head_dim), kc.view(-1, w.num_kv_heads * w.head_dim)
    assert torch.equal(flat_k[int(bad[0])], flat_b[int(bad[0])])       # not written
    assert torch.equal(flat_k[int(bad[2])], flat_b[int(bad[2])])
    assert not torch.equal(flat_k[int(good[1])], flat_b[int(good[1])])  # the good token was

