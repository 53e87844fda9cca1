"""8-bit decode with append (pa_paged_attention_decode_fp8_append) against the two
calls it stands for -- paged_kv_write_fp8 of each sequence's new token, then the
8-bit decode -- and against the oracle, in the launch configuration the bench
times.

The decode kernel's producer warps quantise each token with the scatter's
encoding and store it just before they load the tile that holds it, so codes and
outputs must be bit-identical to the separate calls. A slot that is not that of
position ctx - 1 is reported (PA_DEVERR_SLOT) and not written."""
import numpy as np
import pytest
import torch

import workloads
from gpu_cases import FP8_POISON, assert_close, dev, oracle_decode_fp8, pa_mod, to_f64

pytestmark = pytest.mark.gpu

S = workloads.FP8_SCALE


@pytest.fixture(autouse=True)
def _free_memory():
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


@pytest.fixture(scope="module")
def pa():
    return pa_mod()


def _inputs(w):
    d = dev()
    dt = workloads.torch_dtype(w.dtype)
    shape = (w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim)
    kc = torch.full(shape, FP8_POISON, dtype=torch.uint8, device=d)
    vc = torch.full(shape, FP8_POISON, dtype=torch.uint8, device=d)
    w.fill_cache_torch(kc, vc, include_newest=False)
    kn, vn = w.newest_kv(like=kc)
    q = w.q_values(like=kc).to(dt).contiguous()
    return kc, vc, kn.to(dt).contiguous(), vn.to(dt).contiguous(), q


def _both(pa, w, slots=None, partition_size=0, k_scale=S, v_scale=S):
    """(out, key codes, value codes, error bits) of the fused call and of write + decode."""
    d = dev()
    kc, vc, kn, vn, q = _inputs(w)
    sl = torch.as_tensor(w.slot_mapping if slots is None else slots, device=d)
    bt = torch.as_tensor(w.block_tables, device=d)
    cl = torch.as_tensor(w.context_lens, device=d)
    res = []
    for fused in (True, False):
        k2, v2 = kc.clone(), vc.clone()
        out = torch.full_like(q, float("nan"))
        if fused:
            pa.paged_attention_decode_fp8_append(out, q, kn, vn, sl, k2, v2, bt, cl, w.scale, k_scale, v_scale,
                                                 partition_size=partition_size)
        else:
            pa.paged_kv_write_fp8(kn, vn, sl, k2, v2, k_scale, v_scale)
            pa.paged_attention_decode_fp8(out, q, k2, v2, bt, cl, w.scale, k_scale, v_scale,
                                          partition_size=partition_size)
        torch.cuda.synchronize()
        res.append((out, k2, v2, pa.get_device_error()))
    return res


def _same_out(a, b):
    return torch.equal(a.view(torch.int16), b.view(torch.int16))        # NaN-aware bitwise equality


@pytest.mark.parametrize("dtype,bs,H,Hk", [("bf16", 16, 32, 8), ("f16", 32, 64, 8), ("bf16", 64, 16, 2),
                                            ("bf16", 8, 8, 8), ("f16", 128, 32, 8)])
def test_fp8_append_equals_write_then_decode(pa, dtype, bs, H, Hk):
    ctx = np.array([1, 2, 127, 128, 129, 511, 512, 513, 1000, 3000, 0, 77], np.int32)
    w = workloads.make_decode("fp8_append", 701, ctx, H, Hk, 128, bs, dtype)
    (o1, k1, v1, e1), (o2, k2, v2, e2) = _both(pa, w)
    assert e1 == 0 and e2 == 0
    assert _same_out(o1, o2) and torch.equal(k1, k2) and torch.equal(v1, v2)


@pytest.mark.parametrize("k_scale,v_scale", [(2.0 ** -8, 0.37), (1024.0, 3.0e-3)])
def test_fp8_append_saturating_and_subnormal_scales(pa, k_scale, v_scale):
    """Scales whose quotients saturate at 448 (k / 2^-8) or fall to the subnormal
    codes and signed zeros (k / 1024): the fused encoding is the scatter's."""
    ctx = np.array([3, 128, 300, 17], np.int32)
    w = workloads.make_decode("fp8_append_scales", 702, ctx, 16, 4, 128, 16, "bf16")
    (o1, k1, v1, e1), (o2, k2, v2, e2) = _both(pa, w, k_scale=k_scale, v_scale=v_scale)
    assert e1 == 0 and e2 == 0
    assert torch.equal(k1, k2) and torch.equal(v1, v2) and _same_out(o1, o2)


def test_fp8_append_long_context_partitions(pa):
    w = workloads.long_context(num_seqs=3)
    (o1, k1, v1, e1), (o2, k2, v2, e2) = _both(pa, w, partition_size=512)
    assert e1 == 0 and e2 == 0
    assert _same_out(o1, o2) and torch.equal(k1, k2) and torch.equal(v1, v2)


def test_fp8_append_batch_above_one_launch(pa):
    """More sequences than one partition launch takes: the launch for sequences
    512.. writes their own tokens."""
    rng = np.random.default_rng(7)
    w = workloads.make_decode("fp8_append_many", 703, rng.integers(1, 300, size=700).astype(np.int32), 8, 2, 128,
                              16, "bf16")
    (o1, k1, v1, e1), (o2, k2, v2, e2) = _both(pa, w)
    assert e1 == 0 and e2 == 0
    assert _same_out(o1, o2) and torch.equal(k1, k2) and torch.equal(v1, v2)


def test_fp8_append_skips_minus_one_slots(pa):
    w = workloads.make_decode("fp8_append_skip", 704, np.array([40, 600, 1300, 9], np.int32), 16, 4, 128, 16, "bf16")
    slots = w.slot_mapping.copy()
    slots[1] = -1
    slots[3] = -1
    (o1, k1, v1, e1), (o2, k2, v2, e2) = _both(pa, w, slots=slots)
    assert e1 == 0 and e2 == 0
    assert _same_out(o1, o2) and torch.equal(k1, k2) and torch.equal(v1, v2)


def test_fp8_append_llama8b_full_batch_against_the_oracle(pa):
    """The bench's configuration: the full 8B-shaped batch, a workspace and the host
    bound on the context length."""
    w = workloads.llama8b_decode()
    d = dev()
    kc, vc, kn, vn, q = _inputs(w)
    out = torch.full_like(q, float("nan"))
    mc = int(w.context_lens.max())
    ws = torch.empty(max(pa.decode_workspace_bytes(w.num_seqs, w.num_heads, w.head_dim, mc, 0), 16),
                     dtype=torch.uint8, device=d)
    pa.paged_attention_decode_fp8_append(out, q, kn, vn, torch.as_tensor(w.slot_mapping, device=d), kc, vc,
                                         torch.as_tensor(w.block_tables, device=d),
                                         torch.as_tensor(w.context_lens, device=d), w.scale, S, S,
                                         max_context_len=mc, workspace=ws)
    torch.cuda.synchronize()
    assert pa.get_device_error() == 0
    assert_close(to_f64(out), oracle_decode_fp8(w, range(w.num_seqs)), "bf16", "fp8 append llama8b_decode")


def test_fp8_append_reports_a_slot_that_is_not_the_last_position(pa):
    w = workloads.make_decode("fp8_append_bad", 705, np.array([40, 600, 0], np.int32), 16, 4, 128, 16, "bf16")
    good = w.slot_mapping.copy()
    bad = good.copy()
    bad[0] = good[0] - 1                 # the slot before the sequence's last position
    bad[2] = good[1] + 1                 # an empty context takes only -1
    d = dev()
    kc, vc, kn, vn, q = _inputs(w)
    before = kc.clone()
    out = torch.empty_like(q)
    pa.paged_attention_decode_fp8_append(out, q, kn, vn, torch.as_tensor(bad, device=d), kc, vc,
                                         torch.as_tensor(w.block_tables, device=d),
                                         torch.as_tensor(w.context_lens, device=d), w.scale, S, S)
    torch.cuda.synchronize()
    assert pa.get_device_error() & pa.PA_DEVERR_SLOT
    row = w.num_kv_heads * w.head_dim
    flat_b, flat_k = before.view(-1, row), kc.view(-1, row)
    assert torch.equal(flat_k[int(bad[0])], flat_b[int(bad[0])])       # not written
    assert torch.equal(flat_k[int(bad[2])], flat_b[int(bad[2])])
    assert not torch.equal(flat_k[int(good[1])], flat_b[int(good[1])])  # the good token was
