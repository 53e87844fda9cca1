"""Back-to-back decode calls on one stream, with no host synchronisation between them.

The partition kernels are launched as programmatic dependents and build their item
order before they wait for the kernel ahead of them, and the merge after a
tensor-core partition kernel lets the next launch start early. Each call here reads
its own lengths and writes its own output through one shared workspace, right after
another call's merge; every output must equal the same call run alone, bit for bit."""
import numpy as np
import pytest
import torch

import workloads
from gpu_cases import FP8_POISON, dev, pa_mod

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


def _variants(w, n, seed):
    """n length arrays over the same tables: each sequence keeps a random prefix of
    its context (1 .. ctx tokens), so the calls differ in partitions and in which rows
    the merge combines."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        cl = np.array([int(rng.integers(1, c + 1)) for c in w.context_lens], np.int32)
        out.append(torch.as_tensor(cl, device=dev()))
    return out


@pytest.mark.parametrize("long", [False, True], ids=["warp_merge", "block_merge"])
@pytest.mark.parametrize("fp8", [False, True])
def test_back_to_back_calls_equal_isolated_calls(pa, fp8, long):
    """block_merge: few sequences of 17k-40k tokens in partitions of 512, so rows hold
    up to 79 partitions and the merge of one CTA per row follows the partition kernel."""
    if long:
        ctx = np.random.default_rng(13).integers(17000, 40000, size=4).astype(np.int32)
        part = 512
    else:
        ctx = np.random.default_rng(11).integers(300, 4096, size=48).astype(np.int32)
        part = 0
    w = workloads.make_decode("chain", 811, ctx, 32, 8, 128, 16, "bf16")
    d = dev()
    shape = (w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim)
    if fp8:
        kc = torch.full(shape, FP8_POISON, dtype=torch.uint8, device=d)
        vc = torch.full(shape, FP8_POISON, dtype=torch.uint8, device=d)
    else:
        kc = torch.full(shape, float("nan"), dtype=torch.bfloat16, device=d)
        vc = torch.full(shape, float("nan"), dtype=torch.bfloat16, device=d)
    w.fill_cache_torch(kc, vc, include_newest=True)
    q = w.q_values(like=kc).to(torch.bfloat16).contiguous()
    bt = torch.as_tensor(w.block_tables, device=d)
    lens = _variants(w, 6, 12 + int(fp8))
    mc = int(w.context_lens.max())
    ws = torch.empty(pa.decode_workspace_bytes(w.num_seqs, w.num_heads, w.head_dim, mc, part), dtype=torch.uint8,
                     device=d)

    def call(out, cl):
        if fp8:
            pa.paged_attention_decode_fp8(out, q, kc, vc, bt, cl, w.scale, S, S, max_context_len=mc,
                                          partition_size=part, workspace=ws)
        else:
            pa.paged_attention_decode(out, q, kc, vc, bt, cl, w.scale, max_context_len=mc, partition_size=part,
                                      workspace=ws)

    alone = []
    for cl in lens:
        out = torch.full_like(q, float("nan"))
        call(out, cl)
        torch.cuda.synchronize()
        alone.append(out)
    assert pa.get_device_error() == 0
    chained = [[torch.full_like(q, float("nan")) for _ in lens] for _ in range(3)]
    for r in range(3):
        for out, cl in zip(chained[r], lens):
            call(out, cl)
    torch.cuda.synchronize()
    assert pa.get_device_error() == 0
    for r in range(3):
        for i, (a, b) in enumerate(zip(alone, chained[r])):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16)), (r, i)


def test_back_to_back_appends_equal_isolated_calls(pa):
    """Decode steps with append, back to back: each step writes its sequences' new
    tokens (into the slots of position ctx - 1) and decodes, right after the previous
    step's merge."""
    ctx = np.random.default_rng(21).integers(300, 4096, size=48).astype(np.int32)
    w = workloads.make_decode("chain_append", 812, ctx, 32, 8, 128, 16, "bf16")
    d = dev()
    shape = (w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim)
    kc = torch.full(shape, float("nan"), dtype=torch.bfloat16, device=d)
    vc = torch.full(shape, float("nan"), dtype=torch.bfloat16, device=d)
    w.fill_cache_torch(kc, vc, include_newest=False)
    kn, vn = w.newest_kv(like=kc)
    kn, vn = kn.to(torch.bfloat16).contiguous(), vn.to(torch.bfloat16).contiguous()
    q = w.q_values(like=kc).to(torch.bfloat16).contiguous()
    bt = torch.as_tensor(w.block_tables, device=d)
    cl = torch.as_tensor(w.context_lens, device=d)
    sl = torch.as_tensor(w.slot_mapping, device=d)
    mc = int(w.context_lens.max())
    ws = torch.empty(pa.decode_workspace_bytes(w.num_seqs, w.num_heads, w.head_dim, mc, 0), dtype=torch.uint8,
                     device=d)
    ref = torch.full_like(q, float("nan"))
    pa.paged_attention_decode_append(ref, q, kn, vn, sl, kc, vc, bt, cl, w.scale, max_context_len=mc, workspace=ws)
    torch.cuda.synchronize()
    outs = [torch.full_like(q, float("nan")) for _ in range(8)]
    for out in outs:
        pa.paged_attention_decode_append(out, q, kn, vn, sl, kc, vc, bt, cl, w.scale, max_context_len=mc,
                                         workspace=ws)
    torch.cuda.synchronize()
    assert pa.get_device_error() == 0
    for i, out in enumerate(outs):
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), i
