"""GPU parity: the library against the CPU oracle on the same seeded inputs.

Bit-exact for scatter, block copy and indexing; max/mean abs error within
2e-2 / 2e-3 for bf16 and fp16 outputs and 1e-5 for fp32 outputs.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_cases import (assert_close, check_newest_rows, dev, gpu_decode, oracle_decode, pa_mod,
                       to_f64)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _free_memory():
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


@pytest.fixture(scope="module")
def pa():
    return pa_mod()


def _errors_clear(pa):
    assert pa.get_device_error() == 0


# ---------------------------------------------------------------------------
# the named workloads
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("partition_size", [0, 128])
def test_tiny_fp32(pa, partition_size):
    w = workloads.tiny_fp32()
    out, kc, vc = gpu_decode(w, partition_size=partition_size)
    check_newest_rows(w, kc, vc)
    ref = oracle_decode(w, range(w.num_seqs))
    assert_close(to_f64(out), ref, "f32", "tiny_fp32")
    _errors_clear(pa)


def test_fp32_split_k_with_ragged_partitions(pa):
    # several partitions of 128 tokens and a ragged last one, fp32 tolerance
    ctx = np.array([1, 127, 128, 129, 300, 640, 1000, 77], np.int32)
    w = workloads.make_decode("fp32_split", 11, ctx, 8, 2, 64, 8, "f32")
    out, kc, vc = gpu_decode(w, partition_size=128)
    ref = oracle_decode(w, range(w.num_seqs))
    assert_close(to_f64(out), ref, "f32", "fp32 split-K")
    _errors_clear(pa)


def test_llama8b_decode_full_batch(pa):
    w = workloads.llama8b_decode()
    out, kc, vc = gpu_decode(w)
    check_newest_rows(w, kc, vc)
    ref = oracle_decode(w, range(w.num_seqs))
    assert_close(to_f64(out), ref, "bf16", "llama8b_decode")
    _errors_clear(pa)


def test_long_context_split_k_sampled(pa):
    w = workloads.long_context()
    out, kc, vc = gpu_decode(w, max_context_len=int(w.context_lens.max()), partition_size=512)
    check_newest_rows(w, kc, vc)
    seqs = [int(np.argmin(w.context_lens)), int(np.argmax(w.context_lens))]
    ref = oracle_decode(w, seqs)
    assert_close(to_f64(out)[seqs], ref, "bf16", "long_context")
    # every row is a convex combination of V rows: finite and within the V range
    o = to_f64(out)
    assert np.all(np.isfinite(o)) and np.abs(o).max() <= workloads.CONTENT_MAX + 0.05
    _errors_clear(pa)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("bs", [8, 16, 32])
def test_mixed_serving_step(pa, bs, dtype):
    w = workloads.mixed_serving(block_size=bs, dtype=dtype)
    d = dev()
    tdt = workloads.torch_dtype(dtype)
    out, kc, vc = gpu_decode(w, max_context_len=int(w.context_lens.max()))
    check_newest_rows(w, kc, vc)
    # the 2048-token write to random free slots: bit-exact
    ek, ev = w.extra_write_rows(like=kc)
    slots = torch.as_tensor(w.extra_write_slots, device=d)
    pa.paged_kv_write(ek.to(tdt).contiguous(), ev.to(tdt).contiguous(), slots, kc, vc)
    torch.cuda.synchronize()
    row = w.num_kv_heads * w.head_dim
    got = kc.view(-1, row)[slots.long()].float().cpu().numpy()
    assert np.array_equal(got, workloads.rounded(ek.reshape(-1, row), dtype).cpu().numpy())
    got = vc.view(-1, row)[slots.long()].float().cpu().numpy()
    assert np.array_equal(got, workloads.rounded(ev.reshape(-1, row), dtype).cpu().numpy())
    rng = np.random.default_rng(bs)
    seqs = np.sort(rng.choice(w.num_seqs, 48, replace=False))
    seqs = np.unique(np.concatenate([seqs, [int(np.argmax(w.context_lens)), int(np.argmin(w.context_lens))]]))
    ref = oracle_decode(w, seqs)
    assert_close(to_f64(out)[seqs], ref, dtype, f"mixed bs{bs} {dtype}")
    _errors_clear(pa)


def test_block_size_sweep_gives_the_same_output(pa):
    # same contents at bs 8/16/32; outputs differ only by fp32 summation order
    outs = []
    for bs in (8, 16, 32):
        w = workloads.mixed_serving(block_size=bs, dtype="bf16", num_seqs=64, extra_write=16)
        outs.append(to_f64(gpu_decode(w)[0]))
    assert np.abs(outs[0] - outs[1]).max() <= 2e-2 and np.abs(outs[0] - outs[2]).max() <= 2e-2


def test_shared_prefix_sampling(pa):
    """Prefill, fork 8 samples per prompt, copy-on-write via copy_blocks, private
    tokens via paged_kv_write, then decode -- replayed on the GPU with the
    library allocator and on the CPU with the oracle's model."""
    sc = workloads.shared_prefix(num_prompts=8)
    d = dev()
    tdt = workloads.torch_dtype(sc.dtype)
    nb = sc.pool_blocks()
    a = pa.BlockAllocator(nb, sc.block_size)
    model = oracle.BlockPoolModel(nb, sc.block_size)
    prompt_slots, pairs, private_slots = [], [], []
    for p in range(sc.num_prompts):
        for al in (a, model):
            al.add_seq(p)
        s_lib, _ = a.append(p, sc.prompt_len)
        s_mod, _ = model.append(p, sc.prompt_len)
        assert s_lib.tolist() == s_mod
        prompt_slots.append(s_lib)
        for j in range(sc.samples_per_prompt):
            sid = 1000 + p * sc.samples_per_prompt + j
            a.fork(p, sid)
            model.fork(p, sid)
        a.free_seq(p)
        model.free_seq(p)
    for s in range(sc.num_samples):
        sid = 1000 + s
        sl, pr = a.append(sid, int(sc.private[s]) + 1)
        sm, pm = model.append(sid, int(sc.private[s]) + 1)
        assert sl.tolist() == sm and [tuple(x) for x in pr.tolist()] == pm
        pairs += pr.tolist()
        private_slots.append(sl)
    assert len(pairs) == 7 * sc.num_prompts
    ids = np.arange(sc.num_samples) + 1000
    mb = max(len(a.block_table(int(i))) for i in ids)
    tables, lens = a.export(ids, mb)
    w = sc.workload(tables, nb)
    assert np.array_equal(lens, w.context_lens)

    shape = (nb, sc.block_size, sc.num_kv_heads, sc.head_dim)
    kc = torch.full(shape, float("nan"), dtype=tdt, device=d)
    vc = torch.full(shape, float("nan"), dtype=tdt, device=d)
    # prefill the prompts through paged_kv_write
    for p in range(sc.num_prompts):
        pos = torch.arange(sc.prompt_len, device=d)
        keys = torch.full_like(pos, p)
        k = workloads.content_rows(w.seed, workloads.TID_K, keys, pos, w.row_elems)
        v = workloads.content_rows(w.seed, workloads.TID_V, keys, pos, w.row_elems)
        pa.paged_kv_write(k.to(tdt).view(-1, sc.num_kv_heads, sc.head_dim).contiguous(),
                          v.to(tdt).view(-1, sc.num_kv_heads, sc.head_dim).contiguous(),
                          torch.as_tensor(prompt_slots[p], device=d), kc, vc)
    # copy-on-write of the shared partial blocks, then every private token
    pa.copy_blocks(kc, vc, torch.as_tensor(np.array(pairs, np.int32), device=d))
    seq_idx = np.concatenate([np.full(len(s), i) for i, s in enumerate(private_slots)]).astype(np.int64)
    pos = np.concatenate([np.arange(sc.prompt_len, sc.prompt_len + len(s)) for s in private_slots]).astype(np.int64)
    slots = np.concatenate(private_slots).astype(np.int32)
    k = w.kv_rows(workloads.TID_K, torch.as_tensor(seq_idx, device=d), torch.as_tensor(pos, device=d))
    v = w.kv_rows(workloads.TID_V, torch.as_tensor(seq_idx, device=d), torch.as_tensor(pos, device=d))
    pa.paged_kv_write(k.to(tdt).view(-1, sc.num_kv_heads, sc.head_dim).contiguous(),
                      v.to(tdt).view(-1, sc.num_kv_heads, sc.head_dim).contiguous(),
                      torch.as_tensor(slots, device=d), kc, vc)
    q = w.q_values(like=kc).to(tdt).contiguous()
    out = torch.empty_like(q)
    pa.paged_attention_decode(out, q, kc, vc, torch.as_tensor(tables, device=d),
                              torch.as_tensor(lens, device=d), w.scale)
    torch.cuda.synchronize()
    _errors_clear(pa)

    # every live slot of every sample holds exactly its content (bit-exact)
    ref_cache_k = torch.full_like(kc, float("nan"))
    ref_cache_v = torch.full_like(vc, float("nan"))
    w.fill_cache_torch(ref_cache_k, ref_cache_v, include_newest=True)
    live = ~torch.isnan(ref_cache_k[..., 0, 0])
    assert torch.equal(kc[live], ref_cache_k[live]) and torch.equal(vc[live], ref_cache_v[live])
    seqs = np.arange(0, w.num_seqs, 5)
    ref = oracle_decode(w, seqs)
    assert_close(to_f64(out)[seqs], ref, "bf16", "shared prefix")


# ---------------------------------------------------------------------------
# edge cases
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("H,Hk,D,bs,dtype", [
    (4, 4, 128, 16, "bf16"),     # MHA, G = 1
    (32, 2, 128, 16, "bf16"),    # G = 16
    (12, 4, 64, 8, "f16"),       # G = 3 (padded group), D = 64
    (8, 1, 64, 1, "bf16"),       # block size 1
    (8, 2, 128, 256, "f16"),     # block size 256
    (16, 4, 64, 4, "f32"),       # fp32, small blocks
])
def test_shapes_and_ragged_contexts(pa, H, Hk, D, bs, dtype):
    ctx = np.array([0, 1, 2, bs, bs + 1, 511, 512, 513, 1024, 1537], np.int32)
    w = workloads.make_decode("edge", 17, ctx, H, Hk, D, bs, dtype)
    out, kc, vc = gpu_decode(w, partition_size=256)
    check_newest_rows(w, kc, vc)
    ref = oracle_decode(w, range(w.num_seqs))
    got = to_f64(out)
    assert np.all(got[0] == 0.0)                      # empty context -> zero row
    assert_close(got, ref, dtype, f"edge H{H} Hk{Hk} D{D} bs{bs} {dtype}")
    _errors_clear(pa)


def test_single_token_context_returns_v_exactly(pa):
    ctx = np.array([1, 1, 1], np.int32)
    w = workloads.make_decode("one", 5, ctx, 8, 2, 128, 16, "bf16")
    out, kc, vc = gpu_decode(w)
    kn, vn = w.newest_kv()
    expect = np.repeat(workloads.rounded(vn, "bf16"), 4, axis=1)   # every head of a group sees V_0
    assert np.array_equal(out.float().cpu().numpy(), expect)


def test_workspace_paths_agree(pa):
    w = workloads.llama8b_decode(num_seqs=16)
    a = to_f64(gpu_decode(w, partition_size=256)[0])
    b = to_f64(gpu_decode(w, partition_size=256,
                          workspace=torch.empty(pa.decode_workspace_bytes(16, 32, 128, 4096, 256),
                                                dtype=torch.uint8, device=dev()))[0])
    assert np.array_equal(a, b)
    # library-allocated workspace (NULL pointer through the C ABI)
    d = dev()
    kc = torch.zeros((w.num_blocks, 16, 8, 128), dtype=torch.bfloat16, device=d)
    vc = torch.zeros_like(kc)
    w.fill_cache_torch(kc, vc, include_newest=True)
    q = w.q_values(like=kc).to(torch.bfloat16).contiguous()
    out = torch.empty_like(q)
    bt = torch.as_tensor(w.block_tables, device=d)
    cl = torch.as_tensor(w.context_lens, device=d)
    L = pa.lib()
    rc = L.pa_paged_attention_decode(out.data_ptr(), q.data_ptr(), kc.data_ptr(), vc.data_ptr(),
                                     bt.data_ptr(), bt.shape[1], cl.data_ptr(), 16, 32, 8, 128, 16,
                                     w.num_blocks, w.scale, 0, 256, None, 0, pa.PA_DTYPE_BF16,
                                     torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert np.array_equal(to_f64(out), a)
    small = torch.empty(64, dtype=torch.uint8, device=d)
    rc = L.pa_paged_attention_decode(out.data_ptr(), q.data_ptr(), kc.data_ptr(), vc.data_ptr(),
                                     bt.data_ptr(), bt.shape[1], cl.data_ptr(), 16, 32, 8, 128, 16,
                                     w.num_blocks, w.scale, 0, 256, small.data_ptr(), 64,
                                     pa.PA_DTYPE_BF16, torch.cuda.current_stream().cuda_stream)
    assert rc == pa.PA_ERR_WORKSPACE


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_copy_blocks_bit_exact(pa, dtype):
    rng = np.random.default_rng(21)
    d = dev()
    tdt = workloads.torch_dtype(dtype)
    nb, bs, hk, D = 96, 16, 8, 128
    kc = (torch.randn((nb, bs, hk, D), device=d) * 3).to(tdt)
    vc = (torch.randn((nb, bs, hk, D), device=d) * 3).to(tdt)
    perm = rng.permutation(nb)
    pairs = np.stack([perm[:30], perm[30:60]], 1).astype(np.int32)      # distinct dsts, no dst is a src
    kh = kc.cpu().numpy() if dtype != "bf16" else kc.view(torch.int16).cpu().numpy().view(np.uint16)
    vh = vc.cpu().numpy() if dtype != "bf16" else vc.view(torch.int16).cpu().numpy().view(np.uint16)
    kh, vh = kh.copy(), vh.copy()
    oracle.copy_blocks(kh, vh, pairs, dtype)
    pa.copy_blocks(kc, vc, torch.as_tensor(pairs, device=d))
    torch.cuda.synchronize()
    gk = kc.cpu().numpy() if dtype != "bf16" else kc.view(torch.int16).cpu().numpy().view(np.uint16)
    gv = vc.cpu().numpy() if dtype != "bf16" else vc.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(gk.view(np.uint8), kh.view(np.uint8))
    assert np.array_equal(gv.view(np.uint8), vh.view(np.uint8))
    _errors_clear(pa)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_kv_write_bit_exact_against_oracle(pa, dtype):
    rng = np.random.default_rng(22)
    d = dev()
    nb, bs, hk, D, T = 40, 8, 4, 64, 300
    slots = rng.choice(nb * bs, T, replace=False).astype(np.int32)
    slots[::7] = -1
    keys = np.arange(T, dtype=np.int64)
    k = workloads.content_rows(3, 0, keys, keys, hk * D)
    v = workloads.content_rows(3, 1, keys, keys, hk * D)
    kc = np.zeros((nb, bs, hk, D), np.float32)
    vc = np.zeros_like(kc)
    kst, vst = workloads.to_storage_numpy(kc, dtype), workloads.to_storage_numpy(vc, dtype)
    oracle.kv_write(workloads.to_storage_numpy(k, dtype), workloads.to_storage_numpy(v, dtype), slots,
                    kst, vst, dtype)
    tdt = workloads.torch_dtype(dtype)
    gk = torch.zeros((nb, bs, hk, D), dtype=tdt, device=d)
    gv = torch.zeros_like(gk)
    pa.paged_kv_write(torch.as_tensor(k).to(tdt).view(T, hk, D).to(d),
                      torch.as_tensor(v).to(tdt).view(T, hk, D).to(d),
                      torch.as_tensor(slots, device=d), gk, gv)
    torch.cuda.synchronize()
    assert np.array_equal(workloads.to_storage_numpy(gk.float().cpu().numpy(), dtype), kst)
    assert np.array_equal(workloads.to_storage_numpy(gv.float().cpu().numpy(), dtype), vst)
    _errors_clear(pa)


# ---------------------------------------------------------------------------
# device-side index checks: the bad access is skipped and an error bit set
# ---------------------------------------------------------------------------

def test_bad_slot_sets_the_error_and_skips_only_that_token(pa):
    d = dev()
    kc = torch.zeros((4, 4, 1, 64), dtype=torch.bfloat16, device=d)
    vc = torch.zeros_like(kc)
    k = torch.ones((3, 1, 64), dtype=torch.bfloat16, device=d)
    slots = torch.tensor([2, 16, -7], dtype=torch.int32, device=d)
    pa.paged_kv_write(k, k, slots, kc, vc)
    assert pa.get_device_error() & pa.PA_DEVERR_SLOT
    assert float(kc.float().sum()) == 64.0
    assert pa.get_device_error() == 0                          # read clears


def test_bad_block_id_sets_the_error(pa):
    # the cache is filled through the valid table; only the decode sees the bad id
    w = workloads.make_decode("badid", 3, np.array([40, 40], np.int32), 8, 2, 128, 16, "bf16")
    d = dev()
    kc = torch.zeros((w.num_blocks, 16, 2, 128), dtype=torch.bfloat16, device=d)
    vc = torch.zeros_like(kc)
    w.fill_cache_torch(kc, vc, include_newest=True)
    bad = w.block_tables.copy()
    bad[1, 1] = w.num_blocks + 5
    q = w.q_values(like=kc).to(torch.bfloat16).contiguous()
    out = torch.empty_like(q)
    pa.paged_attention_decode(out, q, kc, vc, torch.as_tensor(bad, device=d),
                              torch.as_tensor(w.context_lens, device=d), w.scale)
    assert pa.get_device_error() & pa.PA_DEVERR_BLOCK_ID
    ref = oracle_decode(w, [0])
    assert_close(to_f64(out)[:1], ref, "bf16", "unaffected sequence")
    assert torch.isfinite(out.float()).all()


def test_context_beyond_table_sets_the_error(pa):
    w = workloads.make_decode("badctx", 3, np.array([40, 40], np.int32), 8, 2, 128, 16, "bf16")
    d = dev()
    kc = torch.zeros((w.num_blocks, 16, 2, 128), dtype=torch.bfloat16, device=d)
    q = torch.zeros((2, 8, 128), dtype=torch.bfloat16, device=d)
    out = torch.empty_like(q)
    lens = torch.tensor([40, 10_000], dtype=torch.int32, device=d)
    pa.paged_attention_decode(out, q, kc, kc, torch.as_tensor(w.block_tables, device=d), lens, 0.1)
    assert pa.get_device_error() & pa.PA_DEVERR_CONTEXT
    assert torch.isfinite(out.float()).all()


def test_bad_copy_pair_sets_the_error(pa):
    d = dev()
    kc = torch.arange(4 * 2 * 1 * 64, dtype=torch.float32, device=d).view(4, 2, 1, 64)
    vc = kc.clone()
    before = kc.clone()
    pa.copy_blocks(kc, vc, torch.tensor([[0, 9], [1, 2]], dtype=torch.int32, device=d))
    assert pa.get_device_error() & pa.PA_DEVERR_COPY_PAIR
    assert torch.equal(kc[2], before[1]) and torch.equal(kc[0], before[0])


# ---------------------------------------------------------------------------
# both decode kernels (tensor-core and SIMT) against the oracle
# ---------------------------------------------------------------------------

@pytest.fixture
def force_kernel(monkeypatch):
    def set_kernel(name):
        monkeypatch.setenv("PA_DECODE_KERNEL", name)
    return set_kernel


@pytest.mark.parametrize("kernel", ["tc", "simt"])
@pytest.mark.parametrize("bs,dtype,H,Hk", [(16, "bf16", 32, 8), (8, "f16", 32, 8), (32, "bf16", 64, 8),
                                           (128, "bf16", 16, 16), (64, "f16", 48, 4)])
def test_decode_kernels_against_oracle(pa, force_kernel, kernel, bs, dtype, H, Hk):
    force_kernel(kernel)
    rng = np.random.default_rng(bs + H)
    ctx = np.concatenate([[0, 1, 127, 128, 129, 511, 512, 513, 1500], rng.integers(1, 3000, size=23)]).astype(np.int32)
    w = workloads.make_decode(f"k_{kernel}", 31, ctx, H, Hk, 128, bs, dtype)
    out, kc, vc = gpu_decode(w, max_context_len=int(ctx.max()))
    check_newest_rows(w, kc, vc)
    ref = oracle_decode(w, range(w.num_seqs))
    got = to_f64(out)
    assert np.all(got[0] == 0.0)
    assert_close(got, ref, dtype, f"{kernel} bs{bs} {dtype} H{H}/{Hk}")
    _errors_clear(pa)


@pytest.mark.parametrize("H", [64, 32])
def test_tc_many_short_items_per_cta(pa, force_kernel, H):
    """About thirty items per CTA, most of one or two tiles, empty contexts among them and
    partitions of 256 splitting the longer ones: at G = 8 each item's finish is deferred
    past the next item's first tile (at G = 4 it is not); every row against the oracle."""
    force_kernel("tc")
    rng = np.random.default_rng(47 + H)
    ctx = rng.integers(1, 700, size=600).astype(np.int32)
    ctx[::7] = 0
    ctx[5::11] = 1
    w = workloads.make_decode(f"short_items_{H}", 47, ctx, H, 8, 128, 16, "bf16")
    out, kc, vc = gpu_decode(w, max_context_len=int(ctx.max()), partition_size=256)
    check_newest_rows(w, kc, vc)
    seqs = np.concatenate([np.arange(0, 600, 13), [1, 5, 6, 7, 16, 597, 598, 599]])
    got = to_f64(out)
    assert np.all(got[ctx == 0] == 0.0)
    assert_close(got[seqs], oracle_decode(w, seqs), "bf16", f"short items H{H}")
    _errors_clear(pa)


def test_tc_kernel_bad_block_id_reads_zeros(pa, force_kernel):
    force_kernel("tc")
    w = workloads.make_decode("badid_tc", 3, np.array([300, 300], np.int32), 8, 2, 128, 16, "bf16")
    d = dev()
    kc = torch.zeros((w.num_blocks, 16, 2, 128), dtype=torch.bfloat16, device=d)
    vc = torch.zeros_like(kc)
    w.fill_cache_torch(kc, vc, include_newest=True)
    bad = w.block_tables.copy()
    bad[1, 3] = -5
    q = w.q_values(like=kc).to(torch.bfloat16).contiguous()
    out = torch.empty_like(q)
    pa.paged_attention_decode(out, q, kc, vc, torch.as_tensor(bad, device=d),
                              torch.as_tensor(w.context_lens, device=d), w.scale)
    assert pa.get_device_error() & pa.PA_DEVERR_BLOCK_ID
    ref = oracle_decode(w, [0])
    assert_close(to_f64(out)[:1], ref, "bf16", "unaffected sequence")
    assert torch.isfinite(out.float()).all()


def test_large_batch_runs_in_chunks(pa):
    # more than 1024 sequences: the tensor-core path runs independent launches
    rng = np.random.default_rng(41)
    ctx = rng.integers(0, 1200, size=2500).astype(np.int32)
    w = workloads.make_decode("big_batch", 41, ctx, 16, 4, 128, 16, "bf16")
    out, kc, vc = gpu_decode(w, max_context_len=int(ctx.max()), partition_size=256)
    seqs = np.concatenate([np.arange(0, 2500, 37), [1023, 1024, 1025, 2047, 2048, 2499]])
    ref = oracle_decode(w, seqs)
    assert_close(to_f64(out)[seqs], ref, "bf16", "2500 sequences")
    _errors_clear(pa)


def test_many_partitions_split_the_launch(pa):
    """64 sequences x 8 kv heads x 157 partitions of 128 tokens is more work items
    than one persistent grid's per-CTA tables hold: the library splits the batch
    into independent launches; every row must still match the oracle."""
    rng = np.random.default_rng(43)
    ctx = rng.integers(19000, 20000, size=64).astype(np.int32)
    ctx[[0, 17, 63]] = [20000, 1, 12345]
    w = workloads.make_decode("many_items", 43, ctx, 32, 8, 128, 16, "bf16")
    out, kc, vc = gpu_decode(w, max_context_len=20000, partition_size=128)
    seqs = [0, 1, 17, 30, 31, 32, 60, 61, 62, 63]
    assert_close(to_f64(out)[seqs], oracle_decode(w, seqs), "bf16", "split launch")
    _errors_clear(pa)
