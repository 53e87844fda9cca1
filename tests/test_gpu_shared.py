"""Sharing-aware decode (each group's shared prefix read once) against the oracle
and against the plain decode, on prefix-sharing layouts produced by forks."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_cases import assert_close, dev, oracle_decode, pa_mod, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _free_memory():
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


@pytest.fixture(scope="module")
def pa():
    return pa_mod()


def _shared_prefix_state(num_prompts):
    """Final tables of the shared-prefix sampling script (the oracle's block manager)."""
    sc = workloads.shared_prefix(num_prompts=num_prompts)
    nb = sc.pool_blocks()
    model = oracle.BlockPoolModel(nb, sc.block_size)
    for p in range(sc.num_prompts):
        model.add_seq(p)
        model.append(p, sc.prompt_len)
        for j in range(sc.samples_per_prompt):
            model.fork(p, 1000 + p * sc.samples_per_prompt + j)
        model.free_seq(p)
    for s in range(sc.num_samples):
        model.append(1000 + s, int(sc.private[s]) + 1)
    ids = np.arange(sc.num_samples) + 1000
    mb = max(len(model.block_table(int(i))) for i in ids)
    tables = np.full((sc.num_samples, mb), -1, np.int32)
    for r, i in enumerate(ids):
        t = model.block_table(int(i))
        tables[r, : len(t)] = t
    return sc, sc.workload(tables, nb)


def _run(pa, w, max_members, partition_size=0):
    d = dev()
    dt = workloads.torch_dtype(w.dtype)
    shape = (w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim)
    kc = torch.full(shape, float("nan"), dtype=dt, device=d)
    vc = torch.full(shape, float("nan"), dtype=dt, device=d)
    w.fill_cache_torch(kc, vc, include_newest=True)
    q = w.q_values(like=kc).to(dt).contiguous()
    bt = torch.as_tensor(w.block_tables, device=d)
    cl = torch.as_tensor(w.context_lens, device=d)
    pl, gm = pa.prefix_groups(w.block_tables, w.context_lens, w.block_size, max_members)
    plain = torch.full_like(q, float("nan"))
    pa.paged_attention_decode(plain, q, kc, vc, bt, cl, w.scale, partition_size=partition_size)
    shared = torch.full_like(q, float("nan"))
    pa.paged_attention_decode_shared(shared, q, kc, vc, bt, cl, torch.as_tensor(pl, device=d),
                                     torch.as_tensor(gm, device=d), w.scale, partition_size=partition_size,
                                     max_prefix_len=int(pl.max()) if pl.size else 0)
    torch.cuda.synchronize()
    return plain, shared, pl, gm


def test_shared_prefix_sampling_reads_prompts_once(pa):
    sc, w = _shared_prefix_state(num_prompts=8)
    plain, shared, pl, gm = _run(pa, w, max_members=8)
    assert gm.shape[0] == sc.num_prompts and np.all(gm >= 0)      # one group of 8 per prompt
    assert np.all(pl == 62 * 16)                                   # the 62 full prompt blocks
    assert pa.get_device_error() == 0
    a, b = to_f64(plain), to_f64(shared)
    assert np.all(np.isfinite(b))
    assert np.abs(a - b).max() <= 2e-2
    seqs = np.arange(0, w.num_seqs, 3)
    w.slot_mapping = np.full(w.num_seqs, -1, np.int32)             # contents already complete
    ref = _oracle_full(w, seqs)
    assert_close(b[seqs], ref, "bf16", "shared-prefix decode")


@pytest.mark.parametrize("partition", [0, 896, 1024, 2048])
def test_shared_prefix_batch_partition_sizes(pa, partition):
    """The bench's forked-sampling batch (32 prompts x 8 samples): the automatic
    partition (1280 tokens: one per group and kv head, covering whole contexts, so
    the per-sequence pass joins the shared partials and no merge runs), and explicit
    sizes that split the 992 shared tokens unevenly (896 + 96), keep the merge (1024)
    or cover shared and private tokens alike (2048)."""
    sc, w = _shared_prefix_state(num_prompts=32)
    pl, gm = pa.prefix_groups(w.block_tables, w.context_lens, w.block_size, 8)
    if partition == 0:
        assert pa.decode_shared_partition_size(w.num_seqs, gm.shape[0], w.num_kv_heads, int(pl.max()),
                                               int(w.block_tables.shape[1]) * w.block_size) == 1280
    plain, shared, pl, gm = _run(pa, w, max_members=8, partition_size=partition)
    assert pa.get_device_error() == 0
    b = to_f64(shared)
    assert np.all(np.isfinite(b))
    assert np.abs(to_f64(plain) - b).max() <= 2e-2
    seqs = np.arange(1, w.num_seqs, 5)
    w.slot_mapping = np.full(w.num_seqs, -1, np.int32)             # contents already complete
    assert_close(b[seqs], _oracle_full(w, seqs), "bf16", f"shared-prefix batch, partition {partition}")


@pytest.mark.parametrize("G,dtype", [(4, "bf16"), (8, "f16"), (1, "bf16"), (16, "bf16")])
def test_whole_context_partition_joins_shared_partials(pa, G, dtype):
    """A partition covering every whole context: the per-sequence pass joins the shared
    pass's partials and writes the final rows itself (no merge; at G = 16 the merge
    still runs). Groups whose members have no private tokens at all (whole context
    shared: an item with no tiles that only joins), members with one private token,
    and single sequences without a group."""
    groups = [(3, 5, 40), (4, 12, 0), (6, 20, 1), (2, 7, 300), (5, 3, 0)]
    w = workloads.make_shared_groups(91 + G, groups, 4, 8 * G, 8, 128, 16, dtype)
    mb = int(w.block_tables.shape[1]) * w.block_size
    plain, shared, pl, gm = _run(pa, w, 8, partition_size=(mb + 127) // 128 * 128)
    assert pa.get_device_error() == 0
    assert np.any((pl > 0) & (pl == w.context_lens))                  # some contexts wholly shared
    b = to_f64(shared)
    assert np.abs(to_f64(plain) - b).max() <= 2e-2
    assert_close(b, _oracle_full(w, np.arange(w.num_seqs)), dtype, f"whole-context partition G{G}")


def _oracle_full(w, seqs):
    view = w.compact_host_view(seqs, include_newest=True)
    kc = workloads.to_storage_numpy(view["key_cache"], w.dtype)
    vc = workloads.to_storage_numpy(view["value_cache"], w.dtype)
    q = workloads.to_storage_numpy(w.q_values()[np.asarray(seqs)], w.dtype)
    return oracle.paged_attention(q, kc, vc, view["block_tables"], view["context_lens"], w.scale, w.dtype,
                                  num_threads=oracle.num_host_threads())


@pytest.mark.parametrize("H,Hk,max_members,partition", [(32, 8, 8, 0), (64, 8, 16, 256), (16, 16, 4, 128)])
def test_random_groups_against_oracle(pa, H, Hk, max_members, partition):
    groups = [(3, 5, 40), (8, 40, 300), (1, 10, 50), (5, 33, 0), (12, 3, 700), (2, 70, 5)]
    w = workloads.make_shared_groups(17 + H, groups, 6, H, Hk, 128, 16, "bf16")
    plain, shared, pl, gm = _run(pa, w, max_members, partition)
    assert gm.shape[0] >= 5 and pl.max() == 70 * 16
    assert pa.get_device_error() == 0
    ref = _oracle_full(w, np.arange(w.num_seqs))
    assert_close(to_f64(shared), ref, "bf16", f"groups H{H}/{Hk}")
    assert np.abs(to_f64(plain) - to_f64(shared)).max() <= 2e-2


@pytest.mark.parametrize("cut", [1, 5, 15, 16, 37])
def test_prefix_lengths_off_block_boundaries(pa, cut):
    """A caller may pass shared-prefix lengths that end inside a block (here the
    groups' lengths minus `cut` tokens); the result is the same attention."""
    groups = [(3, 5, 40), (8, 12, 300), (2, 3, 0)]
    w = workloads.make_shared_groups(29 + cut, groups, 3, 32, 8, 128, 16, "bf16")
    d = dev()
    shape = (w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim)
    kc = torch.full(shape, float("nan"), dtype=torch.bfloat16, device=d)
    vc = torch.full(shape, float("nan"), dtype=torch.bfloat16, device=d)
    w.fill_cache_torch(kc, vc, include_newest=True)
    q = w.q_values(like=kc).to(torch.bfloat16).contiguous()
    pl, gm = pa.prefix_groups(w.block_tables, w.context_lens, w.block_size, 8)
    pl = np.where(pl > 0, np.maximum(pl - cut, 1), 0).astype(np.int32)
    out = torch.full_like(q, float("nan"))
    pa.paged_attention_decode_shared(out, q, kc, vc, torch.as_tensor(w.block_tables, device=d),
                                     torch.as_tensor(w.context_lens, device=d), torch.as_tensor(pl, device=d),
                                     torch.as_tensor(gm, device=d), w.scale, max_prefix_len=int(pl.max()))
    torch.cuda.synchronize()
    assert pa.get_device_error() == 0
    assert_close(to_f64(out), _oracle_full(w, np.arange(w.num_seqs)), "bf16", f"prefix cut {cut}")


def test_batch_above_one_launch_reads_its_own_prefix_lengths(pa):
    """More sequences than one partition launch takes (512): the launch for
    sequences 512.. must read their own shared-prefix lengths. Prefix lengths
    cycle through 2..8 blocks, so another launch's lengths would be wrong."""
    groups = [(10, 2 + (i % 7), 40) for i in range(60)]
    w = workloads.make_shared_groups(83, groups, 20, 32, 8, 128, 16, "bf16")
    assert w.num_seqs > 512
    plain, shared, pl, gm = _run(pa, w, 10)
    assert pa.get_device_error() == 0
    assert np.abs(to_f64(plain) - to_f64(shared)).max() <= 2e-2
    seqs = np.arange(500, w.num_seqs, 5)
    assert_close(to_f64(shared)[seqs], _oracle_full(w, seqs), "bf16", "shared decode, second launch")


def test_random_groups_f16(pa):
    groups = [(4, 6, 60), (6, 20, 200), (2, 3, 0)]
    w = workloads.make_shared_groups(71, groups, 4, 32, 8, 128, 16, "f16")
    plain, shared, pl, gm = _run(pa, w, 8)
    assert pa.get_device_error() == 0
    assert_close(to_f64(shared), _oracle_full(w, np.arange(w.num_seqs)), "f16", "groups f16")


def test_no_groups_equals_plain_decode(pa):
    w = workloads.llama8b_decode(num_seqs=12)
    plain, shared, pl, gm = _run(pa, w, 8)
    assert gm.shape[0] == 0 and np.all(pl == 0)
    assert np.array_equal(to_f64(plain), to_f64(shared))


def test_decode_over_beam_search_beams(pa):
    """Final beams of the beam-search script: prompt and common history shared by
    reference. Cache contents are drawn per physical slot, so the oracle reads the
    very cache the GPU reads, through the same tables."""
    import sys
    sys.path.insert(0, __file__.rsplit("/", 1)[0])
    from test_beam_search import replay
    sc = workloads.beam_search_script(k=6, steps=40)
    model = oracle.BlockPoolModel(512, sc.block_size)
    beams, _, _, _ = replay(model, sc)
    H, Hk, D, bs, nb = 32, 8, 128, sc.block_size, 512
    mb = max(len(model.block_table(b)) for b in beams)
    tables = np.full((len(beams), mb), -1, np.int32)
    lens = np.zeros(len(beams), np.int32)
    for r, b in enumerate(beams):
        t = model.block_table(b)
        tables[r, : len(t)] = t
        lens[r] = model.length(b)
    slots = np.arange(nb * bs, dtype=np.int64)
    kc = workloads.content_rows(3, 0, slots, np.zeros_like(slots), Hk * D).reshape(nb, bs, Hk, D)
    vc = workloads.content_rows(3, 1, slots, np.zeros_like(slots), Hk * D).reshape(nb, bs, Hk, D)
    q = workloads.content_rows(3, 2, np.arange(len(beams), dtype=np.int64), np.zeros(len(beams), np.int64),
                               H * D).reshape(len(beams), H, D)
    d = dev()
    kt = torch.as_tensor(kc).to(torch.bfloat16).to(d)
    vt = torch.as_tensor(vc).to(torch.bfloat16).to(d)
    qt = torch.as_tensor(q).to(torch.bfloat16).to(d)
    pl, gm = pa.prefix_groups(tables, lens, bs, max_members=8)
    assert gm.shape[0] >= 1 and pl.max() >= sc.prompt_len // bs * bs
    out = torch.empty_like(qt)
    pa.paged_attention_decode_shared(out, qt, kt, vt, torch.as_tensor(tables, device=d),
                                     torch.as_tensor(lens, device=d), torch.as_tensor(pl, device=d),
                                     torch.as_tensor(gm, device=d), 1.0 / np.sqrt(D), max_prefix_len=int(pl.max()))
    torch.cuda.synchronize()
    assert pa.get_device_error() == 0
    ref = oracle.paged_attention(workloads.to_storage_numpy(q, "bf16"), workloads.to_storage_numpy(kc, "bf16"),
                                 workloads.to_storage_numpy(vc, "bf16"), tables, lens, 1.0 / np.sqrt(D), "bf16")
    assert_close(to_f64(out), ref, "bf16", "beam-search beams")
