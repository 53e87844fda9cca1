"""Host helper that derives prefix-sharing groups from block tables (no GPU)."""
import numpy as np
import pytest

import workloads


@pytest.fixture(scope="module")
def pa():
    from __graft_entry__ import build
    build()
    import paged_kv_cache_261_gb300 as pa
    return pa


def test_groups_follow_shared_leading_blocks(pa):
    groups = [(3, 5, 40), (8, 40, 300), (1, 10, 50), (5, 33, 0), (12, 3, 700)]
    w = workloads.make_shared_groups(5, groups, 4, 32, 8, 128, 16, "bf16")
    pl, gm = pa.prefix_groups(w.block_tables, w.context_lens, 16, max_members=8)
    # member counts: 3, 8, (single: none), 5, 12 -> 8 + 4
    sizes = sorted(int((row >= 0).sum()) for row in gm)
    assert sizes == [3, 4, 5, 8, 8]
    starts = np.cumsum([0] + [g[0] for g in groups])
    for gi, (m, shared, _) in enumerate(groups):
        members = np.arange(starts[gi], starts[gi] + m)
        expect = shared * 16 if m > 1 else 0
        assert np.all(pl[members] == expect)
    assert np.all(pl[starts[-1]:] == 0)                     # the unshared sequences
    for row in gm:
        mem = row[row >= 0]
        lead = w.block_tables[mem[0], : pl[mem[0]] // 16]
        for b in mem:
            assert np.array_equal(w.block_tables[b, : pl[b] // 16], lead)


def test_shared_prompt_blocks_of_forked_samples(pa):
    import oracle
    model = oracle.BlockPoolModel(400, 16)
    model.add_seq(0)
    model.append(0, 100)                                   # 6 full blocks + 4 tokens
    for s in range(4):
        model.fork(0, 10 + s)
    model.free_seq(0)
    for s in range(4):
        model.append(10 + s, 3 + s)
    tables = np.full((4, 8), -1, np.int32)
    lens = np.zeros(4, np.int32)
    for r in range(4):
        t = model.block_table(10 + r)
        tables[r, : len(t)] = t
        lens[r] = model.length(10 + r)
    pl, gm = pa.prefix_groups(tables, lens, 16, max_members=8)
    assert gm.shape[0] == 1 and sorted(gm[0][gm[0] >= 0].tolist()) == [0, 1, 2, 3]
    assert np.all(pl == 96)                                # the partial block was copied on write


def test_bad_arguments(pa):
    with pytest.raises(pa.PagedAttnError):
        pa.prefix_groups(np.zeros((2, 2), np.int32), np.zeros(2, np.int32), 16, max_members=1)
