"""Pins of the block-manager model (oracle/allocator_model.py) to the pages."""
import numpy as np
import pytest

from conftest import read_golden
from oracle import BlockPoolModel, OutOfBlocks, UnknownSequence


def _fill(pool, seq):
    bs = pool.block_size
    return pool.length(seq) - (len(pool.block_table(seq)) - 1) * bs


def test_demo1_block_table_growth():
    g = read_golden("demo1_block_table.txt")
    nb, bs = int(g["pool_blocks"][0]), int(g["block_size"][0])
    pool = BlockPoolModel(nb, bs)
    junk = [pool.alloc() for _ in range(int(g["junk_allocated"][0]))]
    for i in g["junk_freed_indices"][0].split():
        pool.decref(junk[int(i)])
    pool.add_seq(0)
    rows = [r.split() for r in g["row"]]
    pool.append(0, int(g["prompt_tokens"][0]))
    tables = [pool.block_table(0)]
    got = [(len(pool.block_table(0)), pool.length(0), f"{_fill(pool, 0)}/{bs}")]
    for _ in range(2):
        pool.append(0, 1)
        tables.append(pool.block_table(0))
        got.append((len(pool.block_table(0)), pool.length(0), f"{_fill(pool, 0)}/{bs}"))
    assert got == [(int(r[1]), int(r[2]), r[3]) for r in rows]
    # the rest of the pool is held by the two junk blocks that stay allocated
    assert pool.num_used - len(pool.block_table(0)) == int(g["held_by_others"][0])
    t = tables[-1]
    assert any(abs(a - b) != 1 for a, b in zip(t, t[1:]))        # not contiguous
    freed = {junk[int(i)] for i in g["junk_freed_indices"][0].split()}
    assert set(t) <= freed                                      # freed blocks reused first
    # LIFO regression values of this implementation (not printed on the page)
    assert tables == [[3, 5], [3, 5], [3, 5, 7]]


def test_demo2_last_block_waste():
    g = read_golden("demo2_waste.txt")
    prompts = [int(x) for x in g["prompt_lengths"][0].split()]
    steps = int(g["decode_steps"][0])
    for row in g["waste"]:
        bs, pct = (int(x) for x in row.split())
        pool = BlockPoolModel(260 // bs + 8, bs)
        for i, L in enumerate(prompts):
            pool.add_seq(i)
            pool.append(i, L)
        for _ in range(steps):
            for i in range(len(prompts)):
                pool.append(i, 1)
        need = sum(pool.length(i) for i in range(len(prompts)))
        waste = 1 - need / (pool.num_used * bs)
        assert round(100 * waste) == pct
    # closed form for the two printed rows: 15 blocks (17.1%) and 5 blocks (37.8%)
    assert sum(-(-(L + steps) // 16) for L in prompts) == 15
    assert sum(-(-(L + steps) // 64) for L in prompts) == 5


def test_demo3_copy_on_write_count():
    g = read_golden("demo3_cow.txt")
    L, bs = int(g["prompt_tokens"][0]), int(g["block_size"][0])
    for row in g["cow"]:
        n, copies = (int(x) for x in row.split())
        pool = BlockPoolModel(256, bs)
        pool.add_seq(0)
        pool.append(0, L)
        t = pool.block_table(0)
        assert len(t) == int(g["shared_blocks"][0])
        assert L // bs == int(g["full_blocks"][0]) and L % bs == int(g["partial_tokens"][0])
        for s in range(n):
            pool.fork(0, 100 + s)
        pool.free_seq(0)
        assert all(pool.ref[b] == n for b in t)
        pairs = []
        for s in range(n):
            pairs += pool.append(100 + s, 1)[1]
        assert pool.num_cow_copies == copies == len(pairs)
        assert all(src == t[-1] for src, _ in pairs)
        assert pool.block_table(100 + n - 1)[-1] == t[-1]        # the last sample writes in place
        assert pool.ref[t[-1]] == 1
        for b in t[:-1]:
            assert pool.ref[b] == n                               # full blocks stay shared


def test_shared_prefix_workload_counts():
    # 1000-token prompt, block size 16: 62 full blocks + an 8-token partial block;
    # 8 samples per prompt -> 7 copies per prompt, 224 over 32 prompts.
    pool = BlockPoolModel(32 * 70 + 32 * 8 * 20, 16)
    total = 0
    for p in range(32):
        pool.add_seq(p)
        pool.append(p, 1000)
        assert len(pool.block_table(p)) == 63
        for s in range(8):
            pool.fork(p, 1000 + 8 * p + s)
        pool.free_seq(p)
        for s in range(8):
            total += len(pool.append(1000 + 8 * p + s, 1)[1])
    assert total == 224


def test_p1_main_status():
    g = read_golden("p1_main_status.txt")
    pool = BlockPoolModel(int(g["pool_blocks"][0]), 16)
    pool.add_seq(1)
    pool.append(1, 24)
    pool.add_seq(2)
    pool.append(2, 16)
    st = [r.split() for r in g["status"]]
    assert (pool.num_blocks, pool.num_free, pool.num_seqs) == tuple(int(x) for x in st[0][1:])
    assert len(pool.block_table(1)) == int(g["seq1_blocks"][0])
    assert len(pool.block_table(2)) == int(g["seq2_blocks"][0])
    pool.free_seq(1)
    assert (pool.num_blocks, pool.num_free, pool.num_seqs) == tuple(int(x) for x in st[1][1:])


def test_slots_follow_block_and_offset():
    pool = BlockPoolModel(10, 4)
    pool.add_seq(0)
    slots, pairs = pool.append(0, 9)
    t = pool.block_table(0)
    assert pairs == []
    assert slots == [t[p // 4] * 4 + p % 4 for p in range(9)]


# -- error behaviour where the page's teaching code has none -----------------

def test_out_of_blocks_is_an_error_and_leaves_state_unchanged():
    pool = BlockPoolModel(2, 4)
    pool.add_seq(0)
    pool.append(0, 6)
    before = (pool.block_table(0), pool.length(0), pool.num_free)
    with pytest.raises(OutOfBlocks):
        pool.append(0, 3)
    assert (pool.block_table(0), pool.length(0), pool.num_free) == before


def test_cow_with_empty_pool_is_an_error():
    pool = BlockPoolModel(1, 4)
    pool.add_seq(0)
    pool.append(0, 2)
    pool.fork(0, 1)
    with pytest.raises(OutOfBlocks):
        pool.append(1, 1)
    assert pool.num_cow_copies == 0


def test_unknown_sequence_is_an_error():
    pool = BlockPoolModel(4, 4)
    with pytest.raises(UnknownSequence):
        pool.free_seq(7)
    with pytest.raises(UnknownSequence):
        pool.append(7, 1)
    assert pool.num_seqs == 0


def test_peak_and_free_accounting():
    pool = BlockPoolModel(8, 2)
    for s in range(3):
        pool.add_seq(s)
        pool.append(s, 3)
    assert pool.num_used == 6 and pool.peak_used == 6
    pool.free_seq(1)
    assert pool.num_used == 4 and pool.peak_used == 6
    rng = np.random.default_rng(0)
    assert pool.num_free + pool.num_used == pool.num_blocks
    assert rng is not None
