"""Host metadata parity: the library's C++ allocator against the oracle's model.

Bit-exact block tables, slots and copy-on-write pairs over random operation
sequences, plus the pages' worked examples run through the library allocator.
No GPU needed.
"""
import numpy as np
import pytest

from conftest import read_golden
from oracle import BlockPoolModel, OutOfBlocks, UnknownSequence


@pytest.fixture(scope="module")
def pa():
    from __graft_entry__ import build
    build()
    import paged_kv_cache_261_gb300 as pa
    return pa


def _same_state(lib_alloc, model, seqs):
    st = lib_alloc.stats()
    assert (st.num_blocks, st.num_free, st.num_used, st.peak_used, st.num_cow_copies, st.num_seqs) == (
        model.num_blocks, model.num_free, model.num_used, model.peak_used, model.num_cow_copies,
        model.num_seqs)
    for s in seqs:
        assert lib_alloc.block_table(s) == model.block_table(s)
        assert lib_alloc.length(s) == model.length(s)
    for b in range(model.num_blocks):
        assert lib_alloc.refcount(b) == model.ref[b]


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("bs", [1, 4, 16])
def test_random_operations_match_the_model(pa, seed, bs):
    rng = np.random.default_rng(seed * 100 + bs)
    nb = int(rng.integers(8, 64))
    lib_alloc = pa.BlockAllocator(nb, bs)
    model = BlockPoolModel(nb, bs)
    live, next_id = [], 0
    for _ in range(300):
        op = rng.integers(0, 10)
        if op <= 1 or not live:
            lib_alloc.add_seq(next_id)
            model.add_seq(next_id)
            live.append(next_id)
            next_id += 1
        elif op <= 5:
            s = live[int(rng.integers(len(live)))]
            n = int(rng.integers(0, 3 * bs + 2))
            try:
                ms, mp = model.append(s, n)
            except OutOfBlocks:
                with pytest.raises(pa.PagedAttnError) as e:
                    lib_alloc.append(s, n)
                assert e.value.status == pa.PA_ERR_OUT_OF_BLOCKS
                continue
            ls, lp = lib_alloc.append(s, n)
            assert ls.tolist() == ms
            assert [tuple(p) for p in lp.tolist()] == mp
        elif op <= 7:
            s = live[int(rng.integers(len(live)))]
            lib_alloc.fork(s, next_id)
            model.fork(s, next_id)
            live.append(next_id)
            next_id += 1
        else:
            s = live.pop(int(rng.integers(len(live))))
            lib_alloc.free_seq(s)
            model.free_seq(s)
        _same_state(lib_alloc, model, live)
    if live:
        mb = max(len(model.block_table(s)) for s in live) + 2
        tables, lens = lib_alloc.export(live, mb)
        for i, s in enumerate(live):
            t = model.block_table(s)
            assert tables[i, : len(t)].tolist() == t and np.all(tables[i, len(t):] == -1)
            assert lens[i] == model.length(s)


def test_demo1_through_the_library(pa):
    g = read_golden("demo1_block_table.txt")
    a = pa.BlockAllocator(int(g["pool_blocks"][0]), int(g["block_size"][0]))
    junk = [a.alloc() for _ in range(int(g["junk_allocated"][0]))]
    for i in g["junk_freed_indices"][0].split():
        a.decref(junk[int(i)])
    a.add_seq(0)
    a.append(0, int(g["prompt_tokens"][0]))
    counts = [len(a.block_table(0))]
    for _ in range(2):
        a.append(0, 1)
        counts.append(len(a.block_table(0)))
    assert counts == [int(r.split()[1]) for r in g["row"]]
    assert a.stats().num_used - counts[-1] == int(g["held_by_others"][0])


def test_demo3_cow_through_the_library(pa):
    g = read_golden("demo3_cow.txt")
    for row in g["cow"]:
        n, copies = (int(x) for x in row.split())
        a = pa.BlockAllocator(256, int(g["block_size"][0]))
        a.add_seq(0)
        a.append(0, int(g["prompt_tokens"][0]))
        for s in range(n):
            a.fork(0, 100 + s)
        a.free_seq(0)
        got = sum(len(a.append(100 + s, 1)[1]) for s in range(n))
        assert got == copies == a.stats().num_cow_copies


def test_p1_main_status_through_the_library(pa):
    g = read_golden("p1_main_status.txt")
    a = pa.BlockAllocator(int(g["pool_blocks"][0]), 16)
    a.add_seq(1)
    a.append(1, 24)
    a.add_seq(2)
    a.append(2, 16)
    st = [tuple(int(x) for x in r.split()[1:]) for r in g["status"]]
    s = a.stats()
    assert (s.num_blocks, s.num_free, s.num_seqs) == st[0]
    a.free_seq(1)
    s = a.stats()
    assert (s.num_blocks, s.num_free, s.num_seqs) == st[1]


def test_errors_are_reported_not_hidden(pa):
    a = pa.BlockAllocator(1, 4)
    with pytest.raises(pa.PagedAttnError) as e:
        a.free_seq(3)                      # the teaching code silently creates an entry here
    assert e.value.status == pa.PA_ERR_UNKNOWN_SEQ
    a.add_seq(0)
    with pytest.raises(pa.PagedAttnError) as e:
        a.add_seq(0)
    assert e.value.status == pa.PA_ERR_EXISTS
    a.append(0, 2)
    a.fork(0, 1)
    with pytest.raises(pa.PagedAttnError) as e:
        a.append(1, 1)                     # copy-on-write with an empty free list
    assert e.value.status == pa.PA_ERR_OUT_OF_BLOCKS
    assert a.length(1) == 2 and a.stats().num_cow_copies == 0
    with pytest.raises(pa.PagedAttnError):
        a.export([0, 1], 0)               # table longer than the row
    with pytest.raises(pa.PagedAttnError):
        a.decref(5)
    assert UnknownSequence is not None
