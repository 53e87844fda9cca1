"""Beam search on the block manager: fork, prune and copy-on-write of the last
block ("CS349E lecture 7: 01_paged_attention.py", demo 4), replayed on the
library allocator and on the oracle's model with identical results (no GPU)."""
import numpy as np
import pytest

import oracle
import workloads


@pytest.fixture(scope="module")
def pa():
    from __graft_entry__ import build
    build()
    import paged_kv_cache_261_gb300 as pa
    return pa


def _num_used(alloc):
    return alloc.stats().num_used if hasattr(alloc, "stats") else alloc.num_used


def replay(alloc, sc):
    """Run the script; returns per-step (blocks used, unshared blocks) and copies."""
    bs = sc.block_size
    alloc.add_seq(0)
    alloc.append(0, sc.prompt_len)
    beams = [0]
    next_id = 1
    used, unshared, cow = [], [], []
    for parents in sc.parents:
        children = []
        taken = set()
        for p in parents:
            parent = beams[p]
            if p in taken:
                child = next_id
                next_id += 1
                alloc.fork(parent, child)
            else:
                taken.add(p)
                child = parent                     # the first child continues the parent itself
            children.append(child)
        for i, b in enumerate(beams):
            if i not in taken:
                alloc.free_seq(b)                  # pruned beam
        step_pairs = []
        for c in children:
            step_pairs += [tuple(x) for x in np.asarray(alloc.append(c, 1)[1]).reshape(-1, 2).tolist()]
        cow.append(step_pairs)
        beams = children
        lens = [alloc.length(b) for b in beams]
        used.append(_num_used(alloc))
        unshared.append(sum(-(-L // bs) for L in lens))
    return beams, used, unshared, cow


@pytest.mark.parametrize("k", [2, 4, 6])
def test_library_allocator_matches_model(pa, k):
    sc = workloads.beam_search_script(k=k)
    model = oracle.BlockPoolModel(256, sc.block_size)
    lib = pa.BlockAllocator(256, sc.block_size)
    bm, um, sm, cm = replay(model, sc)
    bl, ul, sl, cl = replay(lib, sc)
    assert cm == cl and um == ul and sm == sl
    for a, b in zip(bm, bl):
        assert model.block_table(a) == lib.block_table(b)


@pytest.mark.parametrize("k", [2, 4, 6])
def test_beam_invariants_and_savings(pa, k):
    sc = workloads.beam_search_script(k=k)
    model = oracle.BlockPoolModel(256, sc.block_size)
    beams, used, unshared, cow = replay(model, sc)
    # every reference is a table entry; every used block is referenced
    refs = sum(len(model.block_table(b)) for b in beams)
    assert refs == sum(model.ref)
    assert model.num_used == sum(1 for r in model.ref if r > 0)
    # a copy only happens when a beam writes into a partially filled shared block,
    # and copies exactly one block (block_size tokens)
    for s, pairs in enumerate(cow):
        pos = sc.prompt_len + s
        if pos % sc.block_size == 0:
            assert pairs == []                     # the token starts a fresh block
        assert len(pairs) <= sc.k - 1
    # sharing never needs more blocks than one private copy per beam
    assert all(u <= v for u, v in zip(used, unshared))
    saving = 1 - sum(used) / sum(unshared)
    assert saving > 0.3                            # shared prompt and common beam history
    # paged copying moves far fewer tokens than copying each child's whole cache
    copied_paged = sum(len(p) for p in cow) * sc.block_size
    copied_full = 0
    for s, parents in enumerate(sc.parents):
        seen = set()
        for p in parents:
            if p in seen:
                copied_full += sc.prompt_len + s
            seen.add(p)
    assert copied_paged < copied_full


def test_single_beam_never_copies(pa):
    sc = workloads.BeamScript(seed=0, prompt_len=20, steps=30, k=1, block_size=16, parents=[[0]] * 30)
    model = oracle.BlockPoolModel(16, 16)
    beams, used, unshared, cow = replay(model, sc)
    assert all(p == [] for p in cow) and used == unshared
