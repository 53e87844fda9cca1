"""Checkpoint / resume of the host allocator (pa_alloc_snapshot / pa_alloc_restore).

An allocator restored from a snapshot hands out the same blocks, slots and
copy-on-write pairs as the original for every later call; damaged images are
refused. No GPU needed."""
import struct

import numpy as np
import pytest


@pytest.fixture(scope="module")
def pa():
    from __graft_entry__ import build
    build()
    import paged_kv_cache_261_gb300 as pa
    return pa


def _step(pa, allocs, rng, state, bs):
    """One random operation applied to every allocator; their answers must agree."""
    live, held = state["live"], state["held"]
    op = int(rng.integers(0, 12))

    def each(fn):
        outs = []
        for a in allocs:
            try:
                outs.append(("ok", fn(a)))
            except pa.PagedAttnError as e:
                outs.append(("err", e.status))
        for o in outs[1:]:
            if o[0] == "ok" and outs[0][0] == "ok" and isinstance(o[1], tuple):
                assert all(np.array_equal(x, y) for x, y in zip(o[1], outs[0][1]))
            else:
                assert o == outs[0]
        return outs[0]

    if op <= 1 or not live:
        each(lambda a: a.add_seq(state["next"]))
        live.append(state["next"])
        state["next"] += 1
    elif op <= 5:
        s = live[int(rng.integers(len(live)))]
        n = int(rng.integers(0, 3 * bs + 2))
        each(lambda a: a.append(s, n))
    elif op <= 7:
        s = live[int(rng.integers(len(live)))]
        each(lambda a: a.fork(s, state["next"]))
        live.append(state["next"])
        state["next"] += 1
    elif op == 8:
        r = each(lambda a: a.alloc())                 # a block held outside any sequence
        if r[0] == "ok":
            held.append(r[1])
    elif op == 9 and held:
        b = held.pop(int(rng.integers(len(held))))
        each(lambda a: a.decref(b))
    else:
        s = live.pop(int(rng.integers(len(live))))
        each(lambda a: a.free_seq(s))


def _same(a, b, live):
    assert a.stats() == b.stats()
    for s in live:
        assert a.block_table(s) == b.block_table(s) and a.length(s) == b.length(s)
    for blk in range(a.num_blocks):
        assert a.refcount(blk) == b.refcount(blk)


@pytest.mark.parametrize("seed", range(4))
@pytest.mark.parametrize("bs", [1, 4, 16])
def test_restored_allocator_continues_identically(pa, seed, bs):
    rng = np.random.default_rng(seed * 31 + bs)
    nb = int(rng.integers(8, 48))
    a = pa.BlockAllocator(nb, bs)
    state = {"live": [], "held": [], "next": 0}
    for _ in range(150):
        _step(pa, [a], rng, state, bs)
    img = a.snapshot()
    b = pa.BlockAllocator.restore(img)
    assert b.num_blocks == nb and b.block_size == bs
    assert b.snapshot() == img
    _same(a, b, state["live"])
    for _ in range(150):
        _step(pa, [a, b], rng, state, bs)
        _same(a, b, state["live"])
    assert a.snapshot() == b.snapshot()


def test_empty_and_fresh_allocators_round_trip(pa):
    for nb, bs in [(0, 16), (5, 4)]:
        a = pa.BlockAllocator(nb, bs)
        img = a.snapshot()
        assert pa.BlockAllocator.restore(img).snapshot() == img


# ---- damaged images ------------------------------------------------------------

def _parse(img):
    assert img[:8] == b"PAALLOC1"
    off = 8
    nb, bs, peak, copies, nfree = struct.unpack_from("<5q", img, off)
    off += 40
    free = list(struct.unpack_from(f"<{nfree}i", img, off))
    off += 4 * nfree
    ref = list(struct.unpack_from(f"<{nb}i", img, off))
    off += 4 * nb
    (nseq,) = struct.unpack_from("<q", img, off)
    off += 8
    seqs = []
    for _ in range(nseq):
        sid, ln, nt = struct.unpack_from("<3q", img, off)
        off += 24
        seqs.append([sid, ln, list(struct.unpack_from(f"<{nt}i", img, off))])
        off += 4 * nt
    assert off == len(img)
    return {"nb": nb, "bs": bs, "peak": peak, "copies": copies, "free": free, "ref": ref, "seqs": seqs}


def _pack(d):
    out = b"PAALLOC1" + struct.pack("<5q", d["nb"], d["bs"], d["peak"], d["copies"], len(d["free"]))
    out += struct.pack(f"<{len(d['free'])}i", *d["free"]) + struct.pack(f"<{d['nb']}i", *d["ref"])
    out += struct.pack("<q", len(d["seqs"]))
    for sid, ln, t in d["seqs"]:
        out += struct.pack("<3q", sid, ln, len(t)) + struct.pack(f"<{len(t)}i", *t)
    return out


@pytest.fixture(scope="module")
def image(pa):
    """Two forked sequences sharing full blocks, a partial last block, a held block."""
    a = pa.BlockAllocator(16, 4)
    a.add_seq(3)
    a.append(3, 10)
    a.fork(3, 7)
    a.append(7, 1)                                   # copy-on-write of the shared partial block
    a.alloc()
    return a.snapshot()


def _refused(pa, img):
    with pytest.raises(pa.PagedAttnError) as e:
        pa.BlockAllocator.restore(img)
    assert e.value.status == pa.PA_ERR_INVALID_ARG


def test_the_parser_reads_the_image_back(image):
    d = _parse(image)
    assert _pack(d) == image
    assert [s[0] for s in d["seqs"]] == [3, 7] and d["copies"] == 1


def test_damaged_images_are_refused(pa, image):
    d0 = _parse(image)

    def damaged(fn):
        d = _parse(image)
        fn(d)
        return _pack(d)

    _refused(pa, b"PAALLOC2" + image[8:])
    for k in range(len(image)):
        _refused(pa, image[:k])
    _refused(pa, image + b"\0")
    shared = next(b for b in range(d0["nb"]) if d0["ref"][b] == 2)
    in_table = d0["seqs"][0][2][0]
    _refused(pa, damaged(lambda d: d["free"].__setitem__(1, d["free"][0])))           # a free id twice
    _refused(pa, damaged(lambda d: d["ref"].__setitem__(d["free"][-1], 1)))           # a free block counted
    _refused(pa, damaged(lambda d: d["ref"].__setitem__(shared, 1)))                  # count below holders
    _refused(pa, damaged(lambda d: d["ref"].__setitem__(in_table, 0)))                # a held block at 0
    _refused(pa, damaged(lambda d: d["seqs"][0][2].__setitem__(0, d["nb"])))          # id out of range
    _refused(pa, damaged(lambda d: d["seqs"].reverse()))                              # ids not increasing
    _refused(pa, damaged(lambda d: d["seqs"][1].__setitem__(1, d["seqs"][1][1] + 4)))  # table too short
    _refused(pa, damaged(lambda d: d["seqs"][0].__setitem__(1, -1)))                  # negative length
    _refused(pa, damaged(lambda d: d.__setitem__("peak", 0)))                         # peak below use
    _refused(pa, damaged(lambda d: d.__setitem__("bs", 0)))


def test_a_count_above_its_tables_is_a_held_block(pa, image):
    d = _parse(image)
    blk = d["seqs"][0][2][0]
    d["ref"][blk] += 1                               # one more holder outside the sequences
    b = pa.BlockAllocator.restore(_pack(d))
    assert b.refcount(blk) == d["ref"][blk]
