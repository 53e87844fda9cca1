"""Invariants of the seeded input generators that the calls' contracts rely on."""
import numpy as np

import workloads


def test_newest_token_slots_are_those_of_the_last_position():
    """Decode with append takes, for each sequence, the slot of position ctx - 1
    (or -1 for an empty context); every generated batch provides exactly that."""
    cases = [workloads.tiny_fp32(), workloads.llama8b_decode(), workloads.long_context(),
             workloads.mixed_serving(block_size=8), workloads.mixed_serving(block_size=32),
             workloads.make_decode("empty", 7, np.array([0, 1, 16, 17, 0], np.int32), 8, 2, 128, 16, "bf16")]
    for w in cases:
        ctx = w.context_lens.astype(np.int64)
        for b in range(w.num_seqs):
            if ctx[b] == 0:
                assert w.slot_mapping[b] == -1
                continue
            pos = ctx[b] - 1
            blk = int(w.block_tables[b, pos // w.block_size])
            assert 0 <= blk < w.num_blocks
            assert w.slot_mapping[b] == blk * w.block_size + pos % w.block_size
        live = w.slot_mapping[w.slot_mapping >= 0]
        assert len(np.unique(live)) == len(live)            # no two sequences write one slot
