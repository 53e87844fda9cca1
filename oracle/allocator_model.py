"""Reference model of the host-side block manager -- TEST INFRASTRUCTURE.

Only tests, the smoke check and the benchmark's CPU-baseline leg use this
module. It shares no code with the C++ allocator of the library; a test drives
both with the same operations and requires identical block tables, slots and
copy-on-write pairs.

Followed passages (web pages, by title and section):
  "PagedAttention实现" (ainanfeng.cn), section "PagedAttention管理器":
    - the pool starts with every block id pushed, in order 0..N-1, onto a free
      stack; allocation takes the most recently pushed id (LIFO) and sets its
      reference count to 1;
    - a write goes to page ``pos // block_size`` at offset ``pos % block_size``;
    - cow_write: when the target block's reference count is above 1, a fresh
      block takes a copy of the whole block, the sequence's table is repointed
      to it, and the old block's count drops by one;
    - free_sequence drops every block's count and returns blocks that reach 0
      to the free stack.
  "CS349E lecture 7: 01_paged_attention.py", demo 1 (a block is allocated only
    when a token falls on a block boundary), demo 3 (forked samples share the
    prompt's blocks by reference count; each of the first n-1 samples to write
    into the shared partial block copies it, the last writes in place).

Readings beyond the page (also listed in the design notes): allocation failure
and unknown sequence ids raise instead of printing or silently creating state
(the page's teaching code has neither check); an append is all-or-nothing.
"""
from __future__ import annotations


class AllocatorError(Exception):
    pass


class OutOfBlocks(AllocatorError):
    pass


class UnknownSequence(AllocatorError):
    pass


class BlockPoolModel:
    def __init__(self, num_blocks: int, block_size: int):
        if num_blocks < 0 or block_size <= 0:
            raise AllocatorError("bad pool shape")
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.free = list(range(num_blocks))       # stack: top is free[-1]
        self.ref = [0] * num_blocks
        self.tables: dict[int, list[int]] = {}
        self.lengths: dict[int, int] = {}
        self.num_cow_copies = 0
        self.peak_used = 0

    # -- pool level -------------------------------------------------------
    @property
    def num_free(self) -> int:
        return len(self.free)

    @property
    def num_used(self) -> int:
        return self.num_blocks - len(self.free)

    def alloc(self) -> int:
        if not self.free:
            raise OutOfBlocks("no free blocks")
        b = self.free.pop()
        self.ref[b] = 1
        self.peak_used = max(self.peak_used, self.num_used)
        return b

    def decref(self, b: int) -> None:
        if not (0 <= b < self.num_blocks) or self.ref[b] <= 0:
            raise AllocatorError("decref of a free or unknown block")
        self.ref[b] -= 1
        if self.ref[b] == 0:
            self.free.append(b)

    # -- sequence level ---------------------------------------------------
    def add_seq(self, seq_id: int) -> None:
        if seq_id in self.tables:
            raise AllocatorError("sequence exists")
        self.tables[seq_id] = []
        self.lengths[seq_id] = 0

    def _table(self, seq_id: int) -> list[int]:
        if seq_id not in self.tables:
            raise UnknownSequence(seq_id)
        return self.tables[seq_id]

    def fork(self, parent: int, child: int) -> None:
        t = self._table(parent)
        if child in self.tables:
            raise AllocatorError("sequence exists")
        for b in t:
            self.ref[b] += 1
        self.tables[child] = list(t)
        self.lengths[child] = self.lengths[parent]

    def blocks_needed(self, seq_id: int, n_tokens: int) -> int:
        t = self._table(seq_id)
        length = self.lengths[seq_id]
        bs = self.block_size
        need = 0
        if n_tokens > 0 and length % bs != 0 and self.ref[t[length // bs]] > 1:
            need += 1                                  # copy-on-write of the partial block
        end = length + n_tokens
        need += (end + bs - 1) // bs - (length + bs - 1) // bs
        return need

    def append(self, seq_id: int, n_tokens: int):
        """Append n_tokens positions. Returns (slots, cow_pairs)."""
        t = self._table(seq_id)
        if n_tokens < 0:
            raise AllocatorError("negative token count")
        if self.blocks_needed(seq_id, n_tokens) > len(self.free):
            raise OutOfBlocks("no free blocks")
        bs = self.block_size
        slots, pairs = [], []
        for _ in range(n_tokens):
            pos = self.lengths[seq_id]
            page = pos // bs
            if page == len(t):
                t.append(self.alloc())
            elif self.ref[t[page]] > 1:
                old = t[page]
                new = self.alloc()
                pairs.append((old, new))
                t[page] = new
                self.ref[old] -= 1
                self.num_cow_copies += 1
            slots.append(t[page] * bs + pos % bs)
            self.lengths[seq_id] = pos + 1
        return slots, pairs

    def free_seq(self, seq_id: int) -> None:
        t = self._table(seq_id)
        for b in t:
            self.decref(b)
        del self.tables[seq_id]
        del self.lengths[seq_id]

    def block_table(self, seq_id: int) -> list[int]:
        return list(self._table(seq_id))

    def length(self, seq_id: int) -> int:
        self._table(seq_id)
        return self.lengths[seq_id]

    @property
    def num_seqs(self) -> int:
        return len(self.tables)
