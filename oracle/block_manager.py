"""Host-side block bookkeeping oracle: free queue, reference counts, on-demand
append and block-level copy-on-write.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

Follows, in order:
  * [P1] §3.2 BlockPool: allocation pops from the head of the free queue and
    sets the reference count to 1 (get_new_blocks); sharing adds one reference
    (touch); freeing drops one reference and a block whose count reaches zero
    is appended to the queue tail (free_blocks).
  * [P2] "7-token prompt" example and [P3] "按需分配": a new block is taken
    only when the sequence's last block is full.
  * [P2] Figure 8 / [P4] "共享前缀，分叉时 Copy-on-write": a writer that finds
    its target block referenced more than once copies that one block to a
    fresh block, moves its own table entry to the copy, drops one reference
    on the original, then writes; a writer that is the last holder writes in
    place.

  * [P1] §3.2 allocate_slots phase 1 and §3.3.1: with a sliding window, the
    blocks before the skipped-token count // B hold no attended token and
    are released (remove_skipped).

Readings: no block id is reserved as a null block (the pages' figures use P0
as an ordinary block); the free order is FIFO as in [P1]'s free_blocks.
"""
from __future__ import annotations

from collections import deque


class OracleBlockManager:
    def __init__(self, num_blocks: int, block_size: int, free_order=None):
        self.num_blocks = num_blocks
        self.block_size = block_size
        order = list(range(num_blocks)) if free_order is None else list(free_order)
        assert sorted(order) == list(range(num_blocks))
        self.free = deque(order)
        self.ref = [0] * num_blocks
        self.tables: dict = {}
        self.lens: dict = {}

    # -- [P1] §3.2.1 get_new_blocks -------------------------------------
    def _take(self) -> int:
        if not self.free:
            raise ValueError("out of blocks")
        b = self.free.popleft()
        assert self.ref[b] == 0
        self.ref[b] = 1
        return b

    # -- [P1] §3.2.4 free_blocks ----------------------------------------
    def _release(self, b: int):
        self.ref[b] -= 1
        assert self.ref[b] >= 0
        if self.ref[b] == 0:
            self.free.append(b)

    def allocate(self, seq, num_tokens: int):
        """Blocks for a new sequence's first num_tokens tokens (prefill)."""
        n = -(-num_tokens // self.block_size)
        self.tables[seq] = [self._take() for _ in range(n)]
        self.lens[seq] = num_tokens
        return list(self.tables[seq])

    def fork(self, parent, child):
        """child shares every block of parent ([P1] §3.2.3 touch: one more
        reference per shared block)."""
        self.tables[child] = list(self.tables[parent])
        self.lens[child] = self.lens[parent]
        for b in self.tables[child]:
            if b is not None:
                self.ref[b] += 1

    def append_slot(self, seq):
        """Reserve the slot for seq's next token. Returns (slot, cow) where
        cow is a (src, dst) block pair to copy before writing, or None."""
        B = self.block_size
        L = self.lens[seq]
        table = self.tables[seq]
        lb = L // B
        cow = None
        if lb == len(table):                 # last block full: take a new one
            table.append(self._take())
        elif self.ref[table[lb]] > 1:        # shared block: copy-on-write
            src = table[lb]
            dst = self._take()
            self._release(src)
            table[lb] = dst
            cow = (src, dst)
        self.lens[seq] = L + 1
        return table[lb] * B + (L - lb * B), cow

    def remove_skipped(self, seq, window: int):
        """Release the leading blocks of seq that hold only tokens before its
        window (the last `window` tokens); their entries become None.
        Returns the released ids in table order."""
        from .paged_attention import skipped_blocks
        table = self.tables[seq]
        gone = []
        for i in range(skipped_blocks(self.lens[seq], window, self.block_size)):
            if table[i] is not None:
                gone.append(table[i])
                self._release(table[i])
                table[i] = None
        return gone

    def free_seq(self, seq):
        for b in self.tables.pop(seq):
            if b is not None:
                self._release(b)
        self.lens.pop(seq)
