"""Host-side block bookkeeping for the decode driver: a free list, reference
counts, on-demand block append and block-level copy-on-write.

Semantics ("PagedAttention 核心创新深度分析" §3.2 BlockPool;
"Visual reading: paged-attention-kv-cache", Figure 8; "Infra:
PagedAttention", copy-on-write figure):
  * taking a block pops the head of the free list and gives it one reference;
  * sharing a block (fork) adds a reference; releasing drops one, and a block
    with no references goes to the tail of the free list;
  * a sequence takes a new block only when its last block is full;
  * a write into a block with more than one reference first moves the writer
    to a fresh copy (the caller runs pa_copy_blocks on the returned pairs
    before the KV write), releasing one reference on the original.

With a sliding window of W tokens, `release_skipped` frees the leading
blocks that hold no token of the window (same page, §3.2 allocate_slots,
phase 1, and §3.3.1: skipped blocks = skipped tokens // B); their table
entries become -1, which the windowed attention call never reads.

The per-step work (`prepare_decode_step`) is batched: it returns, for a list
of sequences each appending one token, the positions, the copy pairs and the
updated dense block-table rows, ready to upload in one copy each.
"""
from __future__ import annotations

from collections import deque
from typing import Dict, List, Sequence, Tuple

import numpy as np


class BlockPool:
    def __init__(self, num_blocks: int, block_size: int, free_order: Sequence[int] | None = None):
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)
        order = range(self.num_blocks) if free_order is None else free_order
        self._free: deque = deque(int(b) for b in order)
        if len(self._free) != self.num_blocks:
            raise ValueError("free_order must list every block once")
        self.refcount = np.zeros(self.num_blocks, dtype=np.int32)
        self.blocks: Dict[object, List[int]] = {}
        self.num_tokens: Dict[object, int] = {}

    # ---- primitive moves ---------------------------------------------------
    def num_free(self) -> int:
        return len(self._free)

    def _pop(self) -> int:
        if not self._free:
            raise MemoryError("KV block pool exhausted")
        blk = self._free.popleft()
        self.refcount[blk] = 1
        return blk

    def _drop(self, blk: int) -> None:
        self.refcount[blk] -= 1
        if self.refcount[blk] == 0:
            self._free.append(blk)

    # ---- sequence lifecycle -------------------------------------------------
    def add_sequence(self, seq, num_tokens: int) -> List[int]:
        """Blocks for a new sequence holding num_tokens tokens."""
        if seq in self.blocks:
            raise KeyError(f"sequence {seq!r} exists")
        need = (num_tokens + self.block_size - 1) // self.block_size
        if need > len(self._free):
            raise MemoryError("KV block pool exhausted")
        self.blocks[seq] = [self._pop() for _ in range(need)]
        self.num_tokens[seq] = int(num_tokens)
        return list(self.blocks[seq])

    def fork(self, parent, child) -> None:
        """child starts as a copy of parent's table; every block gains a
        reference."""
        if child in self.blocks:
            raise KeyError(f"sequence {child!r} exists")
        row = self.blocks[parent]
        self.blocks[child] = list(row)
        self.num_tokens[child] = self.num_tokens[parent]
        held = np.asarray([b for b in row if b >= 0], dtype=np.int64)
        np.add.at(self.refcount, held, 1)

    def release(self, seq) -> None:
        for blk in self.blocks.pop(seq):
            if blk >= 0:
                self._drop(blk)
        del self.num_tokens[seq]

    def release_skipped(self, seq, window: int) -> List[int]:
        """Drop one reference on each leading block of seq that holds no
        token of its last `window` tokens (window <= 0: none) and mark the
        entry -1. Returns the blocks released, in table order."""
        n = self.num_tokens[seq]
        if window <= 0 or n <= window:
            return []
        skip = (n - window) // self.block_size
        row = self.blocks[seq]
        out = []
        for i in range(min(skip, len(row))):
            if row[i] >= 0:
                out.append(row[i])
                self._drop(row[i])
                row[i] = -1
        return out

    # ---- one decode step ----------------------------------------------------
    def prepare_decode_step(self, seqs: Sequence) -> Tuple[np.ndarray, List[Tuple[int, int]]]:
        """Reserve one new token slot for each sequence, in order.

        Returns (positions int64 [len(seqs)], copy pairs [(src, dst), ...]).
        The new token of seqs[i] is at position positions[i]; its slot comes
        from the slot-mapping kernel applied to the updated tables."""
        B = self.block_size
        positions = np.empty(len(seqs), dtype=np.int64)
        pairs: List[Tuple[int, int]] = []
        for i, seq in enumerate(seqs):
            n = self.num_tokens[seq]
            row = self.blocks[seq]
            idx, filled = divmod(n, B)
            if filled == 0 and idx == len(row):
                row.append(self._pop())
            else:
                blk = row[idx]
                if self.refcount[blk] > 1:
                    fresh = self._pop()
                    self._drop(blk)
                    row[idx] = fresh
                    pairs.append((blk, fresh))
            positions[i] = n
            self.num_tokens[seq] = n + 1
        return positions, pairs

    def table_rows(self, seqs: Sequence, width: int | None = None) -> np.ndarray:
        """Dense int32 [len(seqs), width] block table; -1 past each row."""
        w = width or max((len(self.blocks[s]) for s in seqs), default=1)
        out = np.full((len(seqs), w), -1, dtype=np.int32)
        for i, s in enumerate(seqs):
            row = self.blocks[s]
            if len(row) > w:
                raise ValueError("table width too small")
            out[i, :len(row)] = row
        return out

    def saving(self, seqs: Sequence | None = None) -> float:
        """Share of logical block mappings served by an already-counted
        physical block."""
        seqs = list(self.blocks) if seqs is None else seqs
        rows = [[b for b in self.blocks[s] if b >= 0] for s in seqs]
        logical = sum(map(len, rows))
        unique = len(set().union(*map(set, rows))) if rows else 0
        return 0.0 if logical == 0 else (logical - unique) / logical
