"""Block lifetime: copy-on-write and release of shared KV blocks, sequential.

Sources:

* INMS walkthrough §2.2: blocks are shared by fingerprint with a reference
  count; every shared block is read-only; when a sequence is about to write
  into a block that others also reference, it gets a private copy of the
  block and writes there, while the other referrers keep their view
  (write_to_block: if ref_count[old] > 1, copy the block, decrement the old
  block's count, map the sequence's position to the copy; else write in
  place).  Blocks whose count reaches zero are reclaimed.
* INMS walkthrough §3.3: the sequence-destroy interface decrements the counts
  of the sequence's blocks and reclaims what becomes unused.
* INMS walkthrough §5.3: a missed release leaks shared blocks; every path
  must return the counts to zero.

Readings (the pages give the rule, not the bookkeeping): unused blocks sit on
a free stack; the stack starts with every block of count zero pushed in
descending id order, so the smallest free id is on top; a write batch is
applied in list order, each write exactly as write_to_block; a release call
first decrements every referenced block of every released sequence, then
pushes the blocks that reached zero in descending id order, and clears the
released rows to -1.  A block is referenced by a row at logical block b when
b < ceil(seq_len / block_tokens).

Test infrastructure only: nothing under shared_paged_kv_gb300/ imports this.
"""
from __future__ import annotations

import numpy as np


class BlockManager:
    """Sequential reference implementation of the block bookkeeping."""

    def __init__(self, block_table, seq_len, refcount, block_tokens: int, slabs=None):
        self.table = np.array(block_table, dtype=np.int32, copy=True)
        self.seq_len = np.array(seq_len, dtype=np.int64, copy=True)
        self.ref = np.array(refcount, dtype=np.int64, copy=True)
        self.B = block_tokens
        # slabs: list of arrays [capacity][...] copied along with a block
        self.slabs = [np.array(s, copy=True) for s in (slabs or [])]
        zero = [p for p in range(len(self.ref)) if self.ref[p] == 0]
        self.free = sorted(zero, reverse=True)   # top of the stack = last element = smallest id
        self.errors = set()

    def n_blocks(self, a: int) -> int:
        return int(-(-int(self.seq_len[a]) // self.B))

    def write_to_block(self, a: int, b: int) -> None:
        """The pages' write_to_block: copy-on-write when the block is shared."""
        old = int(self.table[a, b])
        if old < 0 or old >= len(self.ref):
            self.errors.add("block_id")
            return
        if self.ref[old] > 1:
            if not self.free:
                self.errors.add("capacity")
                return
            new = self.free.pop()
            for s in self.slabs:
                s[new] = s[old]
            self.ref[old] -= 1
            self.ref[new] = 1
            self.table[a, b] = new
        # else: written in place

    def write_batch(self, seqs, blocks) -> None:
        for a, b in zip(seqs, blocks):
            self.write_to_block(int(a), int(b))

    def release(self, seqs) -> None:
        """Destroy the given sequences: decrement, then reclaim zeros."""
        touched = set()
        for a in seqs:
            a = int(a)
            for b in range(self.n_blocks(a)):
                p = int(self.table[a, b])
                self.ref[p] -= 1
                if self.ref[p] < 0:
                    self.errors.add("refcount")
                touched.add(p)
            self.table[a, :] = -1
            self.seq_len[a] = 0
        freed = sorted((p for p in touched if self.ref[p] == 0), reverse=True)
        self.free.extend(freed)

    def referenced_counts(self) -> np.ndarray:
        """References per block counted from the table (the invariant)."""
        cnt = np.zeros(len(self.ref), dtype=np.int64)
        for a in range(self.table.shape[0]):
            for b in range(self.n_blocks(a)):
                cnt[int(self.table[a, b])] += 1
        return cnt
