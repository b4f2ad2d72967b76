"""Block-manager oracle — test infrastructure only.

A plain Python model of the host bookkeeping around a paged KV cache, written
from the pages so that a reader can check it line by line:

- Blocks of B tokens in one pool; a sequence's block table maps its logical
  block i (tokens i*B .. i*B+B-1) to a physical block ("PagedAttention — Math
  + Memory Model", section "PagedAttention: blocks and the block table").
- Allocation on demand: a sequence starts with no blocks and takes one free
  block from the pool when it fills its last block (same section).
- Sharing by reference with a per-block reference count; a block returns to
  the free pool the moment its count reaches zero (same page, section
  "Copy-on-write: sharing blocks across samples").
- Copy-on-write: writing into a block others still share copies that one
  block to a fresh block, decrements the original's count, and the writer
  continues in its copy (same section). fork() gives a child the parent's
  table with every count raised by one (same section: samples and beams of
  one prompt point at the same blocks).
- Prefix caching: identical prompt prefixes share their physical blocks
  across requests ("KV-Cache Optimization & PagedAttention for Long-Context
  Agents", section "Key KV-Cache Optimization Principles", item 3). A full
  prefix block is identified by a caller-given hash; a hit shares the
  registered block, a miss allocates one and registers it.

Readings where the pages are silent:
- Free-pool order: the most recently freed block is taken first; a fresh pool
  hands out blocks 0, 1, 2, ... A sequence's blocks are freed in table order.
- A hash is registered only for blocks allocated for a prefix, and dropped
  when the block is freed.
- An append that needs more blocks than are free fails and changes nothing.
"""
from __future__ import annotations

from typing import Dict, List, Sequence, Tuple


class OutOfBlocks(RuntimeError):
    pass


class BlockManagerOracle:
    def __init__(self, num_blocks: int, block_size: int):
        self.B = block_size
        self.num_blocks = num_blocks
        self.free: List[int] = list(range(num_blocks - 1, -1, -1))   # pop() -> 0, 1, 2, ...
        self.ref: List[int] = [0] * num_blocks
        self.tables: Dict[int, List[int]] = {}
        self.lens: Dict[int, int] = {}
        self.by_hash: Dict[int, int] = {}
        self.hash_of: Dict[int, int] = {}

    # ---------------------------------------------------------------- helpers
    def _take(self) -> int:
        b = self.free.pop()
        self.ref[b] = 1
        return b

    def _drop(self, b: int) -> None:
        self.ref[b] -= 1
        if self.ref[b] == 0:
            self.free.append(b)
            h = self.hash_of.pop(b, None)
            if h is not None:
                del self.by_hash[h]

    # ---------------------------------------------------------------- calls
    def add_sequence(self, seq: int, prefix_hashes: Sequence[int] = ()) -> List[bool]:
        """New sequence whose first len(prefix_hashes) blocks are full prompt
        blocks identified by hash. Returns, per block, whether it was a hit."""
        assert seq not in self.tables
        misses = sum(1 for h in prefix_hashes if h not in self.by_hash)
        if misses > len(self.free):
            raise OutOfBlocks(f"{misses} blocks needed, {len(self.free)} free")
        table, hits = [], []
        for h in prefix_hashes:
            if h in self.by_hash:
                b = self.by_hash[h]
                self.ref[b] += 1
                hits.append(True)
            else:
                b = self._take()
                self.by_hash[h] = b
                self.hash_of[b] = h
                hits.append(False)
            table.append(b)
        self.tables[seq] = table
        self.lens[seq] = len(prefix_hashes) * self.B
        return hits

    def append(self, seq: int, n: int) -> Tuple[List[int], List[Tuple[int, int]]]:
        """Room for n new tokens at the end of `seq`. Returns their slots
        (block * B + offset) and the (src, dst) block copies that must run
        before the tokens are written."""
        table, L, B = self.tables[seq], self.lens[seq], self.B
        # blocks this call takes: new blocks for the tokens past the last
        # block, plus one copy if the first write lands in a shared block
        new_blocks = -(-(L + n) // B) - len(table)
        cow = n > 0 and L % B != 0 and self.ref[table[-1]] > 1
        if new_blocks + cow > len(self.free):
            raise OutOfBlocks(f"{new_blocks + cow} blocks needed, {len(self.free)} free")
        slots, copies = [], []
        for _ in range(n):
            if L % B == 0:
                table.append(self._take())
            elif self.ref[table[-1]] > 1:
                src = table[-1]
                dst = self._take()
                copies.append((src, dst))
                self._drop(src)
                table[-1] = dst
            slots.append(table[L // B] * B + L % B)
            L += 1
        self.lens[seq] = L
        return slots, copies

    def fork(self, parent: int, child: int) -> None:
        assert child not in self.tables
        self.tables[child] = list(self.tables[parent])
        self.lens[child] = self.lens[parent]
        for b in self.tables[child]:
            self.ref[b] += 1

    def free_sequence(self, seq: int) -> None:
        for b in self.tables.pop(seq):
            self._drop(b)
        del self.lens[seq]

    # ---------------------------------------------------------------- views
    def table(self, seq: int) -> List[int]:
        return list(self.tables[seq])

    def num_free(self) -> int:
        return len(self.free)

    def used_blocks(self) -> int:
        return self.num_blocks - len(self.free)

    def tokens(self) -> int:
        return sum(self.lens.values())
