"""Reference block manager: free list, allocate-on-full, fork, copy-on-write, free.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The rules, restated from the pages:

* "How vLLM and PagedAttention Actually Work" §6 (Python blueprint) and
  "PagedAttention Explained" (copy-on-write section): the free list starts as
  every block id in order and hands out its FRONT entry; a freed block goes to
  its BACK.
* "vLLM — PagedAttention", Block Table Data Structure and "vLLM PagedAttention",
  block-table section: a sequence takes a new physical block only when its last
  block is full (``length % B == 0``).
* "vLLM — PagedAttention", Copy-on-Write Logic: before writing into a block
  whose reference count is above one, take a fresh block, copy the old one into
  it, point this sequence's table at the copy and drop one reference from the
  old block.  With a count of one the sequence writes in place.
* "vLLM — PagedAttention", Three Core API Methods: fork shares every block of
  the parent (each count grows by one); free drops one reference per block.

Every copy the rules decide is recorded as a ``(src, dst)`` pair; the pairs of a
step are what the batched block-copy launch consumes.
"""

from __future__ import annotations

from typing import Dict, List, Tuple


class CowBlockManager:
    def __init__(self, num_blocks: int, block_size: int):
        if num_blocks <= 0 or block_size <= 0:
            raise ValueError("num_blocks and block_size must be positive")
        self.block_size = block_size
        self.free: List[int] = list(range(num_blocks))
        self.ref: Dict[int, int] = {}
        self.tables: Dict[str, List[int]] = {}
        self.lengths: Dict[str, int] = {}
        self.pending_copies: List[Tuple[int, int]] = []

    # -- allocation ---------------------------------------------------------
    def _take(self) -> int:
        if not self.free:
            raise MemoryError("no free block: the scheduler must preempt")
        b = self.free.pop(0)
        self.ref[b] = 1
        return b

    def _drop(self, b: int) -> None:
        self.ref[b] -= 1
        if self.ref[b] == 0:
            self.free.append(b)

    # -- sequence operations ------------------------------------------------
    def new_sequence(self, seq: str) -> None:
        if seq in self.tables:
            raise KeyError(f"sequence {seq!r} exists")
        self.tables[seq] = []
        self.lengths[seq] = 0

    def append_slot(self, seq: str) -> int:
        """Make room for one more token of ``seq``; return its flat slot.

        New block when the last one is full; copy-on-write when the last block
        is shared.  The slot is ``phys * B + offset``.
        """
        table = self.tables[seq]
        n = self.lengths[seq]
        off = n % self.block_size
        if off == 0:
            table.append(self._take())
        elif self.ref[table[-1]] > 1:
            old = table[-1]
            new = self._take()
            self.pending_copies.append((old, new))
            self.ref[old] -= 1          # still > 0: another sequence holds it
            table[-1] = new
        self.lengths[seq] = n + 1
        return table[-1] * self.block_size + off

    def fork(self, parent: str, child: str, num_tokens: int | None = None) -> None:
        """Start ``child`` sharing the parent's first ``num_tokens`` tokens.

        With ``num_tokens`` None the child shares the whole parent, partial
        last block included (parallel sampling).  Otherwise only whole blocks
        may be shared (full-block prefix sharing), so ``num_tokens`` must be a
        multiple of the block size.
        """
        if num_tokens is None:
            num_tokens = self.lengths[parent]
            nb = len(self.tables[parent])
        else:
            if num_tokens % self.block_size:
                raise ValueError("only whole blocks can be shared by prefix")
            nb = num_tokens // self.block_size
        shared = self.tables[parent][:nb]
        for b in shared:
            self.ref[b] += 1
        self.tables[child] = list(shared)
        self.lengths[child] = num_tokens

    def free_sequence(self, seq: str) -> None:
        for b in self.tables.pop(seq):
            self._drop(b)
        del self.lengths[seq]

    # -- queries ------------------------------------------------------------
    def take_copies(self) -> List[Tuple[int, int]]:
        out, self.pending_copies = self.pending_copies, []
        return out

    def blocks_in_use(self) -> int:
        return sum(1 for c in self.ref.values() if c > 0)
