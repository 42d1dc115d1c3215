"""Host-side block bookkeeping for a paged KV cache.

What it does (tonho.wtf "vllm", "como funciona"; techtrendfeed "KV Cache
Administration", "How PagedAttention Works", steps 3-4):

* a sequence's tokens fill its blocks left to right; a new physical block is
  taken from the free list only when the sequence's last block is full, so a
  sequence never holds more than one partly filled block;
* the block table of a sequence maps logical block i to a physical block id;
* ``fork`` makes a child that maps every block of its parent (reference count
  +1 per block) -- parallel sampling maps the prompt blocks into each sample;
* ``append_token`` into a last block whose reference count is above 1 first
  copies that block (and only it) to a fresh one: it returns the (src, dst)
  pair for ``copy_blocks`` and the slot to write;
* ``free`` drops a sequence's references; blocks at count 0 return to the
  free list.

The kernels never see this object: it produces the slot mapping, the block
tables and the copy-on-write pairs that the C ABI consumes.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Iterable


class OutOfBlocks(RuntimeError):
    pass


@dataclass
class _Seq:
    table: list[int] = field(default_factory=list)
    num_tokens: int = 0


class BlockManager:
    def __init__(self, num_blocks: int, block_size: int, free_order: Iterable[int] | None = None):
        if num_blocks < 1 or block_size < 1:
            raise ValueError("num_blocks and block_size must be >= 1")
        self.num_blocks = num_blocks
        self.block_size = block_size
        if free_order is None:
            self._free = list(range(num_blocks - 1, -1, -1))  # pop() takes block 0 first
        else:
            order = [int(b) for b in free_order]
            if sorted(order) != list(range(num_blocks)):
                raise ValueError("free_order must be a permutation of range(num_blocks)")
            self._free = order[::-1]  # pop() takes free_order[0] first
        self.refcount = [0] * num_blocks
        self._seqs: dict[int, _Seq] = {}

    # -- queries ---------------------------------------------------------
    @property
    def num_free(self) -> int:
        return len(self._free)

    def block_table(self, seq: int) -> list[int]:
        return list(self._seqs[seq].table)

    def num_tokens(self, seq: int) -> int:
        return self._seqs[seq].num_tokens

    def sequences(self) -> list[int]:
        return list(self._seqs)

    def slot(self, seq: int, pos: int) -> int:
        """Flat slot of token position ``pos``: table[pos // bs] * bs + pos % bs."""
        s = self._seqs[seq]
        if not 0 <= pos < s.num_tokens:
            raise IndexError(f"position {pos} outside sequence of {s.num_tokens} tokens")
        return s.table[pos // self.block_size] * self.block_size + pos % self.block_size

    # -- operations --------------------------------------------------------
    def _take(self) -> int:
        if not self._free:
            raise OutOfBlocks("no free block")
        b = self._free.pop()
        self.refcount[b] = 1
        return b

    def add_sequence(self, seq: int) -> None:
        if seq in self._seqs:
            raise ValueError(f"sequence {seq} exists")
        self._seqs[seq] = _Seq()

    def append_token(self, seq: int) -> tuple[int, tuple[int, int] | None]:
        """Reserve the slot of the sequence's next token.

        Returns (slot, cow) where cow is the (src, dst) block pair to copy
        before writing, or None.
        """
        s = self._seqs[seq]
        bs = self.block_size
        pos = s.num_tokens
        cow = None
        if pos % bs == 0:
            s.table.append(self._take())  # previous block full (or none yet): fresh block
        else:
            last = s.table[-1]
            if self.refcount[last] > 1:  # writing into a shared block: copy it, and only it
                new = self._take()
                self.refcount[last] -= 1
                s.table[-1] = new
                cow = (last, new)
        s.num_tokens = pos + 1
        return s.table[pos // bs] * bs + pos % bs, cow

    def append_tokens(self, seq: int, n: int) -> tuple[list[int], list[tuple[int, int]]]:
        slots, cows = [], []
        for _ in range(n):
            slot, cow = self.append_token(seq)
            slots.append(slot)
            if cow is not None:
                cows.append(cow)
        return slots, cows

    def fork(self, parent: int, child: int) -> None:
        """The child maps every block of the parent (shared, reference counted)."""
        if child in self._seqs:
            raise ValueError(f"sequence {child} exists")
        p = self._seqs[parent]
        for b in p.table:
            self.refcount[b] += 1
        self._seqs[child] = _Seq(table=list(p.table), num_tokens=p.num_tokens)

    def free(self, seq: int) -> None:
        s = self._seqs.pop(seq)
        for b in s.table:
            self.refcount[b] -= 1
            if self.refcount[b] == 0:
                self._free.append(b)
