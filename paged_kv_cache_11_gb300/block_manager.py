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

* ``swap_out`` / ``swap_in`` move a whole sequence between a GPU pool's
  manager and a host pool's manager (tonho.wtf "vllm", "como funciona":
  eviction is all-or-nothing per sequence, and a sequence comes back by swap
  from CPU RAM) and return the (src, dst) block pairs for ``swap_blocks``;
* ``needs_compaction`` / ``compact`` implement the trigger and the target
  allocation of token-level compaction (gist.science "Zipage", Compressed
  PagedAttention: a request may hold at most N_max blocks; when it has N_max
  and the last is full, the tokens it keeps are written into fresh target
  blocks, at most N_max - 1 of them, so that blocks shared with other
  requests stay intact) and return the (src slot, dst slot) pairs for
  ``compact_tokens``.  Which tokens to keep is the caller's choice.

The kernels never see this object: it produces the slot mapping, the block
tables and the copy pairs that the C ABI consumes.
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
        self._deferred: list[int] = []

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

    # -- token-level compaction ----------------------------------------------
    def needs_compaction(self, seq: int, n_max: int) -> bool:
        """True when the sequence holds n_max blocks (or more) and its last block is full."""
        s = self._seqs[seq]
        return len(s.table) >= n_max and s.num_tokens % self.block_size == 0 and s.num_tokens > 0

    def compact(self, seq: int, keep_positions, defer_free: bool = False) -> tuple[list[int], list[int]]:
        """Rewrite the kept token positions (ascending) into fresh target blocks.

        The sequence's table becomes the target blocks and its length the
        number of kept tokens; its old blocks lose one reference each (blocks
        still shared with other sequences stay).  Returns (src_slots,
        dst_slots) for compact_tokens.  With defer_free, blocks that drop to
        zero references stay out of the free list until release_deferred():
        several compactions can then share one compact_tokens launch without
        a later one's targets landing on an earlier one's sources.
        """
        s = self._seqs[seq]
        keep = [int(p) for p in keep_positions]
        if any(b <= a for a, b in zip(keep, keep[1:])) or (keep and not 0 <= keep[0] <= keep[-1] < s.num_tokens):
            raise ValueError("keep_positions must be ascending positions of the sequence")
        bs = self.block_size
        targets = [self._take() for _ in range((len(keep) + bs - 1) // bs)]
        src = [s.table[p // bs] * bs + p % bs for p in keep]
        dst = [targets[i // bs] * bs + i % bs for i in range(len(keep))]
        for b in s.table:
            self.refcount[b] -= 1
            if self.refcount[b] == 0:
                (self._deferred if defer_free else self._free).append(b)
        s.table = targets
        s.num_tokens = len(keep)
        return src, dst

    def release_deferred(self) -> int:
        """Return the blocks held back by compact(defer_free=True) to the free list."""
        n = len(self._deferred)
        self._free.extend(self._deferred)
        self._deferred.clear()
        return n


def swap_out(gpu: BlockManager, cpu: BlockManager, seq: int) -> list[tuple[int, int]]:
    """Move a sequence from the GPU pool's manager to the host pool's manager.

    Every block of the sequence gets a host block; the GPU blocks lose the
    sequence's reference.  Returns the (gpu block, host block) pairs to copy
    with swap_blocks before the GPU blocks are reused.
    """
    return _move(gpu, cpu, seq)


def swap_in(cpu: BlockManager, gpu: BlockManager, seq: int) -> list[tuple[int, int]]:
    """Bring a swapped-out sequence back; returns the (host block, gpu block) pairs."""
    return _move(cpu, gpu, seq)


def _move(src: BlockManager, dst: BlockManager, seq: int) -> list[tuple[int, int]]:
    if src.block_size != dst.block_size:
        raise ValueError("pools must use the same block size")
    n = src.num_tokens(seq)
    table = src.block_table(seq)
    if dst.num_free < len(table):
        raise OutOfBlocks("destination pool full")
    dst.add_sequence(seq)
    dst._seqs[seq].num_tokens = n
    pairs = []
    for b in table:
        nb = dst._take()
        dst._seqs[seq].table.append(nb)
        pairs.append((b, nb))
    src.free(seq)
    return pairs
