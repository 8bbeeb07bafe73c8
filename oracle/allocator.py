"""Block pool with a free list, reference counts, fork and copy-on-write.
Test infrastructure only (see package doc).

What the pages fix:
  * The KV cache is cut into fixed-size blocks handed out one at a time, when
    needed, from anywhere in the pool ([vLLM2] block-table section; [KV02]
    section 2: a new block is taken when the token fills the current one).
  * A sequence appends into its current block; when the block is full a free
    physical block is allocated and the table extended.  When a request ends,
    blocks nobody references any more go back to the free pool ([PA] "Block
    Table 如何工作").
  * Several logical sequences may point at the same physical blocks (shared
    prefix, parallel sampling, beam search); blocks carry a reference count,
    and a new block is allocated and copied only when a branch really writes
    different content (copy-on-write) ([PA] "支持块级共享"; [KV02] section 2
    "블록을 함께 쓰기").
  * Waste is confined to the unfilled tail of each sequence's last block:
    ceil(600/16) = 38 blocks = 608 token slots for 600 tokens ([PA] "先看直观
    解释"), fewer than block_size slots per request ([KV02] section 2).

Readings where the pages leave a step open:
  * free-list order: the list starts in the given order (identity by
    default); ``allocate`` takes the front; a block whose count drops to 0 is
    appended at the back.
  * ``append_slot``: position pos = current length.  pos % bs == 0 -> allocate
    a fresh block.  Otherwise, if the last block's count is > 1 -> allocate a
    new block, report (old, new) as a copy pair, drop one reference to old and
    put new in this sequence's table; a sole holder writes in place.  The slot
    is table[pos // bs] * bs + pos % bs.  On exhaustion nothing changes.
  * ``free_seq`` releases the sequence's blocks in table order.
  * sequence ids count up from 0 and are never reused.
"""
from __future__ import annotations

from collections import deque


class AllocatorOOM(RuntimeError):
    """No free block left; the allocator state is unchanged."""


def blocks_for(num_tokens: int, block_size: int) -> int:
    """Blocks a sequence of ``num_tokens`` tokens holds: ceil(n / bs)."""
    return -(-int(num_tokens) // int(block_size))


def slack_for(num_tokens: int, block_size: int) -> int:
    """Unused token slots in the last block."""
    return blocks_for(num_tokens, block_size) * block_size - int(num_tokens)


class OracleAllocator:
    def __init__(self, num_blocks: int, block_size: int, free_order=None):
        if num_blocks <= 0 or block_size <= 0:
            raise ValueError("num_blocks and block_size must be positive")
        order = list(range(num_blocks)) if free_order is None else [int(b) for b in free_order]
        if sorted(order) != list(range(num_blocks)):
            raise ValueError("free_order must be a permutation of 0..num_blocks-1")
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.free = deque(order)
        self.ref = [0] * num_blocks
        self.tables: dict[int, list[int]] = {}
        self.lens: dict[int, int] = {}
        self._next_seq = 0

    # ---- block level -----------------------------------------------------
    def num_free(self) -> int:
        return len(self.free)

    def refcount(self, b: int) -> int:
        return self.ref[b]

    def allocate(self) -> int:
        """Take the front of the free list (count 1); -1 when the pool is empty."""
        if not self.free:
            return -1
        b = self.free.popleft()
        self.ref[b] = 1
        return b

    def incref(self, b: int) -> None:
        if self.ref[b] <= 0:
            raise ValueError(f"block {b} is free")
        self.ref[b] += 1

    def decref(self, b: int) -> None:
        if self.ref[b] <= 0:
            raise ValueError(f"block {b} is already free")
        self.ref[b] -= 1
        if self.ref[b] == 0:
            self.free.append(b)

    # ---- sequence level --------------------------------------------------
    def seq_create(self) -> int:
        s = self._next_seq
        self._next_seq += 1
        self.tables[s] = []
        self.lens[s] = 0
        return s

    def fork(self, parent: int) -> int:
        """A new sequence sharing every block of ``parent`` (counts + 1)."""
        child = self.seq_create()
        self.tables[child] = list(self.tables[parent])
        self.lens[child] = self.lens[parent]
        for b in self.tables[child]:
            self.incref(b)
        return child

    def append_slot(self, seq: int):
        """Reserve the slot of the sequence's next token.

        Returns (slot, cow_src, cow_dst); cow_src = cow_dst = -1 when no copy
        is needed.  Raises AllocatorOOM (state unchanged) if a block is needed
        and none is free.
        """
        table = self.tables[seq]
        pos = self.lens[seq]
        bs = self.block_size
        cow = (-1, -1)
        if pos % bs == 0:
            nb = self.allocate()
            if nb < 0:
                raise AllocatorOOM("pool exhausted")
            table.append(nb)
        else:
            last = table[pos // bs]
            if self.ref[last] > 1:
                nb = self.allocate()
                if nb < 0:
                    raise AllocatorOOM("pool exhausted")
                self.decref(last)
                table[pos // bs] = nb
                cow = (last, nb)
        self.lens[seq] = pos + 1
        slot = table[pos // bs] * bs + pos % bs
        return slot, cow[0], cow[1]

    def append_tokens(self, seq: int, n: int) -> list:
        """``n`` successive append_slot calls; returns their slots."""
        out = []
        for _ in range(n):
            slot, a, b = self.append_slot(seq)
            if a >= 0:
                raise AssertionError("append_tokens is meant for unshared sequences")
            out.append(slot)
        return out

    def free_seq(self, seq: int) -> None:
        for b in self.tables.pop(seq):
            self.decref(b)
        del self.lens[seq]

    def block_table(self, seq: int) -> list:
        return list(self.tables[seq])

    def seq_len(self, seq: int) -> int:
        return self.lens[seq]

    def live_seqs(self) -> list:
        return sorted(self.tables)

    def snapshot(self):
        """(free list in order, reference counts, {seq: (table, len)})."""
        return (list(self.free), list(self.ref),
                {s: (list(self.tables[s]), self.lens[s]) for s in sorted(self.tables)})
