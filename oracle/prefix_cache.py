"""Automatic prefix caching on top of the block pool.  Test infrastructure only.

[KV02] section 4 "프리픽스 캐시: 같은 앞부분은 한 번만 계산" -- requests that
share the front of their prompt (a system prompt, a document asked about
several times, a replayed conversation) have the same K/V there, so blocks
already on the GPU are reused and that much prefill is skipped:
  * each block gets a key = hash(previous block's key, this block's token
    ids, extra information); the extra information carries what separates
    requests (adapter, input hashes, a per-user cache salt);
  * because the previous key is hashed in, one key stands for the whole
    prefix up to its block: the same block_size tokens after a different
    prefix give a different key;
  * only full blocks are cached;
  * a finished request's blocks are not wiped: they wait, empty but with
    their contents, in a queue and are evicted least recently used first
    when space is needed; a finished request's blocks enter that queue from
    the back (its tail first), so the tails, least likely to be reused, go
    first;
  * the default hash is sha256.

Readings where the page leaves a step open:
  * byte layout of a key's input: the previous key (32 zero bytes for a
    sequence's first block), then the block's token ids as little-endian
    int32, then the request's extra bytes; hash = SHA-256 (hashlib);
  * the eviction queue is the pool's free list: a block whose count reaches
    zero keeps its key and goes to the back; allocation takes the front and
    drops that block's key; a cache hit takes its block off the list;
  * a new request reuses cached blocks from its first block on, up to the
    first miss; a key already cached for another block leaves a new block
    unkeyed (the first holder keeps the key);
  * a sequence appended to without token ids (plain slot reservations) stops
    being keyed.
"""
from __future__ import annotations

import hashlib

import numpy as np

from .allocator import AllocatorOOM, OracleAllocator, blocks_for


def block_key(prev_key, token_ids, extra: bytes = b"") -> bytes:
    """SHA-256(prev_key or 32 zero bytes || token ids as <i4 || extra)."""
    h = hashlib.sha256()
    h.update(bytes(32) if prev_key is None else bytes(prev_key))
    h.update(np.asarray(token_ids, dtype="<i4").tobytes())
    h.update(bytes(extra))
    return h.digest()


class OraclePrefixCacheAllocator(OracleAllocator):
    def __init__(self, num_blocks: int, block_size: int, free_order=None):
        super().__init__(num_blocks, block_size, free_order)
        self.key_of_block: dict[int, bytes] = {}
        self.cache: dict[bytes, int] = {}
        self.track: dict[int, dict] = {}  # seq -> tokens, extra, keyed blocks, last key

    # ---- eviction: allocation takes the front and drops its key ----------
    def allocate(self) -> int:
        b = super().allocate()
        if b >= 0 and b in self.key_of_block:
            del self.cache[self.key_of_block.pop(b)]
        return b

    # ---- sequences ----------------------------------------------------------
    def fork(self, parent: int) -> int:
        child = super().fork(parent)
        if parent in self.track:
            st = self.track[parent]
            self.track[child] = dict(tokens=list(st["tokens"]), extra=st["extra"], keyed=st["keyed"],
                                     last=st["last"])
        return child

    def append_slot(self, seq: int):
        out = super().append_slot(seq)
        self.track.pop(seq, None)  # no token id: the sequence is no longer keyed
        return out

    def free_seq(self, seq: int) -> None:
        for b in reversed(self.tables.pop(seq)):  # tail first into the queue
            self.decref(b)
        del self.lens[seq]
        self.track.pop(seq, None)

    def _register(self, seq: int) -> None:
        st = self.track.get(seq)
        if st is None:
            return
        bs = self.block_size
        while st["keyed"] < self.lens[seq] // bs:
            j = st["keyed"]
            k = block_key(st["last"], st["tokens"][j * bs:(j + 1) * bs], st["extra"])
            b = self.tables[seq][j]
            if b not in self.key_of_block and k not in self.cache:
                self.key_of_block[b] = k
                self.cache[k] = b
            st["last"] = k
            st["keyed"] += 1

    def seq_create_prefix(self, token_ids, extra: bytes = b""):
        """(seq, cached_tokens, slots) for a new request of these tokens."""
        ids = [int(t) for t in token_ids]
        bs, n = self.block_size, len(ids)
        hits, keys = [], []
        for j in range(n // bs):
            k = block_key(keys[-1] if keys else None, ids[j * bs:(j + 1) * bs], extra)
            b = self.cache.get(k)
            if b is None:
                break
            hits.append(b)
            keys.append(k)
        in_queue = sum(1 for b in hits if self.ref[b] == 0)
        if blocks_for(n, bs) - len(hits) > len(self.free) - in_queue:
            raise AllocatorOOM("pool exhausted")
        s = self.seq_create()
        for b in hits:
            if self.ref[b] == 0:
                self.free.remove(b)
            self.ref[b] += 1
            self.tables[s].append(b)
        self.lens[s] = len(hits) * bs
        self.track[s] = dict(tokens=ids, extra=bytes(extra), keyed=len(hits),
                             last=keys[-1] if keys else None)
        for _ in range(self.lens[s], n):
            OracleAllocator.append_slot(self, s)
        slots = [self.tables[s][t // bs] * bs + t % bs for t in range(n)]
        self._register(s)
        return s, len(hits) * bs, slots

    def append_token_ids(self, seq: int, token_ids) -> list:
        """Unshared append of these tokens; completed blocks get their keys."""
        ids = [int(t) for t in token_ids]
        bs, pos = self.block_size, self.lens[seq]
        if pos % bs and self.ref[self.tables[seq][pos // bs]] > 1:
            raise ValueError("the last block is shared: append with copy-on-write instead")
        if blocks_for(pos + len(ids), bs) - len(self.tables[seq]) > len(self.free):
            raise AllocatorOOM("pool exhausted")
        slots = [OracleAllocator.append_slot(self, seq)[0] for _ in ids]
        if seq in self.track:
            self.track[seq]["tokens"].extend(ids)
            self._register(seq)
        return slots

    def snapshot(self):
        """Base snapshot plus {block: key} of the keyed blocks."""
        free, refs, seqs = super().snapshot()
        return free, refs, seqs, dict(sorted(self.key_of_block.items()))
